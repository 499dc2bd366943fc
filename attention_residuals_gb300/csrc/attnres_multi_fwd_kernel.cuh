// attnres_multi_fwd_kernel.cuh -- forward kernel of the multi-query read, a
// template included by attnres_multi_fwd.cu (precompiled instances) and
// compiled at run time for one plan's exact shape (attnres_jit.cu).
//
// "Fast Attention Residuals", section "Multi-query AttnRes": the same
// sources are read with M queries (1 <= M <= 16); each query has its own
// source weights and its own full-width output.  Per token and query m
// (section "Equation"):
//   r_s = 1/sqrt(mean(t_s^2) + eps),  z_ms = scale * r_s * <t_s, q_m>,
//   alpha_m = softmax_s(z_m),          y_m = sum_s alpha_ms v_s.
// The key statistics r_s do not depend on the query, so they are formed once
// per token.
//
// GB300 mapping: the single-query forward's streaming design, serving MB
// queries per pass over a token.  Persistent CTAs (two per SM when a thread
// owns at most two vectors, so one CTA's barrier and softmax phases overlap
// the other's streaming); a producer thread streams the token's rows into a
// ring of chunks with 1-D TMA bulk copies; the softmax runs online over
// groups of whole chunks, so a token never has to fit in shared memory.
//   pass 1: one warp per row; lanes stride over the key vectors and form the
//           key sum of squares (first block only) and the MB query dots with
//           mixed-precision bf16 FMAs, then one reduce-scatter per row;
//   softmax: after one CTA barrier every warp updates the MB running maxima
//           and denominators itself (identical inputs, identical results),
//           so no second barrier is needed;
//   pass 2: thread t owns fixed 16-byte column vectors and accumulates the
//           MB outputs in FP32 registers (each row unpacked once for all MB
//           queries, packed FFMA2), releasing each chunk after its rows.
// With M > MB the queries are served in blocks of MB: a token that fits in
// one softmax group stays in shared memory for every block; a longer token is
// streamed once per block, all passes but the last asking L2 to keep the rows
// (evict_last), so the re-reads are served from L2 and HBM sees each row once.
// With a few queries these are bandwidth-bound per-token reductions; nine or
// more queries make the per-token products dense enough for the tensor-core
// form (attnres_multi_fwd_mma.cu), which runs instead where it applies.
#pragma once

#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"

// Anonymous in the precompiled units; named by the run-time compiler.
#ifndef ATTNRES_FWD_NS
#define ATTNRES_FWD_NS
#endif

namespace attnres {
namespace ATTNRES_FWD_NS {

// First failed wait of any multi-query forward launch (0 = none).
__device__ unsigned int g_multi_error = 0;

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// SC, GC, GGC, KC > 0 fix S, the rows per chunk, the softmax group rows and
// the ring depth at compile time (the run-time-compiled form for one plan);
// 0 reads them from the arguments.
template <int VPT, int MB, bool SEL, int MQ, int SC = 0, int GC = 0, int GGC = 0, int KC = 0>
__global__ void __launch_bounds__(kMaxThreads, multi_fwd_ctas_per_sm(VPT))
    attnres_multi_fwd_kernel(const __grid_constant__ MultiFwdArgs a) {
    constexpr int KV = 1 + MB;                     // values reduced per row
    constexpr int KR = KV <= 2 ? 2 : (KV <= 4 ? 4 : 8);  // reduce-scatter width
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = KC > 0 ? KC : a.chunks;
    const int G = GC > 0 ? GC : a.rows;
    const int GG = GGC > 0 ? GGC : a.group;
    const int S = SC > 0 ? SC : a.S;
    const int M = MQ > 0 ? MQ : a.M;               // MQ > 0: the query count is fixed at compile time
    const int s_pad = a.s_pad;
    const int nblk = (M + MB - 1) / MB;            // register blocks of queries
    // A token that fits in one softmax group is loaded once and every block
    // reads it from shared memory; otherwise it is streamed once per block.
    const bool one_group = S <= GG;
    const int npass = one_group ? 1 : nblk;
    const MultiFwdLayout L = make_multi_fwd_layout(K, G, a.slot_bytes, s_pad, a.qrows, a.nkv);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    float* red = reinterpret_cast<float*>(smem + L.red);    // [2][KV][kMaxGroup]
    float* zall = reinterpret_cast<float*>(smem + L.zall);  // [MB][s_pad]
    float* rall = reinterpret_cast<float*>(smem + L.rall);  // [s_pad]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const uint32_t sb = static_cast<uint32_t>(a.slot_bytes);
    const uint32_t cb = static_cast<uint32_t>(G) * sb;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // the backward may start launching (it waits for this grid before it
    // touches global memory)
    pdl_launch_dependents();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_last = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            const uint32_t bytes = static_cast<uint32_t>(a.D) * 2u;
            unsigned char* ring = smem + L.ring;
            int k = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (long long n = blockIdx.x; n < N && !*abort_flag; n += gridDim.x) {
                for (int b = 0; b < npass && !*abort_flag; ++b) {
                    const uint64_t pol = b + 1 < npass ? pol_keep : pol_last;
                    for (int g0 = 0; g0 < S; g0 += G) {
                        const int gs = min(G, S - g0);
                        if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_multi_error, kSiteFwdProducer)) break;
                        mbar_arrive_expect_tx(full + k, bytes * static_cast<uint32_t>(gs));
                        for (int r = 0; r < gs; ++r) {
                            const unsigned char* src =
                                static_cast<const unsigned char*>(a.src[g0 + r]) + (n * a.src_ld) * 2;
                            tma_load_1d(ring + k * cb + r * sb, src, bytes, full + k, pol);
                        }
                        ++issued;
                        if (++k == K) {
                            k = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA can exit.
                for (int c = 0; c < K && c < issued; ++c) {
                    const long long fills = (issued - 1 - c) / K + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_error, kSiteDrain);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = a.D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    const int kv0 = a.kv0, nkv = a.nkv;
    const int kw = nkv * 8;
    const uint32_t kwb = static_cast<uint32_t>(nkv) * 16u;  // bytes per query row in shared memory
    const bool selected = SEL;                       // per-token queries from a bank (a.ids set)
    const bool q_once = !selected && a.qrows >= M;         // every query stays in shared memory
    const bool bank_res = selected && a.bank_rows > 0;     // the whole bank stays in shared memory
    int col[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * nct;
        col[i] = c < ncv ? c : -1;
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t voff = static_cast<uint32_t>(col[0] < 0 ? 0 : col[0]) * 16u;
    const uint32_t vstep = static_cast<uint32_t>(nct) * 16u;
    const uint32_t ring_raw = sbase + L.ring;
    const uint32_t ring_lo = ring_raw + voff;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    const uint32_t qsm_s = sbase + L.qsm;
    uint16_t* qsm = reinterpret_cast<uint16_t*>(smem + L.qsm);
    // queries m0 .. m0+rows-1 by key channel: row j holds channels
    // 8*kv0 .. 8*(kv0+nkv), zero outside the key and past M
    const bool key_aligned = ((ko | kend) & 7) == 0;
    // With an aligned key and a 16-byte aligned query array a query row is
    // copied as whole 16-byte vectors (the key window is then exactly R).
    const bool q_vec = key_aligned && (reinterpret_cast<uintptr_t>(a.q) & 15u) == 0;
    // Source row of query m of token n: the query array, or the bank row the
    // token selects (an id outside [0, E) is recorded as an error and reads
    // as a zero query).
    auto qsrc = [&](long long n, int m) -> const uint16_t* {
        if (!selected) return a.q + static_cast<long long>(m) * a.R;
        const long long id = a.ids[n * M + m];
        if (id < 0 || id >= a.E) {
            atomicCAS(&g_multi_error, 0u, static_cast<unsigned>(kSiteBadId));
            return nullptr;
        }
        return a.q + id * a.R;
    };
    auto load_q = [&](long long n, int m0, int rows) {
        if (q_vec) {
#pragma unroll 4
            for (int i = threadIdx.x; i < rows * nkv; i += nct) {
                const int j = i / nkv;
                const int m = m0 + j;
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                const uint16_t* src = m < M ? qsrc(n, m) : nullptr;
                if (src) w = ld_global_nc_v4(src + 8 * (i - j * nkv));
                *reinterpret_cast<uint4*>(qsm + 8 * i) = w;
            }
        } else {
#pragma unroll 4
            for (int i = threadIdx.x; i < rows * kw; i += nct) {
                const int j = i / kw;
                const int c = 8 * kv0 + (i - j * kw);
                const int m = m0 + j;
                const uint16_t* src = (m < M && c >= ko && c < kend) ? qsrc(n, m) : nullptr;
                qsm[i] = src ? src[c - ko] : static_cast<uint16_t>(0);
            }
        }
    };
    if (q_once) load_q(0, 0, a.qrows);
    if (bank_res) {
        // the bank by key channel, and a zero row (index E) read for ids outside [0, E)
        if (q_vec) {
            for (int i = threadIdx.x; i < a.bank_rows * nkv; i += nct) {
                const int row = i / nkv;
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (row < a.E) w = ld_global_nc_v4(a.q + static_cast<long long>(row) * a.R + 8 * (i - row * nkv));
                *reinterpret_cast<uint4*>(qsm + 8 * i) = w;
            }
        } else {
            for (int i = threadIdx.x; i < a.bank_rows * kw; i += nct) {
                const int row = i / kw;
                const int c = 8 * kv0 + (i - row * kw);
                qsm[i] = (row < a.E && c >= ko && c < kend) ? a.q[static_cast<long long>(row) * a.R + (c - ko)]
                                                            : static_cast<uint16_t>(0);
            }
        }
    }
    named_bar_sync(1, nct);
    // Resident bank: lane m < M of every warp holds the bank row of slot m,
    // loaded one token ahead; an id outside [0, E) is recorded and reads the
    // zero row.
    auto row_of = [&](long long id) -> int {
        if (id < 0 || id >= a.E) {
            atomicCAS(&g_multi_error, 0u, static_cast<unsigned>(kSiteBadId));
            return a.E;
        }
        return static_cast<int>(id);
    };
    long long id_next = (bank_res && lane < M) ? a.ids[static_cast<long long>(blockIdx.x) * M + lane] : 0;

    int ck = 0;            // current chunk
    uint32_t cphase = 0;   // its fill parity
    uint32_t cbase = ring_lo;
    int rbuf = 0;

    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        int my_row = 0;
        if (bank_res) {
            my_row = lane < M ? row_of(id_next) : a.E;
            const long long nn = n + gridDim.x;
            id_next = (lane < M && nn < N) ? a.ids[nn * M + lane] : 0;
        }
        for (int b = 0; b < nblk; ++b) {
            const int m0 = b * MB;
            const bool first = b == 0;
            if (!q_once && !bank_res) {
                // every warp finished the previous block's pass 1 before its last barrier
                load_q(n, m0, MB);
                named_bar_sync(1, nct);
            }
            const uint32_t qbase = qsm_s + static_cast<uint32_t>(q_once ? m0 : 0) * kwb;
            uint32_t qaddr[MB];  // shared-memory row of each query of the block
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                const int r = __shfl_sync(0xffffffffu, my_row, (m0 + j) & 31);
                qaddr[j] = bank_res ? qsm_s + static_cast<uint32_t>(m0 + j < M ? r : a.E) * kwb
                                    : qbase + static_cast<uint32_t>(j) * kwb;
            }
            float2 acc[MB][VPT][4];
#pragma unroll
            for (int j = 0; j < MB; ++j)
#pragma unroll
                for (int i = 0; i < VPT; ++i)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) acc[j][i][kk] = make_float2(0.0f, 0.0f);
            float m_run[MB], l_run[MB];  // running softmax state (same in every warp)
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                m_run[j] = -FLT_MAX;
                l_run[j] = 0.0f;
            }

            const bool load_rows = !one_group || b == 0;          // wait for the rows
            const bool free_rows = !one_group || b + 1 == nblk;   // release them after pass 2
            for (int g0 = 0; g0 < S; g0 += GG) {
                const int gs = min(GG, S - g0);
                if (load_rows) {
                    int k = ck;
                    uint32_t ph = cphase;
                    for (int r0 = 0; r0 < gs; r0 += G) {
                        mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_multi_error, kSiteFwdConsumer);
                        if (++k == K) {
                            k = 0;
                            ph ^= 1u;
                        }
                    }
                }
                // pass 1: one warp per row
                for (int r = warp; r < gs; r += ncw) {
                    int rr = r;
                    int kc = ck;
                    while (rr >= G) {
                        rr -= G;
                        if (++kc == K) kc = 0;
                    }
                    const uint32_t row = ring_raw + static_cast<uint32_t>(kc) * cb + static_cast<uint32_t>(rr) * sb +
                                         16u * static_cast<uint32_t>(kv0);
                    float s0 = 0.0f, s1 = 0.0f;
                    float t[MB][2];
#pragma unroll
                    for (int j = 0; j < MB; ++j) t[j][0] = t[j][1] = 0.0f;
                    for (int v = lane; v < nkv; v += 32) {
                        uint4 x = lds128(row + 16u * v);
                        if (!key_aligned) x = mask_bf16x8(x, 8 * (kv0 + v), ko, kend);
                        if (first) bf16_sq8(x, s0, s1);
#pragma unroll
                        for (int j = 0; j < MB; ++j) {
                            const uint4 qv = lds128(qaddr[j] + 16u * v);
                            bf16_dot8(x, qv, t[j][0], t[j][1]);
                        }
                    }
                    float part[KR];
                    part[0] = s0 + s1;
#pragma unroll
                    for (int j = 0; j < MB; ++j) part[1 + j] = t[j][0] + t[j][1];
#pragma unroll
                    for (int e = KV; e < KR; ++e) part[e] = 0.0f;
                    warp_reduce_scatter<KR>(part, lane);
                    constexpr int W = 32 / KR;  // lanes per reduced value
                    if ((lane & (W - 1)) == 0) {
                        const int e = lane / W;
                        if (e < KV) red[(rbuf * KV + e) * kMaxGroup + r] = part[0];
                    }
                }
                named_bar_sync(1, nct);
                // Every warp updates the running softmax of each of the MB
                // queries itself; lane l holds row g0 + l.
                float e[MB], corr[MB];
                {
                    float rs = 0.0f;
                    if (lane < gs)
                        rs = first ? rsqrtf(fmaf(red[(rbuf * KV) * kMaxGroup + lane], inv_r, a.eps)) : rall[g0 + lane];
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        const float qt = lane < gs ? red[(rbuf * KV + 1 + j) * kMaxGroup + lane] : 0.0f;
                        const float z = a.scale * rs * qt;
                        const float m_new = fmaxf(m_run[j], warp_max(lane < gs ? z : -FLT_MAX));
                        e[j] = lane < gs ? __expf(z - m_new) : 0.0f;
                        const float esum = warp_sum(e[j]);
                        corr[j] = __expf(m_run[j] - m_new);
                        l_run[j] = fmaf(l_run[j], corr[j], esum);
                        m_run[j] = m_new;
                        if (warp == 0 && lane < gs) zall[j * s_pad + g0 + lane] = z;
                    }
                    if (first && warp == 0 && lane < gs) rall[g0 + lane] = rs;
                }
                rbuf ^= 1;
                // pass 2: rescale the running sums and add this group's rows
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    const float2 c2 = make_float2(corr[j], corr[j]);
#pragma unroll
                    for (int i = 0; i < VPT; ++i)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) acc[j][i][kk] = fmul2(acc[j][i][kk], c2);
                }
                int lk = ck;            // chunk cursor of this pass
                uint32_t lbase = cbase;
                uint32_t lphase = cphase;
                for (int r0 = 0; r0 < gs; r0 += G) {
                    const int rn = min(G, gs - r0);
                    uint32_t dep = 0;
                    uint32_t rowa = lbase;
                    for (int r = 0; r < rn; ++r) {
                        float2 es2[MB];
#pragma unroll
                        for (int j = 0; j < MB; ++j) {
                            const float es = __shfl_sync(0xffffffffu, e[j], r0 + r);
                            es2[j] = make_float2(es, es);
                        }
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            if (col[i] >= 0) {
                                const uint4 xv = lds128(rowa + i * vstep);
                                dep ^= xv.x;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const float2 x2 = bf2_to_f2(u4_get(xv, kk));
#pragma unroll
                                    for (int j = 0; j < MB; ++j) acc[j][i][kk] = ffma2(es2[j], x2, acc[j][i][kk]);
                                }
                            }
                        }
                        rowa += sb;
                    }
                    if (free_rows) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive_after(empty_s + 8u * lk, dep);
                    }
                    lbase += cb;
                    if (++lk == K) {
                        lk = 0;
                        lbase = ring_lo;
                        lphase ^= 1u;
                    }
                }
                if (free_rows) {
                    ck = lk;
                    cbase = lbase;
                    cphase = lphase;
                }
            }
            // this block's outputs and statistics
            float inv_l[MB];
#pragma unroll
            for (int j = 0; j < MB; ++j) inv_l[j] = 1.0f / l_run[j];
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                if (m0 + j < M) {
                    const float2 il2 = make_float2(inv_l[j], inv_l[j]);
                    uint16_t* yrow = a.y + static_cast<long long>(m0 + j) * a.y_ms + n * a.y_ns;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (col[i] >= 0 && ATTNRES_IN_BOUNDS(n < a.N && 8 * col[i] + 8 <= a.D, &g_multi_error)) {
                            st_global_cs_v4(yrow + 8 * col[i],
                                            make_uint4(pack_f2(fmul2(acc[j][i][0], il2)), pack_f2(fmul2(acc[j][i][1], il2)),
                                                       pack_f2(fmul2(acc[j][i][2], il2)), pack_f2(fmul2(acc[j][i][3], il2))));
                        }
                    }
                }
            }
            if (warp == 0) {
                __syncwarp();
                for (int s = lane; s < S; s += 32) {
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        if (m0 + j < M) {
                            const float z = zall[j * s_pad + s];
                            a.alpha[(n * M + m0 + j) * S + s] = __expf(z - m_run[j]) * inv_l[j];
                            a.logit[(n * M + m0 + j) * S + s] = z;
                        }
                    }
                    if (first) a.rstd[n * S + s] = rall[s];
                }
            }
        }
    }
}

}  // namespace ATTNRES_FWD_NS
}  // namespace attnres
