// attnres_fwd_kernel.cuh -- forward kernel of the Attention Residuals read
// operator, a template included by attnres_fwd.cu (precompiled instances)
// and compiled at run time for one plan's exact shape (attnres_jit.cu).
//
// Per token ("Fast Attention Residuals", section "Equation"): key statistics
// of every source's key slice, a softmax over sources of the scaled query
// dot, and the routing-weighted full-width sum; optionally the output
// RMSNorm whose reciprocal RMS is saved for the backward ("[Perf]
// Parallelize AttnRes long-sequence reduction", Summary).
//
// GB300 mapping.  Persistent CTAs (two per SM when a thread owns at most two
// vectors, so that one CTA's barrier and softmax phases overlap the other's
// streaming work) walk tokens n = blockIdx.x, blockIdx.x + gridDim.x, ...  A producer thread streams every source row of
// the token into a ring of shared-memory row slots with 1-D TMA bulk copies
// (one cp.async.bulk per row).  The ring is organised in chunks of G rows
// with one "full" and one "empty" mbarrier each, so waits and releases cost
// one barrier operation per G rows.  Consumer thread t owns the 16-byte
// column vectors t, t + 32*ncw, ... of every row, so each warp reads 512
// contiguous bytes per shared load.  A softmax group is a whole number of
// chunks (the whole token when it fits beside two loading chunks): the
// consumers wait for its chunks, then pass 1 gives each row to one warp,
// which accumulates the row's key sum of squares and query dot with
// mixed-precision FMAs on the bf16 halves (query in shared memory) and
// reduces them within the warp; after one CTA barrier every warp updates
// the running softmax maximum and denominator itself (redundantly, so no
// second barrier is needed), and pass 2 adds the weighted rows into FP32
// registers, thread t owning fixed columns, and releases the chunks.  The output norm needs one more CTA reduction per
// token.  The pre-norm mixture o is written (FP32) only when asked for.
// Fused block-partial sum ("Fast Attention Residuals", section "Full and
// Block schedules": the caller sums the partial block before the read): with
// `delta` set, the producer also streams the token's delta row into a small
// slot ring, and the warp whose pass-1 row is the last source first replaces
// that row in shared memory by the bf16 sum src[S-1] + delta and stores it
// as the new partial sum; the group barrier then orders those writes before
// pass 2, so the sum is never re-read from HBM.
// This is a bandwidth-bound per-token reduction: no tensor cores.
#pragma once

#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"

// The kernel lives in an anonymous namespace in the precompiled units; the
// run-time compiler names it so its instances can be looked up.
#ifndef ATTNRES_FWD_NS
#define ATTNRES_FWD_NS
#endif

namespace attnres {
namespace ATTNRES_FWD_NS {

// First failed wait of any forward launch (0 = none).
__device__ unsigned int g_fwd_error = 0;

// FULL: every consumer thread owns VPT whole vectors (D == 8 * VPT * 32 * ncw).
// FUSED: the block-partial sum is formed in the read (a.delta set); a
// compile-time flag so the plain read carries none of its code.
// NORM: output RMSNorm mode (0 none, 1 on, 2 on and the FP32 o also stored
// to a.o_pre), likewise fixed at compile time.
// SC, GC, GGC, KC > 0 fix S, the rows per chunk, the softmax group rows and
// the ring depth at compile time (the run-time-compiled form for one plan);
// 0 reads them from the arguments.
template <int VPT, bool FULL, bool FUSED, int NORM, int SC = 0, int GC = 0, int GGC = 0, int KC = 0>
__global__ void __launch_bounds__(kMaxThreads, fwd_ctas_per_sm(VPT)) attnres_fwd_kernel(const __grid_constant__ FwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = KC > 0 ? KC : a.chunks;  // ring depth in chunks
    const int G = GC > 0 ? GC : a.rows;    // rows per chunk
    const int GG = GGC > 0 ? GGC : a.group;  // softmax group rows (whole chunks)
    constexpr int DSL = FUSED ? kDeltaSlots : 0;  // slots for the added rows (fused partial sum)
    const SmemLayout L = make_layout(K, G, a.slot_bytes, DSL, a.s_pad, false);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* dfull = reinterpret_cast<uint64_t*>(smem + L.dyfull);
    uint64_t* dempty = reinterpret_cast<uint64_t*>(smem + L.dyempty);
    float* red = reinterpret_cast<float*>(smem + L.red);     // [2][red_rows][kRedPitch]
    float* zall = reinterpret_cast<float*>(smem + L.coef);  // [s_pad]
    float* rall = zall + a.s_pad;                           // [s_pad]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int S = SC > 0 ? SC : a.S;
    const uint32_t sb = static_cast<uint32_t>(a.slot_bytes);
    const uint32_t cb = static_cast<uint32_t>(G) * sb;  // chunk bytes

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        for (int k = 0; k < DSL; ++k) {
            mbar_init(dfull + k, 1);
            mbar_init(dempty + k, 1);  // released by the one warp that forms the sum
        }
        *abort_flag = 0;
        // the consumers' wait limit (microseconds, 0 = the default): nonzero
        // only in a test of the recovery path
        abort_flag[2] = static_cast<int>(a.test_wait_ns / 1000ull);
        mbar_fence_init();
    }
    __syncthreads();
    // the backward may start launching (it waits for this grid before it
    // touches global memory)
    pdl_launch_dependents();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = static_cast<uint32_t>(a.D) * 2u;
            unsigned char* ring = smem + L.ring;
            int k = 0;
            uint32_t phase = 0;
            long long issued = 0;  // chunk fills started
            int dk = 0;
            uint32_t dphase = 0;
            long long d_issued = 0;
            for (long long n = blockIdx.x; n < N && !*abort_flag; n += gridDim.x) {
                if (DSL) {
                    // the row added to the last source, into its own slot
                    if (!mbar_wait(dempty + dk, dphase ^ 1u, abort_flag, &g_fwd_error, kSiteFwdProducer)) break;
                    mbar_arrive_expect_tx(dfull + dk, bytes);
                    tma_load_1d(smem + L.dyring + dk * sb, a.delta + n * a.delta_ld, bytes, dfull + dk, pol);
                    ++d_issued;
                    if (++dk == DSL) {
                        dk = 0;
                        dphase ^= 1u;
                    }
                }
                bool withheld = false;
                for (int g0 = 0; g0 < S; g0 += G) {
                    const int gs = min(G, S - g0);
                    if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_fwd_error, kSiteFwdProducer)) break;
                    if (a.test_withhold > 0 && blockIdx.x == 0 && issued + 1 == a.test_withhold) {
                        withheld = true;  // test hook: this fill never comes
                        break;
                    }
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
                if (withheld) break;
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA can exit.
                for (int c = 0; c < K && c < issued; ++c) {
                    const long long fills = (issued - 1 - c) / K + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_fwd_error, kSiteDrain);
                }
                for (int c = 0; c < DSL && c < d_issued; ++c) {
                    const long long fills = (d_issued - 1 - c) / (DSL > 0 ? DSL : 1) + 1;
                    volatile int no_abort = 0;
                    mbar_wait(dfull + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_fwd_error, kSiteDrain);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = a.D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    int col[VPT];
    uint4 wb[VPT];         // output-norm weight bits (1.0 without the norm)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * nct;
        col[i] = c < ncv ? c : -1;
        uint32_t ww[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t wv = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = 8 * c + 2 * kk + h;
                const uint32_t wh = (NORM != 0 && col[i] >= 0) ? a.w_o[j] : 0x3f80u;
                wv |= wh << (16 * h);
            }
            ww[kk] = wv;
        }
        wb[i] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);
    const float inv_d = 1.0f / static_cast<float>(a.D);

    // 32-bit shared addresses; chunk row addresses include this thread's
    // first vector offset.
    const uint32_t sbase = smem_u32(smem);
    const uint32_t voff = static_cast<uint32_t>(col[0] < 0 ? 0 : col[0]) * 16u;
    const uint32_t vstep = static_cast<uint32_t>(nct) * 16u;  // between a thread's vectors
    const uint32_t ring_lo = sbase + L.ring + voff;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    const uint32_t red_s = sbase + L.red;
    const int red_rows = L.red_rows;
    const int nq = (ncw + 3) >> 2;  // 16-byte loads per reduction row

    // warp partials never written stay zero in the reduction scratch; the
    // query goes to shared memory indexed by channel (zero outside the key)
    for (int k = threadIdx.x; k < 2 * red_rows * kRedPitch; k += nct) red[k] = 0.0f;
    {
        uint16_t* qsm = reinterpret_cast<uint16_t*>(smem + L.qsm);
        for (int j = threadIdx.x; j < a.slot_bytes / 2; j += nct)
            qsm[j] = (j >= ko && j < kend) ? a.q[j - ko] : static_cast<uint16_t>(0);
    }
    named_bar_sync(1, nct);
    const uint32_t ring_raw = sbase + L.ring;  // row addresses without a column offset
    const uint32_t qsm_s = sbase + L.qsm;
    const int kv0 = ko >> 3, kv1 = (kend + 7) >> 3;  // key vectors of a row
    const bool key_aligned = ((ko | kend) & 7) == 0;

    auto red_sum = [&](int buf, int row) -> float {
        const uint32_t base = red_s + static_cast<uint32_t>(((buf * red_rows + row) * kRedPitch) * 4);
        float t = 0.0f;
        for (int q4 = 0; q4 < nq; ++q4) {
            const float4 v = lds128f(base + 16u * q4);
            t += (v.x + v.y) + (v.z + v.w);
        }
        return t;
    };

    int ck = 0;            // current chunk
    uint32_t cphase = 0;   // its fill parity
    uint32_t cbase = ring_lo;
    int rbuf = 0;
    int dslot = 0;               // slot of this token's added row (fused partial sum)
    uint32_t dslot_phase = 0;
    const uint32_t dfull_s = sbase + L.dyfull;
    const uint32_t dempty_s = sbase + L.dyempty;

    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        float2 acc[VPT][4];
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) acc[i][kk] = make_float2(0.0f, 0.0f);
        float m_run = -FLT_MAX;  // running softmax maximum (same in every warp)
        float l_run = 0.0f;      // running softmax denominator

        for (int g0 = 0; g0 < S; g0 += GG) {
            const int gs = min(GG, S - g0);
            // wait for every chunk of the group (rows [g0, g0 + gs))
            {
                int k = ck;
                uint32_t ph = cphase;
                for (int r0 = 0; r0 < gs; r0 += G) {
                    mbar_wait_ctl_s(full_s + 8u * k, ph, abort_flag, &g_fwd_error, kSiteFwdConsumer);
                    if (++k == K) {
                        k = 0;
                        ph ^= 1u;
                    }
                }
            }
            // pass 1: key sum of squares and query dot.  One warp per row
            // (rows warp, warp + ncw, ...): lanes stride over the row's key
            // vectors and multiply the bf16 halves directly, then one warp
            // reduction gives the row's totals.  No cross-warp sums needed.
            for (int r = warp; r < gs; r += ncw) {
                int rr = r;
                int kc = ck;
                while (rr >= G) {
                    rr -= G;
                    if (++kc == K) kc = 0;
                }
                const uint32_t row_raw = ring_raw + static_cast<uint32_t>(kc) * cb + static_cast<uint32_t>(rr) * sb;
                if (DSL && g0 + r == S - 1) {
                    // fused block-partial sum: the last source becomes
                    // src[S-1] + delta (bf16 add) in place, and is stored
                    mbar_wait_s(dfull_s + 8u * dslot, dslot_phase, abort_flag, &g_fwd_error, kSiteFwdConsumer);
                    const uint32_t drow = sbase + L.dyring + static_cast<uint32_t>(dslot) * sb;
                    uint16_t* prow = a.partial_out + n * a.partial_ld;
                    uint32_t ddep = 0;
                    for (int w = lane; w < ncv; w += 32) {
                        const uint4 dv = lds128(drow + 16u * w);
                        ddep ^= dv.x;
                        const uint4 pv = add_bf16x8(lds128(row_raw + 16u * w), dv);
                        sts128(row_raw + 16u * w, pv);
                        if (ATTNRES_IN_BOUNDS(n < N && 8 * w + 8 <= a.D, &g_fwd_error)) st_global_cs_v4(prow + 8 * w, pv);
                    }
                    __syncwarp();  // the sums are visible to every lane of this warp
                    if (lane == 0) mbar_arrive_after(dempty_s + 8u * dslot, ddep);
                }
                float s0 = 0.0f, s1 = 0.0f, t0 = 0.0f, t1 = 0.0f;
                float s2 = 0.0f, s3 = 0.0f, t2 = 0.0f, t3 = 0.0f;
                int v = kv0 + lane;
                if (key_aligned) {
                    // four iterations unrolled: more of a row's loads in flight
                    // (measured 0.508 -> 0.489 ms on the long workload)
#pragma unroll 4
                    for (; v + 32 < kv1; v += 64) {
                        const uint4 x0 = lds128(row_raw + 16u * v);
                        const uint4 q0 = lds128(qsm_s + 16u * v);
                        const uint4 x1 = lds128(row_raw + 16u * (v + 32));
                        const uint4 q1 = lds128(qsm_s + 16u * (v + 32));
                        bf16_sq_dot(x0, q0, s0, s1, t0, t1);
                        bf16_sq_dot(x1, q1, s2, s3, t2, t3);
                    }
                    if (v < kv1) {
                        const uint4 x0 = lds128(row_raw + 16u * v);
                        const uint4 q0 = lds128(qsm_s + 16u * v);
                        bf16_sq_dot(x0, q0, s0, s1, t0, t1);
                    }
                } else {
                    for (; v < kv1; v += 32) {
                        uint4 x0 = lds128(row_raw + 16u * v);
                        const uint4 q0 = lds128(qsm_s + 16u * v);
                        // zero the channels of a boundary vector outside [ko, kend)
                        uint32_t w[4] = {x0.x, x0.y, x0.z, x0.w};
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int j = 8 * v + 2 * kk;
                            if (j < ko || j >= kend) w[kk] &= 0xffff0000u;
                            if (j + 1 < ko || j + 1 >= kend) w[kk] &= 0x0000ffffu;
                        }
                        x0 = make_uint4(w[0], w[1], w[2], w[3]);
                        bf16_sq_dot(x0, q0, s0, s1, t0, t1);
                    }
                }
                float part[2] = {(s0 + s1) + (s2 + s3), (t0 + t1) + (t2 + t3)};
                warp_reduce_scatter<2>(part, lane);
                // lane 0 holds the sum of squares, lane 16 the query dot
                if ((lane & 15) == 0) red[(rbuf * red_rows + (lane >> 4) * 32 + r) * kRedPitch] = part[0];
            }
            named_bar_sync(1, nct);
            // Every warp derives the group's logits and softmax update itself
            // (identical inputs and operations, so identical results), which
            // saves a second CTA barrier per group.  Lane l holds row g0 + l.
            float e;
            float corr;
            {
                float ss = 0.0f, qt = 0.0f;
                if (lane < gs) {
                    ss = red[(rbuf * red_rows + lane) * kRedPitch];
                    qt = red[(rbuf * red_rows + 32 + lane) * kRedPitch];
                }
                const float r = rsqrtf(fmaf(ss, inv_r, a.eps));
                const float z = a.scale * r * qt;
                const float m_new = fmaxf(m_run, warp_max(lane < gs ? z : -FLT_MAX));
                e = lane < gs ? __expf(z - m_new) : 0.0f;
                const float esum = warp_sum(e);
                corr = __expf(m_run - m_new);
                l_run = fmaf(l_run, corr, esum);
                m_run = m_new;
                if (warp == 0 && lane < gs) {
                    zall[g0 + lane] = z;
                    rall[g0 + lane] = r;
                }
            }
            rbuf ^= 1;
            // pass 2: rescale the running sum and add this group's weighted
            // rows; each chunk is released once its rows are read
            const float2 corr2 = make_float2(corr, corr);
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) acc[i][kk] = fmul2(acc[i][kk], corr2);
            for (int r0 = 0; r0 < gs; r0 += G) {
                const int rn = min(G, gs - r0);
                uint32_t dep = 0;
                uint32_t rowa = cbase;
#pragma unroll 2
                for (int r = 0; r < rn; ++r) {
                    const float es = __shfl_sync(0xffffffffu, e, r0 + r);
                    const float2 es2 = make_float2(es, es);
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (FULL || col[i] >= 0) {
                            const uint4 xv = lds128(rowa + i * vstep);
                            dep ^= xv.x;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) acc[i][kk] = ffma2(es2, bf2_to_f2(u4_get(xv, kk)), acc[i][kk]);
                        }
                    }
                    rowa += sb;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_after(empty_s + 8u * ck, dep);
                cbase += cb;
                if (++ck == K) {
                    ck = 0;
                    cbase = ring_lo;
                    cphase ^= 1u;
                }
            }
        }
        const float inv_l = 1.0f / l_run;
        const float2 inv_l2 = make_float2(inv_l, inv_l);
        float rho = 1.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) acc[i][kk] = fmul2(acc[i][kk], inv_l2);
        if constexpr (NORM != 0) {
            float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (FULL || col[i] >= 0)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) ss2 = ffma2(acc[i][kk], acc[i][kk], ss2);
            const float ss = warp_sum(ss2.x + ss2.y);
            if (lane == 0) red[(rbuf * red_rows) * kRedPitch + warp] = ss;
            named_bar_sync(1, nct);
            const float tot = red_sum(rbuf, 0);
            rbuf ^= 1;
            rho = rsqrtf(fmaf(tot, inv_d, a.eps));
            if (threadIdx.x == 0) a.o_rstd[n] = rho;
        }
        uint16_t* yrow = a.y + n * static_cast<long long>(a.D);
        float* prow = NORM == 2 ? a.o_pre + n * static_cast<long long>(a.D) : nullptr;
        const float2 rho2 = make_float2(rho, rho);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if ((FULL || col[i] >= 0) && ATTNRES_IN_BOUNDS(n < N && 8 * col[i] + 8 <= a.D, &g_fwd_error)) {
                uint32_t yw[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    yw[kk] = pack_f2(fmul2(fmul2(acc[i][kk], rho2), bf2_to_f2(u4_get(wb[i], kk))));
                st_global_cs_v4(yrow + 8 * col[i], make_uint4(yw[0], yw[1], yw[2], yw[3]));
                if (prow) {
                    st_global_cs_v4(prow + 8 * col[i],
                                    make_uint4(__float_as_uint(acc[i][0].x), __float_as_uint(acc[i][0].y),
                                               __float_as_uint(acc[i][1].x), __float_as_uint(acc[i][1].y)));
                    st_global_cs_v4(prow + 8 * col[i] + 4,
                                    make_uint4(__float_as_uint(acc[i][2].x), __float_as_uint(acc[i][2].y),
                                               __float_as_uint(acc[i][3].x), __float_as_uint(acc[i][3].y)));
                }
            }
        }
        if (warp == 0) {
            __syncwarp();
            for (int s = lane; s < S; s += 32) {
                const float z = zall[s];
                a.alpha[n * S + s] = __expf(z - m_run) * inv_l;
                a.rstd[n * S + s] = rall[s];
                a.logit[n * S + s] = z;
            }
        }
        if (DSL && ++dslot == DSL) {
            dslot = 0;
            dslot_phase ^= 1u;
        }
    }
}

}  // namespace ATTNRES_FWD_NS
}  // namespace attnres
