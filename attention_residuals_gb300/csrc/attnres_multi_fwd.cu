// attnres_multi_fwd.cu -- forward kernel of the multi-query read.
//
// "Fast Attention Residuals", section "Multi-query AttnRes": the same
// sources are read with M queries (1 <= M <= 16); each query has its own
// source weights and its own full-width output.  Per token and query m
// (section "Equation"):
//   r_s = 1/sqrt(mean(t_s^2) + eps),  z_ms = scale * r_s * <t_s, q_m>,
//   alpha_m = softmax_s(z_m),          y_m = sum_s alpha_ms v_s.
// The key statistics r_s do not depend on the query, so they are formed once.
//
// GB300 mapping.  One persistent CTA per SM; a producer thread streams every
// source row of a token into a ring of shared-memory chunks with 1-D TMA
// bulk copies, and the token stays resident while all M queries are served,
// so each source row is read from HBM once for all M outputs.
//   pass 1: one warp per source row; lanes stride over the key vectors and
//           accumulate the key sum of squares and the M query dots with
//           mixed-precision bf16 FMAs (queries in shared memory), then one
//           reduce-scatter per four queries gives the row's totals.
//   softmax: after one CTA barrier, one warp per query forms its logits and
//           weights (lanes over sources) into a shared table.
//   pass 2: after a second barrier, thread t owns fixed 16-byte column
//           vectors and accumulates MB outputs at a time in FP32 registers
//           (packed FFMA2), so each source row is unpacked once per MB
//           queries; the last block releases each chunk once read.
// Bandwidth-bound per-token reductions: no tensor cores.
#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {

namespace {

// First failed wait of any multi-query forward launch (0 = none).
__device__ unsigned int g_multi_error = 0;

template <int VPT, int MB>
__global__ void __launch_bounds__(kMaxThreads, 1) attnres_multi_fwd_kernel(const __grid_constant__ MultiFwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = a.chunks;
    const int G = a.rows;
    const int S = a.S;
    const int M = a.M;
    const int s_pad = a.s_pad, m_pad = a.m_pad;
    const MultiLayout L = make_multi_layout(K, G, a.slot_bytes, M, 0, s_pad, m_pad, a.nkv, 0, false);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    float* ss_t = reinterpret_cast<float*>(smem + L.tab);  // [s_pad]
    float* dot_t = ss_t + s_pad;                           // [m_pad][s_pad]
    float* al_t = dot_t + m_pad * s_pad;                   // [s_pad][m_pad]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const uint32_t sb = static_cast<uint32_t>(a.slot_bytes);
    const uint32_t cb = static_cast<uint32_t>(G) * sb;
    const int cpt = (S + G - 1) / G;  // chunks per token

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    // weights of padded queries stay zero
    for (int i = threadIdx.x; i < s_pad * m_pad; i += blockDim.x) al_t[i] = 0.0f;
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = static_cast<uint32_t>(a.D) * 2u;
            unsigned char* ring = smem + L.ring;
            int k = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (long long n = blockIdx.x; n < N && !*abort_flag; n += gridDim.x) {
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
            if (*abort_flag) {
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
    const uint32_t kwb = static_cast<uint32_t>(nkv) * 16u;  // bytes per query row in shared memory
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
    {
        // queries by key channel: row m holds channels 8*kv0 .. 8*(kv0+nkv)
        uint16_t* qsm = reinterpret_cast<uint16_t*>(smem + L.qsm);
        const int kw = nkv * 8;
        for (int i = threadIdx.x; i < m_pad * kw; i += nct) {
            const int m = i / kw;
            const int c = 8 * kv0 + (i - m * kw);
            qsm[i] = (m < M && c >= ko && c < kend) ? a.q[static_cast<long long>(m) * a.R + (c - ko)]
                                                    : static_cast<uint16_t>(0);
        }
    }
    named_bar_sync(1, nct);
    const bool key_aligned = ((ko | kend) & 7) == 0;

    int ck = 0;
    uint32_t cphase = 0;
    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        {
            int k = ck;
            uint32_t ph = cphase;
            for (int c = 0; c < cpt; ++c) {
                mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_multi_error, kSiteFwdConsumer);
                if (++k == K) {
                    k = 0;
                    ph ^= 1u;
                }
            }
        }
        // pass 1: one warp per row, four queries per reduce-scatter
        for (int r = warp; r < S; r += ncw) {
            int kc = ck + r / G;
            if (kc >= K) kc -= K;
            const uint32_t row = ring_raw + static_cast<uint32_t>(kc) * cb +
                                 static_cast<uint32_t>(r % G) * sb + 16u * static_cast<uint32_t>(kv0);
            for (int qb = 0; qb < m_pad; qb += 4) {
                float s0 = 0.0f, s1 = 0.0f;
                float t[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) t[j][0] = t[j][1] = 0.0f;
                const uint32_t qrow = qsm_s + static_cast<uint32_t>(qb) * kwb;
                for (int v = lane; v < nkv; v += 32) {
                    uint4 x = lds128(row + 16u * v);
                    if (!key_aligned) x = mask_bf16x8(x, 8 * (kv0 + v), ko, kend);
                    if (qb == 0) bf16_sq8(x, s0, s1);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 qv = lds128(qrow + static_cast<uint32_t>(j) * kwb + 16u * v);
                        bf16_dot8(x, qv, t[j][0], t[j][1]);
                    }
                }
                float part[8] = {s0 + s1, t[0][0] + t[0][1], t[1][0] + t[1][1], t[2][0] + t[2][1],
                                 t[3][0] + t[3][1], 0.0f, 0.0f, 0.0f};
                warp_reduce_scatter<8>(part, lane);
                if ((lane & 3) == 0) {
                    const int e = lane >> 2;
                    if (e == 0) {
                        if (qb == 0) ss_t[r] = part[0];
                    } else if (e <= 4) {
                        dot_t[(qb + e - 1) * s_pad + r] = part[0];
                    }
                }
            }
        }
        named_bar_sync(1, nct);
        // softmax: one warp per query, lanes over sources
        for (int m = warp; m < M; m += ncw) {
            float z[4], rr[4];
            float mx = -FLT_MAX;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = lane + 32 * i;
                z[i] = -FLT_MAX;
                rr[i] = 0.0f;
                if (s < S) {
                    rr[i] = rsqrtf(fmaf(ss_t[s], inv_r, a.eps));
                    z[i] = a.scale * rr[i] * dot_t[m * s_pad + s];
                    mx = fmaxf(mx, z[i]);
                }
            }
            mx = warp_max(mx);
            float e[4];
            float es = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                e[i] = (lane + 32 * i < S) ? __expf(z[i] - mx) : 0.0f;
                es += e[i];
            }
            const float inv_l = 1.0f / warp_sum(es);
            float* arow = a.alpha + (n * M + m) * S;
            float* zrow = a.logit + (n * M + m) * S;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = lane + 32 * i;
                if (s < S) {
                    const float al = e[i] * inv_l;
                    al_t[s * m_pad + m] = al;
                    arow[s] = al;
                    zrow[s] = z[i];
                    if (m == 0) a.rstd[n * S + s] = rr[i];
                }
            }
        }
        named_bar_sync(1, nct);
        // pass 2: MB outputs at a time; the last block releases the chunks
        for (int mb = 0; mb < M; mb += MB) {
            const bool last = mb + MB >= M;
            float2 acc[MB][VPT][4];
#pragma unroll
            for (int j = 0; j < MB; ++j)
#pragma unroll
                for (int i = 0; i < VPT; ++i)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) acc[j][i][kk] = make_float2(0.0f, 0.0f);
            int kc = ck;
            for (int r0 = 0; r0 < S; r0 += G) {
                const int rn = min(G, S - r0);
                uint32_t dep = 0;
                uint32_t rowa = ring_lo + static_cast<uint32_t>(kc) * cb;
                for (int r = 0; r < rn; ++r) {
                    const float* al_row = al_t + (r0 + r) * m_pad + mb;
                    float2 w2[MB];
#pragma unroll
                    for (int j = 0; j < MB; ++j) w2[j] = make_float2(al_row[j], al_row[j]);
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (col[i] >= 0) {
                            const uint4 xv = lds128(rowa + i * vstep);
                            dep ^= xv.x;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const float2 x2 = bf2_to_f2(u4_get(xv, kk));
#pragma unroll
                                for (int j = 0; j < MB; ++j) acc[j][i][kk] = ffma2(w2[j], x2, acc[j][i][kk]);
                            }
                        }
                    }
                    rowa += sb;
                }
                if (last) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_after(empty_s + 8u * kc, dep);
                }
                if (++kc == K) kc = 0;
            }
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                if (mb + j < M) {
                    uint16_t* yrow = a.y + static_cast<long long>(mb + j) * a.y_ms + n * a.y_ns;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (col[i] >= 0) {
                            st_global_cs_v4(yrow + 8 * col[i],
                                            make_uint4(pack_f2(acc[j][i][0]), pack_f2(acc[j][i][1]),
                                                       pack_f2(acc[j][i][2]), pack_f2(acc[j][i][3])));
                        }
                    }
                }
            }
        }
        for (int c = 0; c < cpt; ++c) {
            if (++ck == K) {
                ck = 0;
                cphase ^= 1u;
            }
        }
    }
}

template <int VPT, int MB>
cudaError_t launch_t(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_multi_fwd_kernel<VPT, MB>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_fwd));
    if (err != cudaSuccess) return err;
    kern<<<plan.grid, (plan.ncw + 1) * 32, plan.smem_fwd, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

unsigned take_multi_fwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_error, &zero, sizeof zero);
    return v;
}

cudaError_t launch_multi_fwd(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    const int key = plan.vpt * 10 + plan.mb_f;
    switch (key) {
        case 11: return launch_t<1, 1>(plan, a, stream);
        case 12: return launch_t<1, 2>(plan, a, stream);
        case 14: return launch_t<1, 4>(plan, a, stream);
        case 21: return launch_t<2, 1>(plan, a, stream);
        case 22: return launch_t<2, 2>(plan, a, stream);
        case 24: return launch_t<2, 4>(plan, a, stream);
        case 41: return launch_t<4, 1>(plan, a, stream);
        case 42: return launch_t<4, 2>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace attnres
