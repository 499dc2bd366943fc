// attnres_fwd.cu -- forward kernel of the Attention Residuals read operator.
//
// Per token ("Fast Attention Residuals", section "Equation"): key statistics
// of every source's key slice, a softmax over sources of the scaled query
// dot, and the routing-weighted full-width sum; optionally the output
// RMSNorm whose reciprocal RMS is saved for the backward ("[Perf]
// Parallelize AttnRes long-sequence reduction", Summary).
//
// GB300 mapping.  One persistent CTA per SM walks tokens n = blockIdx.x,
// blockIdx.x + gridDim.x, ...  A producer thread streams every source row of
// the token into a ring of shared-memory row slots with 1-D TMA bulk copies
// (one cp.async.bulk per row, completion counted on an mbarrier).  Consumer
// thread t owns the 16-byte column vectors t, t + 32*ncw, ... of every row,
// so each warp reads 512 contiguous bytes per shared load.  Sources are taken
// in groups of GP: one pass over the group's rows accumulates the key
// sum-of-squares and the query dot, a warp reduce-scatter plus one
// cross-warp step yields the group's logits, warp 0 updates the running
// softmax maximum and denominator, and a second pass over the same
// resident rows adds the weighted rows into FP32 registers before the slots
// are released.  The output norm needs one more CTA reduction per token.
// The pre-norm mixture o is written (FP32) only when the caller asks for it.
// This is a bandwidth-bound per-token reduction: no tensor cores.
#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {

namespace {

// First failed wait of any forward launch (0 = none).
__device__ unsigned int g_fwd_error = 0;

struct VecInfo {
    int col;          // 16-byte column vector index, -1 when not owned
    unsigned kmask;   // bit e: channel 8*col+e lies in the key slice
};

__device__ __forceinline__ void advance(int& slot, uint32_t& phase, int slots) {
    if (++slot == slots) {
        slot = 0;
        phase ^= 1u;
    }
}

template <int VPT, int GP>
__global__ void __launch_bounds__(kMaxThreads, 1) attnres_fwd_kernel(const __grid_constant__ FwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int slots = a.slots;
    const SmemLayout L = make_layout(slots, a.slot_bytes, ncw, a.s_pad, false);
    unsigned char* ring = smem + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* zall = reinterpret_cast<float*>(smem + L.coef);
    float* rall = zall + a.s_pad;
    float* coef = rall + a.s_pad;  // [2][64]: e_s (s < 32), corr at 32, 1/l at 33
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int S = a.S;

    if (threadIdx.x == 0) {
        for (int k = 0; k < slots; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = static_cast<uint32_t>(a.D) * 2u;
            int slot = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (long long n = blockIdx.x; n < N && !*abort_flag; n += gridDim.x) {
                for (int s = 0; s < S; ++s) {
                    if (!mbar_wait(empty + slot, phase ^ 1u, abort_flag, &g_fwd_error, kSiteFwdProducer)) break;
                    mbar_arrive_expect_tx(full + slot, bytes);
                    const unsigned char* src =
                        static_cast<const unsigned char*>(a.src[s]) + (n * a.src_ld) * 2;
                    tma_load_1d(ring + static_cast<size_t>(slot) * a.slot_bytes, src, bytes,
                                full + slot, pol);
                    ++issued;
                    advance(slot, phase, slots);
                }
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA can exit.
                for (int k = 0; k < slots && k < issued; ++k) {
                    const long long fills = (issued - 1 - k) / slots + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + k, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_fwd_error, kSiteDrain);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = a.D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    VecInfo vi[VPT];
    float qf[VPT][8];
    float wf[VPT][8];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * nct;
        vi[i].col = c < ncv ? c : -1;
        unsigned m = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * c + e;
            const bool in_key = vi[i].col >= 0 && j >= ko && j < kend;
            m |= in_key ? (1u << e) : 0u;
            qf[i][e] = in_key ? bf16_bits_to_float(a.q[j - ko]) : 0.0f;
            wf[i][e] = (a.out_norm && vi[i].col >= 0) ? bf16_bits_to_float(a.w_o[j]) : 1.0f;
        }
        vi[i].kmask = m;
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);
    const float inv_d = 1.0f / static_cast<float>(a.D);
    constexpr int K2 = 2 * GP;
    constexpr int SH = 5 - log2_const<K2>();

    int slot = 0;
    uint32_t phase = 0;
    int rbuf = 0;

    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        float acc[VPT][8];
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
        float m_run = -FLT_MAX;  // meaningful in warp 0
        float l_run = 0.0f;
        int cbuf = 0;

        for (int g0 = 0; g0 < S; g0 += GP) {
            const int gs = min(GP, S - g0);
            const int gslot = slot;
            const uint32_t gphase = phase;
            float part[K2];
#pragma unroll
            for (int k = 0; k < K2; ++k) part[k] = 0.0f;
            // pass 1: key sum of squares and query dot per source
#pragma unroll
            for (int s = 0; s < GP; ++s) {
                if (s < gs) {
                    mbar_wait(full + slot, phase, abort_flag, &g_fwd_error, kSiteFwdConsumer);
                    const unsigned char* row = ring + static_cast<size_t>(slot) * a.slot_bytes;
                    float ss = 0.0f, qt = 0.0f;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (vi[i].kmask) {
                            float x[8];
                            unpack8(ld_shared_v4(row + vi[i].col * 16), x);
                            if (vi[i].kmask == 0xffu) {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    ss = fmaf(x[e], x[e], ss);
                                    qt = fmaf(qf[i][e], x[e], qt);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float xm = ((vi[i].kmask >> e) & 1u) ? x[e] : 0.0f;
                                    ss = fmaf(xm, xm, ss);
                                    qt = fmaf(qf[i][e], xm, qt);
                                }
                            }
                        }
                    }
                    part[s] = ss;
                    part[GP + s] = qt;
                    advance(slot, phase, slots);
                }
            }
            warp_reduce_scatter<K2>(part, lane);
            if ((lane & ((1 << SH) - 1)) == 0)
                red[(rbuf * ncw + warp) * kReduceStride + (lane >> SH)] = part[0];
            named_bar_sync(1, nct);
            if (warp == 0) {
                float ss = 0.0f, qt = 0.0f;
                if (lane < gs) {
                    for (int w = 0; w < ncw; ++w) {
                        ss += red[(rbuf * ncw + w) * kReduceStride + lane];
                        qt += red[(rbuf * ncw + w) * kReduceStride + GP + lane];
                    }
                }
                const float r = rsqrtf(fmaf(ss, inv_r, a.eps));
                const float z = a.scale * r * qt;
                const float m_new = fmaxf(m_run, warp_max(lane < gs ? z : -FLT_MAX));
                const float e = lane < gs ? __expf(z - m_new) : 0.0f;
                const float esum = warp_sum(e);
                const float corr = __expf(m_run - m_new);
                l_run = fmaf(l_run, corr, esum);
                m_run = m_new;
                if (lane < gs) {
                    coef[cbuf * 64 + lane] = e;
                    zall[g0 + lane] = z;
                    rall[g0 + lane] = r;
                }
                if (lane == 0) {
                    coef[cbuf * 64 + 32] = corr;
                    coef[cbuf * 64 + 33] = 1.0f / l_run;
                }
            }
            rbuf ^= 1;
            named_bar_sync(1, nct);
            // pass 2: rescale the running sum and add this group's weighted rows
            const float corr = coef[cbuf * 64 + 32];
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] *= corr;
            slot = gslot;
            phase = gphase;
#pragma unroll
            for (int s = 0; s < GP; ++s) {
                if (s < gs) {
                    const float es = coef[cbuf * 64 + s];
                    const unsigned char* row = ring + static_cast<size_t>(slot) * a.slot_bytes;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (vi[i].col >= 0) {
                            float x[8];
                            unpack8(ld_shared_v4(row + vi[i].col * 16), x);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(es, x[e], acc[i][e]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty + slot);
                    advance(slot, phase, slots);
                }
            }
            cbuf ^= 1;
        }
        const float inv_l = coef[(cbuf ^ 1) * 64 + 33];
        float rho = 1.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] *= inv_l;
        if (a.out_norm) {
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (vi[i].col >= 0)
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(acc[i][e], acc[i][e], ss);
            ss = warp_sum(ss);
            if (lane == 0) red[(rbuf * ncw + warp) * kReduceStride] = ss;
            named_bar_sync(1, nct);
            float tot = 0.0f;
            for (int w = 0; w < ncw; ++w) tot += red[(rbuf * ncw + w) * kReduceStride];
            rbuf ^= 1;
            rho = rsqrtf(fmaf(tot, inv_d, a.eps));
            if (threadIdx.x == 0) a.o_rstd[n] = rho;
        }
        uint16_t* yrow = a.y + n * static_cast<long long>(a.D);
        float* prow = a.o_pre ? a.o_pre + n * static_cast<long long>(a.D) : nullptr;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (vi[i].col >= 0) {
                float yv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) yv[e] = acc[i][e] * rho * wf[i][e];
                st_global_cs_v4(yrow + 8 * vi[i].col, pack8(yv));
                if (prow) {
                    const uint4 lo = make_uint4(__float_as_uint(acc[i][0]), __float_as_uint(acc[i][1]),
                                                __float_as_uint(acc[i][2]), __float_as_uint(acc[i][3]));
                    const uint4 hi = make_uint4(__float_as_uint(acc[i][4]), __float_as_uint(acc[i][5]),
                                                __float_as_uint(acc[i][6]), __float_as_uint(acc[i][7]));
                    st_global_cs_v4(prow + 8 * vi[i].col, lo);
                    st_global_cs_v4(prow + 8 * vi[i].col + 4, hi);
                }
            }
        }
        if (warp == 0) {
            const float inv_lw = 1.0f / l_run;
            for (int s = lane; s < S; s += 32) {
                const float z = zall[s];
                a.alpha[n * S + s] = __expf(z - m_run) * inv_lw;
                a.rstd[n * S + s] = rall[s];
                a.logit[n * S + s] = z;
            }
        }
    }
}

template <int VPT, int GP>
cudaError_t launch_fwd_t(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_fwd_kernel<VPT, GP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_fwd));
    if (err != cudaSuccess) return err;
    kern<<<plan.grid, (plan.ncw + 1) * 32, plan.smem_fwd, stream>>>(a);
    return cudaGetLastError();
}

template <int VPT>
cudaError_t dispatch_gp(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    switch (plan.gp_fwd) {
        case 2: return launch_fwd_t<VPT, 2>(plan, a, stream);
        case 4: return launch_fwd_t<VPT, 4>(plan, a, stream);
        case 8: return launch_fwd_t<VPT, 8>(plan, a, stream);
        case 16: return launch_fwd_t<VPT, 16>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace

unsigned take_fwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fwd_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_fwd_error, &zero, sizeof zero);
    return v;
}

cudaError_t launch_fwd(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    switch (plan.vpt) {
        case 1: return dispatch_gp<1>(plan, a, stream);
        case 2: return dispatch_gp<2>(plan, a, stream);
        case 4: return dispatch_gp<4>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace attnres
