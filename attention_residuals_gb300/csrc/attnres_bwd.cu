// attnres_bwd.cu -- backward kernel and dq/dw_o finalize of the Attention
// Residuals read operator.
//
// Per token, with the forward's saved alpha, rstd, logit (and o_rstd when the
// output RMSNorm is on; "[Perf] Parallelize AttnRes long-sequence
// reduction", Summary):
//   out-norm:  o = sum_s alpha_s v_s (rebuilt in FP32, or the caller's FP32
//              copy), yhat = o * o_rstd, dw_o += dy * yhat, g = dy * w_o,
//              do = o_rstd * (g - yhat * <g, yhat> / D);   else do = dy
//   da_s  = <do, v_s>,   delta = sum_s alpha_s da_s,  dz_s = alpha_s (da_s - delta)
//   dv_s  = alpha_s do  +  on key channels: c1_s q + c2_s t_s
//           with c1_s = rstd_s scale dz_s,  c2_s = -rstd_s^2 dz_s z_s / R
//   dq   += sum_s c1_s t_s
// (chain rule through "Fast Attention Residuals", section "Equation").
//
// GB300 mapping.  As in the forward, one persistent CTA per SM, a producer
// thread filling a shared-memory row ring with 1-D TMA copies, and consumer
// threads that own fixed 16-byte column vectors.  Per token the ring
// receives dy and the S source rows.  When the S rows fit in the ring
// ("resident"), each source row is read from HBM once: the o rebuild (with
// the output norm), the dot pass and the write pass all read it from shared
// memory.  Otherwise the producer streams the rows once per pass (served
// from L2 when it still holds them), and the write pass gets key slices only.  The saved per-token statistics arrive
// through small cp.async copies into a separate 4-deep ring.
//
// dq and dw_o: every consumer thread owns the same columns for every token,
// so its dq/dw_o contributions accumulate in registers across all of the
// CTA's tokens; each CTA writes one FP32 partial row.  For long N ("four
// programs accumulate FP32 partials and a separate kernel finalizes", the
// page's split-N path) a finalize kernel sums the partial rows in CTA order.
// For short N the sum finishes inside this kernel: the last CTA of each
// group of kGroupTicket CTAs (atomic ticket, no waiting) adds its group's
// rows in order, and the last group adds the group sums in order.  Both
// orders are fixed, so the results are bitwise reproducible.
#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {
namespace {

// First failed wait of any backward launch (0 = none).
__device__ unsigned int g_bwd_error = 0;

struct VecInfo {
    int col;
    unsigned kmask;
};

__device__ __forceinline__ void advance(int& slot, uint32_t& phase, int slots) {
    if (++slot == slots) {
        slot = 0;
        phase ^= 1u;
    }
}

__device__ __forceinline__ float ldcg_f32(const float* p) { return __ldcg(p); }

template <int VPT, int GP>
__global__ void __launch_bounds__(kMaxThreads, 1) attnres_bwd_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int slots = a.slots;
    const int s_pad = a.s_pad;
    const SmemLayout L = make_layout(slots, a.slot_bytes, ncw, s_pad, true);
    unsigned char* ring = smem + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* tok = reinterpret_cast<float*>(smem + L.tok);  // [kTokSlots][3*s_pad + 4]
    float* cA = reinterpret_cast<float*>(smem + L.coef);  // alpha_s
    float* c1 = cA + s_pad;
    float* c2 = c1 + s_pad;
    float* da_all = c2 + s_pad;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    volatile int* ticket_flag = abort_flag + 1;
    const int tstride = 3 * s_pad + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int S = a.S;
    const int D = a.D;

    if (threadIdx.x == 0) {
        for (int k = 0; k < slots; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        for (int k = 0; k < kTokSlots; ++k) {
            mbar_init(tfull + k, 32);
            mbar_init(tempty + k, 1);
        }
        *abort_flag = 0;
        *ticket_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
        // Key slice of the second pass: only the key channels when they
        // start and end on 16-byte boundaries, else the whole row.
        const bool key_only = ((a.ko & 7) == 0) && ((a.R & 7) == 0);
        const uint32_t key_off_b = key_only ? static_cast<uint32_t>(a.ko) * 2u : 0u;
        const uint32_t key_bytes = key_only ? static_cast<uint32_t>(a.R) * 2u : row_bytes;
        int slot = 0;
        uint32_t phase = 0;
        int ts = 0;
        uint32_t tphase = 0;
        long long issued = 0;
        for (long long n = blockIdx.x; n < N; n += gridDim.x) {
            if (*abort_flag) break;
            // token statistics -> tok[ts] (all 32 lanes arrive on tfull)
            mbar_wait(tempty + ts, tphase ^ 1u, abort_flag, &g_bwd_error, kSiteBwdProducer);
            float* dst = tok + ts * tstride;
            for (int e = lane; e < S; e += 32) {
                cp_async_4(dst + e, a.alpha + n * S + e);
                cp_async_4(dst + s_pad + e, a.rstd + n * S + e);
                cp_async_4(dst + 2 * s_pad + e, a.logit + n * S + e);
            }
            if (a.out_norm && lane == 0) cp_async_4(dst + 3 * s_pad, a.o_rstd + n);
            cp_async_arrive_noinc(tfull + ts);
            if (++ts == kTokSlots) {
                ts = 0;
                tphase ^= 1u;
            }
            if (lane == 0) {
                // Row schedule of one token: dy; then, when o must be rebuilt
                // from streamed rows, S rows for that pass; S rows for the dot
                // pass (in resident mode these also serve the other passes);
                // when streaming, S key slices for the write pass.
                const int pass_a = (a.out_norm && !a.o_pre && !a.resident) ? S : 0;
                const int pass_c = a.resident ? 0 : S;
                const int nrows = 1 + pass_a + S + pass_c;
                for (int r = 0; r < nrows; ++r) {
                    const unsigned char* src;
                    uint32_t off = 0, bytes = row_bytes;
                    if (r == 0) {
                        src = reinterpret_cast<const unsigned char*>(a.dy + n * D);
                    } else {
                        int s = r - 1;
                        if (s >= pass_a) s -= pass_a;  // rows of the o pass come first
                        if (r - 1 >= pass_a + S) {      // write-pass key slices
                            off = key_off_b;
                            bytes = key_bytes;
                        }
                        if (s >= S) s -= S;
                        src = static_cast<const unsigned char*>(a.src[s]) + (n * a.src_ld) * 2 + off;
                    }
                    if (!mbar_wait(empty + slot, phase ^ 1u, abort_flag, &g_bwd_error, kSiteBwdProducer)) break;
                    mbar_arrive_expect_tx(full + slot, bytes);
                    tma_load_1d(ring + static_cast<size_t>(slot) * a.slot_bytes + off, src, bytes,
                                full + slot, pol);
                    ++issued;
                    advance(slot, phase, slots);
                }
            }
            __syncwarp();
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0 && *abort_flag) {
            for (int k = 0; k < slots && k < issued; ++k) {
                const long long fills = (issued - 1 - k) / slots + 1;
                volatile int no_abort = 0;
                mbar_wait(full + k, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_bwd_error, kSiteDrain);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    VecInfo vi[VPT];
    float qf[VPT][8];
    float wf[VPT][8];
    float dq_acc[VPT][8];
    float dw_acc[VPT][8];
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
            qf[i][e] = in_key ? a.scale * bf16_bits_to_float(a.q[j - ko]) : 0.0f;
            wf[i][e] = (a.out_norm && vi[i].col >= 0) ? bf16_bits_to_float(a.w_o[j]) : 1.0f;
            dq_acc[i][e] = 0.0f;
            dw_acc[i][e] = 0.0f;
        }
        vi[i].kmask = m;
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);
    const float inv_d = 1.0f / static_cast<float>(D);
    constexpr int SH = 5 - log2_const<GP>();

    int slot = 0;
    uint32_t phase = 0;
    int ts = 0;
    uint32_t tphase = 0;
    int rbuf = 0;

    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        mbar_wait(tfull + ts, tphase, abort_flag, &g_bwd_error, kSiteBwdTokStat);
        const float* tk = tok + ts * tstride;

        // ---- gradient wrt the mixture o (kept in registers)
        float dout[VPT][8];
        const int dy_slot = slot;
        mbar_wait(full + slot, phase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
        advance(slot, phase, slots);
        const unsigned char* dy_row = ring + static_cast<size_t>(dy_slot) * a.slot_bytes;
        if (a.out_norm) {
            // o = sum_s alpha_s v_s in FP32: from the caller's saved copy, or
            // rebuilt from the source rows (resident: the rows the dot pass
            // uses next; streaming: a dedicated pass of rows).
            float o[VPT][8];
            if (a.o_pre) {
                const float* prow = a.o_pre + n * static_cast<long long>(D);
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    if (vi[i].col >= 0) {
                        const uint4 lo = ld_global_nc_v4(prow + 8 * vi[i].col);
                        const uint4 hi = ld_global_nc_v4(prow + 8 * vi[i].col + 4);
                        o[i][0] = __uint_as_float(lo.x); o[i][1] = __uint_as_float(lo.y);
                        o[i][2] = __uint_as_float(lo.z); o[i][3] = __uint_as_float(lo.w);
                        o[i][4] = __uint_as_float(hi.x); o[i][5] = __uint_as_float(hi.y);
                        o[i][6] = __uint_as_float(hi.z); o[i][7] = __uint_as_float(hi.w);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < VPT; ++i)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[i][e] = 0.0f;
                int aslot = slot;
                uint32_t aphase = phase;
                for (int s = 0; s < S; ++s) {
                    mbar_wait(full + aslot, aphase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
                    const unsigned char* row = ring + static_cast<size_t>(aslot) * a.slot_bytes;
                    const float al = tk[s];
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (vi[i].col >= 0) {
                            float x[8];
                            unpack8(ld_shared_v4(row + vi[i].col * 16), x);
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[i][e] = fmaf(al, x[e], o[i][e]);
                        }
                    }
                    if (!a.resident) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(empty + aslot);
                    }
                    advance(aslot, aphase, slots);
                }
                if (!a.resident) {  // the streamed o-pass rows are consumed
                    slot = aslot;
                    phase = aphase;
                }
            }
            const float rho = tk[3 * s_pad];
            float gy = 0.0f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (vi[i].col >= 0) {
                    float g[8];
                    unpack8(ld_shared_v4(dy_row + vi[i].col * 16), g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float yh = o[i][e] * rho;
                        o[i][e] = yh;
                        dw_acc[i][e] = fmaf(g[e], yh, dw_acc[i][e]);
                        g[e] *= wf[i][e];
                        gy = fmaf(g[e], yh, gy);
                        dout[i][e] = g[e];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) dout[i][e] = 0.0f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + dy_slot);
            gy = warp_sum(gy);
            if (lane == 0) red[(rbuf * ncw + warp) * kReduceStride] = gy;
            named_bar_sync(1, nct);
            float tot = 0.0f;
            for (int w = 0; w < ncw; ++w) tot += red[(rbuf * ncw + w) * kReduceStride];
            rbuf ^= 1;
            const float cg = tot * inv_d;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) dout[i][e] = rho * fmaf(-o[i][e], cg, dout[i][e]);
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (vi[i].col >= 0) {
                    unpack8(ld_shared_v4(dy_row + vi[i].col * 16), dout[i]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) dout[i][e] = 0.0f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + dy_slot);
        }

        // ---- dot pass: da_s = <do, v_s>
        const int v_slot0 = slot;
        const uint32_t v_phase0 = phase;
        for (int g0 = 0; g0 < S; g0 += GP) {
            const int gs = min(GP, S - g0);
            float part[GP];
#pragma unroll
            for (int k = 0; k < GP; ++k) part[k] = 0.0f;
#pragma unroll
            for (int s = 0; s < GP; ++s) {
                if (s < gs) {
                    mbar_wait(full + slot, phase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
                    const unsigned char* row = ring + static_cast<size_t>(slot) * a.slot_bytes;
                    float d = 0.0f;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (vi[i].col >= 0) {
                            float x[8];
                            unpack8(ld_shared_v4(row + vi[i].col * 16), x);
#pragma unroll
                            for (int e = 0; e < 8; ++e) d = fmaf(dout[i][e], x[e], d);
                        }
                    }
                    part[s] = d;
                    if (!a.resident) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(empty + slot);
                    }
                    advance(slot, phase, slots);
                }
            }
            warp_reduce_scatter<GP>(part, lane);
            if ((lane & ((1 << SH) - 1)) == 0)
                red[(rbuf * ncw + warp) * kReduceStride + (lane >> SH)] = part[0];
            named_bar_sync(1, nct);
            if (warp == 0 && lane < gs) {
                float d = 0.0f;
                for (int w = 0; w < ncw; ++w) d += red[(rbuf * ncw + w) * kReduceStride + lane];
                da_all[g0 + lane] = d;
            }
            rbuf ^= 1;
        }

        // ---- per-source coefficients (warp 0)
        if (warp == 0) {
            __syncwarp();
            float part_delta = 0.0f;
            for (int s = lane; s < S; s += 32) part_delta = fmaf(tk[s], da_all[s], part_delta);
            const float delta = warp_sum(part_delta);
            for (int s = lane; s < S; s += 32) {
                const float al = tk[s];
                const float r = tk[s_pad + s];
                const float z = tk[2 * s_pad + s];
                const float dz = al * (da_all[s] - delta);
                cA[s] = al;
                c1[s] = r * dz;  // qf carries `scale`, so c1 * qf = rstd * scale * dz * q
                c2[s] = -(r * r) * dz * z * inv_r;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + ts);
        }
        if (++ts == kTokSlots) {
            ts = 0;
            tphase ^= 1u;
        }
        named_bar_sync(1, nct);

        // ---- write pass: dv_s rows and dq contributions
        if (a.resident) {
            slot = v_slot0;
            phase = v_phase0;
        }
        for (int s = 0; s < S; ++s) {
            if (!a.resident) mbar_wait(full + slot, phase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
            const unsigned char* row = ring + static_cast<size_t>(slot) * a.slot_bytes;
            const float al = cA[s];
            const float k1 = c1[s];
            const float k2 = c2[s];
            uint16_t* drow = static_cast<uint16_t*>(a.dsrc[s]) + n * a.dsrc_ld;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (vi[i].col >= 0) {
                    float dv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) dv[e] = al * dout[i][e];
                    if (vi[i].kmask) {
                        float x[8];
                        unpack8(ld_shared_v4(row + vi[i].col * 16), x);
                        if (vi[i].kmask != 0xffu) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] = ((vi[i].kmask >> e) & 1u) ? x[e] : 0.0f;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            dv[e] = fmaf(k1, qf[i][e], fmaf(k2, x[e], dv[e]));
                            dq_acc[i][e] = fmaf(k1, x[e], dq_acc[i][e]);
                        }
                    }
                    st_global_cs_v4(drow + 8 * vi[i].col, pack8(dv));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + slot);
            advance(slot, phase, slots);
        }
    }

    // ---------------------------------------------- per-CTA partial sums
    const int R = a.R;
    const int Dw = a.out_norm ? D : 0;
    const int W = R + Dw;
    float* my_part = a.part + static_cast<size_t>(blockIdx.x) * W;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        if (vi[i].col >= 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * vi[i].col + e;
                // dq = scale * sum_s dz_s k_s = scale * sum_s c1_s t_s
                if ((vi[i].kmask >> e) & 1u) my_part[j - ko] = a.scale * dq_acc[i][e];
                if (a.out_norm) my_part[R + j] = dw_acc[i][e];
            }
        }
    }
    if (a.split) return;

    // ------------------------------ in-kernel two-level ordered reduction
    __threadfence();
    named_bar_sync(1, nct);
    const int grp = blockIdx.x / kGroupTicket;
    const int g_first = grp * kGroupTicket;
    const int g_size = min(kGroupTicket, static_cast<int>(gridDim.x) - g_first);
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&a.tickets[grp], 1u);
        *ticket_flag = (t == static_cast<unsigned>(g_size - 1)) ? 1 : 0;
    }
    named_bar_sync(1, nct);
    if (!*ticket_flag) return;
    __threadfence();
    float* gsum = a.gpart + static_cast<size_t>(grp) * W;
    for (int c = threadIdx.x; c < W; c += nct) {
        float acc = 0.0f;
        for (int b = 0; b < g_size; ++b) acc += ldcg_f32(a.part + static_cast<size_t>(g_first + b) * W + c);
        gsum[c] = acc;
    }
    __threadfence();
    named_bar_sync(1, nct);
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&a.tickets[a.ngroups], 1u);
        *ticket_flag = (t == static_cast<unsigned>(a.ngroups - 1)) ? 2 : 0;
    }
    named_bar_sync(1, nct);
    if (*ticket_flag != 2) return;
    __threadfence();
    for (int c = threadIdx.x; c < W; c += nct) {
        float acc = 0.0f;
        for (int g = 0; g < a.ngroups; ++g) acc += ldcg_f32(a.gpart + static_cast<size_t>(g) * W + c);
        const uint16_t h = static_cast<uint16_t>(pack_bf16x2(acc, 0.0f) & 0xffffu);
        if (c < R) {
            a.dq[c] = h;
            if (a.dq_f32) a.dq_f32[c] = acc;
        } else {
            a.dw_o[c - R] = h;
            if (a.dw_o_f32) a.dw_o_f32[c - R] = acc;
        }
    }
}

// Finalize for the split-N path: column c of dq/dw_o is the sum of the
// per-CTA partial rows taken in CTA order.
__global__ void __launch_bounds__(256) attnres_finalize_kernel(const float* __restrict__ part, int P, int R,
                                                               int W, uint16_t* dq, float* dq_f32,
                                                               uint16_t* dw_o, float* dw_o_f32) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= W) return;
    float acc = 0.0f;
    int b = 0;
    for (; b + 8 <= P; b += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(part + static_cast<size_t>(b + k) * W + c);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc += v[k];
    }
    for (; b < P; ++b) acc += __ldcg(part + static_cast<size_t>(b) * W + c);
    const uint16_t h = static_cast<uint16_t>(pack_bf16x2(acc, 0.0f) & 0xffffu);
    if (c < R) {
        dq[c] = h;
        if (dq_f32) dq_f32[c] = acc;
    } else {
        dw_o[c - R] = h;
        if (dw_o_f32) dw_o_f32[c - R] = acc;
    }
}

template <int VPT, int GP>
cudaError_t launch_bwd_t(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_bwd_kernel<VPT, GP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_bwd));
    if (err != cudaSuccess) return err;
    kern<<<plan.grid, (plan.ncw + 1) * 32, plan.smem_bwd, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess || !plan.split) return err;
    const int W = a.R + (a.out_norm ? a.D : 0);
    attnres_finalize_kernel<<<(W + 255) / 256, 256, 0, stream>>>(a.part, plan.grid, a.R, W, a.dq,
                                                                 a.dq_f32, a.dw_o, a.dw_o_f32);
    return cudaGetLastError();
}

template <int VPT>
cudaError_t dispatch_gp(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    switch (plan.gp_bwd) {
        case 2: return launch_bwd_t<VPT, 2>(plan, a, stream);
        case 4: return launch_bwd_t<VPT, 4>(plan, a, stream);
        case 8: return launch_bwd_t<VPT, 8>(plan, a, stream);
        case 16: return launch_bwd_t<VPT, 16>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace

unsigned take_bwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof zero);
    return v;
}

cudaError_t launch_bwd(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    switch (plan.vpt) {
        case 1: return dispatch_gp<1>(plan, a, stream);
        case 2: return dispatch_gp<2>(plan, a, stream);
        case 4: return dispatch_gp<4>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace attnres
