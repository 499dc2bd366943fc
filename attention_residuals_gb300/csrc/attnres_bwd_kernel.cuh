// attnres_bwd_kernel.cuh -- backward kernel and dq/dw_o finalize of the
// Attention Residuals read operator, as a template that each including
// translation unit instantiates for one output-norm mode (NORM: 1 o rebuilt
// from the sources, 2 the caller's FP32 o; -1 the mode read from the
// arguments at run time), so the units compile in parallel.
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
// threads that own fixed 16-byte column vectors.  dy rows go through a small
// ring of their own; source rows through a ring of chunks of G rows with one
// "full" and one "empty" mbarrier per chunk.  When a token's S rows fit
// ("resident"), each source row is read from HBM once: the o rebuild (with
// the output norm), the dot pass and the write pass all read it from shared
// memory, and the write pass releases the chunks.  Otherwise the producer
// streams the rows once per pass (served from L2 when it still holds them),
// and the write pass gets key slices only.  The saved per-token statistics arrive
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
#pragma once

#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"
#include "launch_pdl.cuh"

namespace attnres {
namespace {

// First failed wait of any backward launch of this unit (0 = none).
__device__ unsigned int g_bwd_error = 0;

__device__ __forceinline__ float ldcg_f32(const float* p) { return __ldcg(p); }

// KEYALL: every channel is a key channel (R == D), so no per-vector masks.
// FULL: every consumer thread owns VPT whole vectors (D == 8 * VPT * 32 * ncw).
// ADDLAST: a gradient is added to the last source's (a.dlast_add set); a
// compile-time flag so the plain backward carries none of its code.
// NORM: output RMSNorm mode fixed by the including unit: 1 o rebuilt from
// the sources, 2 the caller's FP32 o in a.o_pre, -1 read from a.out_norm and
// a.o_pre at run time (the form the launches without the norm use: with
// the norm code compiled in but skipped, they measured faster than a fixed
// no-norm mode).
// NJ: groups of 32 sources whose coefficients each lane holds (1: S <= 32,
// 4: up to 128 sources).
template <int VPT, bool KEYALL, bool FULL, bool ADDLAST, int NORM, int NJ>
__global__ void __launch_bounds__(kMaxThreads, 1) attnres_bwd_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const bool norm_on = NORM < 0 ? a.out_norm != 0 : NORM != 0;  // output RMSNorm
    const bool o_saved = NORM < 0 ? a.o_pre != nullptr : NORM == 2;  // o from the caller
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = a.chunks;   // ring depth in chunks
    const int G = a.rows;     // rows per chunk
    const int DS = a.dy_slots;
    const int s_pad = a.s_pad;
    const SmemLayout L = make_layout(K, G, a.slot_bytes, DS, s_pad, true);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* dyfull = reinterpret_cast<uint64_t*>(smem + L.dyfull);
    uint64_t* dyempty = reinterpret_cast<uint64_t*>(smem + L.dyempty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    float* red = reinterpret_cast<float*>(smem + L.red);  // [2][red_rows][kRedPitch]
    float* tok = reinterpret_cast<float*>(smem + L.tok);  // [kTokSlots][3*s_pad + 4]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    volatile int* ticket_flag = abort_flag + 1;
    const int tstride = 3 * s_pad + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int S = a.S;
    const int D = a.D;
    const uint32_t sb = static_cast<uint32_t>(a.slot_bytes);
    const uint32_t cb = static_cast<uint32_t>(G) * sb;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        for (int k = 0; k < DS; ++k) {
            mbar_init(dyfull + k, 1);
            mbar_init(dyempty + k, ncw);
        }
        for (int k = 0; k < kTokSlots; ++k) {
            mbar_init(tfull + k, 32);
            mbar_init(tempty + k, ncw);
        }
        *abort_flag = 0;
        *ticket_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // set-up above overlaps the previous kernel's tail; global memory only after it
    pdl_wait();
    pdl_launch_dependents();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
        // Key slice of the write pass: only the key channels when they
        // start and end on 16-byte boundaries, else the whole row.
        const bool key_only = ((a.ko & 7) == 0) && ((a.R & 7) == 0);
        const uint32_t key_off_b = key_only ? static_cast<uint32_t>(a.ko) * 2u : 0u;
        const uint32_t key_bytes = key_only ? static_cast<uint32_t>(a.R) * 2u : row_bytes;
        // Passes over the source rows per token: resident -> one; streaming
        // -> (o rebuild when needed), dot pass, write pass (key slices).
        const int npass = a.resident ? 1 : ((norm_on && !o_saved) ? 3 : 2);
        unsigned char* ring = smem + L.ring;
        unsigned char* dyring = smem + L.dyring;
        int k = 0;
        uint32_t phase = 0;
        int dk = 0;
        uint32_t dphase = 0;
        int ts = 0;
        uint32_t tphase = 0;
        long long issued = 0, dy_issued = 0;
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
            if (norm_on && lane == 0) cp_async_4(dst + 3 * s_pad, a.o_rstd + n);
            cp_async_arrive_noinc(tfull + ts);
            if (++ts == kTokSlots) {
                ts = 0;
                tphase ^= 1u;
            }
            if (lane == 0) {
                // the caller's FP32 o of this token: into L2 while the consumers
                // finish the previous token, so their loads of it hit
                if (o_saved) prefetch_l2_bulk(a.o_pre + n * D, row_bytes * 2u);
                if (mbar_wait(dyempty + dk, dphase ^ 1u, abort_flag, &g_bwd_error, kSiteBwdProducer)) {
                    mbar_arrive_expect_tx(dyfull + dk, row_bytes);
                    tma_load_1d(dyring + dk * sb, a.dy + n * D, row_bytes, dyfull + dk, pol);
                    ++dy_issued;
                    if (++dk == DS) {
                        dk = 0;
                        dphase ^= 1u;
                    }
                    if constexpr (ADDLAST) {
                        // the gradient added to the last source rides in the next dy slot
                        if (mbar_wait(dyempty + dk, dphase ^ 1u, abort_flag, &g_bwd_error, kSiteBwdProducer)) {
                            mbar_arrive_expect_tx(dyfull + dk, row_bytes);
                            tma_load_1d(dyring + dk * sb, a.dlast_add + n * a.dlast_add_ld, row_bytes, dyfull + dk,
                                        pol);
                            ++dy_issued;
                            if (++dk == DS) {
                                dk = 0;
                                dphase ^= 1u;
                            }
                        }
                    }
                }
                for (int pass = 0; pass < npass && !*abort_flag; ++pass) {
                    const bool keys = !a.resident && pass == npass - 1;
                    const uint32_t off = keys ? key_off_b : 0u;
                    const uint32_t bytes = keys ? key_bytes : row_bytes;
                    for (int g0 = 0; g0 < S; g0 += G) {
                        const int gs = min(G, S - g0);
                        if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_bwd_error, kSiteBwdProducer)) break;
                        mbar_arrive_expect_tx(full + k, bytes * static_cast<uint32_t>(gs));
                        for (int r = 0; r < gs; ++r) {
                            const unsigned char* src =
                                static_cast<const unsigned char*>(a.src[g0 + r]) + (n * a.src_ld) * 2 + off;
                            tma_load_1d(ring + k * cb + r * sb + off, src, bytes, full + k, pol);
                        }
                        ++issued;
                        if (++k == K) {
                            k = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            __syncwarp();
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0 && *abort_flag) {
            for (int c = 0; c < K && c < issued; ++c) {
                const long long fills = (issued - 1 - c) / K + 1;
                volatile int no_abort = 0;
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_bwd_error, kSiteDrain);
            }
            for (int c = 0; c < DS && c < dy_issued; ++c) {
                const long long fills = (dy_issued - 1 - c) / DS + 1;
                volatile int no_abort = 0;
                mbar_wait(dyfull + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_bwd_error, kSiteDrain);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    int col[VPT];
    unsigned kmask[VPT];
    float2 qs[VPT][4];     // scale * q at the owned key channels, 0 elsewhere
    uint4 wb[VPT];         // output-norm weight bits
    float2 dq_acc[VPT][4];
    float2 dw_acc[VPT][4];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * nct;
        col[i] = c < ncv ? c : -1;
        unsigned m = 0;
        uint32_t ww[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float qv[2];
            uint32_t wv = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = 8 * c + 2 * kk + h;
                const bool in_key = col[i] >= 0 && j >= ko && j < kend;
                m |= in_key ? (1u << (2 * kk + h)) : 0u;
                qv[h] = in_key ? a.scale * bf16_bits_to_float(a.q[j - ko]) : 0.0f;
                const uint32_t wh = (norm_on && col[i] >= 0) ? a.w_o[j] : 0x3f80u;
                wv |= wh << (16 * h);
            }
            qs[i][kk] = make_float2(qv[0], qv[1]);
            ww[kk] = wv;
            dq_acc[i][kk] = make_float2(0.0f, 0.0f);
            dw_acc[i][kk] = make_float2(0.0f, 0.0f);
        }
        kmask[i] = m;
        wb[i] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);
    const float inv_d = 1.0f / static_cast<float>(D);

    // 32-bit shared addresses (row addresses include this thread's first
    // vector offset).
    const uint32_t sbase = smem_u32(smem);
    const uint32_t voff = static_cast<uint32_t>(col[0] < 0 ? 0 : col[0]) * 16u;
    const uint32_t vstep = static_cast<uint32_t>(nct) * 16u;
    const uint32_t ring_lo = sbase + L.ring + voff;
    const uint32_t dy_lo = sbase + L.dyring + voff;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    const uint32_t dyfull_s = sbase + L.dyfull;
    const uint32_t dyempty_s = sbase + L.dyempty;
    const uint32_t tfull_s = sbase + L.tfull;
    const uint32_t tempty_s = sbase + L.tempty;
    const uint32_t red_s = sbase + L.red;
    const int red_rows = L.red_rows;
    const int nq = (ncw + 3) >> 2;
    const long long dld_b = a.dsrc_ld * 2;
    const long long d_off = static_cast<long long>(col[0] < 0 ? 0 : col[0]) * 16;

    for (int k = threadIdx.x; k < 2 * red_rows * kRedPitch; k += nct) red[k] = 0.0f;
    named_bar_sync(1, nct);

    auto red_sum = [&](int buf, int row) -> float {
        const uint32_t base = red_s + static_cast<uint32_t>(((buf * red_rows + row) * kRedPitch) * 4);
        float t = 0.0f;
        for (int q4 = 0; q4 < nq; ++q4) {
            const float4 v = lds128f(base + 16u * q4);
            t += (v.x + v.y) + (v.z + v.w);
        }
        return t;
    };

    // chunk-ring position (chunk index, fill parity, row-0 address)
    int ck = 0;
    uint32_t cphase = 0;
    uint32_t cbase = ring_lo;
    auto next_chunk = [&](int& k, uint32_t& ph, uint32_t& base) {
        base += cb;
        if (++k == K) {
            k = 0;
            ph ^= 1u;
            base = ring_lo;
        }
    };
    int dk = 0;
    uint32_t dphase = 0;
    int ts = 0;
    uint32_t tphase = 0;
    int rbuf = 0;

    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        mbar_wait_s(tfull_s + 8u * ts, tphase, abort_flag, &g_bwd_error, kSiteBwdTokStat);
        const float* tk = tok + ts * tstride;

        // ---- dy into registers; its slot is free again at once
        uint4 dyv[VPT];
        {
            mbar_wait_s(dyfull_s + 8u * dk, dphase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
            uint32_t dep = 0;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                dyv[i] = col[i] >= 0 ? lds128(dy_lo + dk * sb + i * vstep) : make_uint4(0u, 0u, 0u, 0u);
                dep ^= dyv[i].x;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_after(dyempty_s + 8u * dk, dep);
            if (++dk == DS) {
                dk = 0;
                dphase ^= 1u;
            }
        }
        // the added gradient's slot (held until the write pass has used it)
        int gk = 0;
        if constexpr (ADDLAST) {
            gk = dk;
            mbar_wait_s(dyfull_s + 8u * dk, dphase, abort_flag, &g_bwd_error, kSiteBwdConsumer);
            if (++dk == DS) {
                dk = 0;
                dphase ^= 1u;
            }
        }
        // first chunk of this token's rows (resident: used by every pass)
        const int tk_ck = ck;
        const uint32_t tk_phase = cphase, tk_base = cbase;

        // ---- gradient wrt the mixture o (kept in registers)
        float2 dout[VPT][4];
        if (norm_on) {
            // o = sum_s alpha_s v_s in FP32: the caller's saved copy, or
            // rebuilt from the source rows (resident: the rows the other
            // passes use; streaming: a dedicated pass of chunks).
            float2 o[VPT][4];
            if (o_saved) {
                const float* prow = a.o_pre + n * static_cast<long long>(D);
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    if (col[i] >= 0) {
                        const uint4 lo = ld_global_nc_v4(prow + 8 * col[i]);
                        const uint4 hi = ld_global_nc_v4(prow + 8 * col[i] + 4);
                        o[i][0] = make_float2(__uint_as_float(lo.x), __uint_as_float(lo.y));
                        o[i][1] = make_float2(__uint_as_float(lo.z), __uint_as_float(lo.w));
                        o[i][2] = make_float2(__uint_as_float(hi.x), __uint_as_float(hi.y));
                        o[i][3] = make_float2(__uint_as_float(hi.z), __uint_as_float(hi.w));
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) o[i][kk] = make_float2(0.0f, 0.0f);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < VPT; ++i)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) o[i][kk] = make_float2(0.0f, 0.0f);
                int k = ck;
                uint32_t ph = cphase, base = cbase;
                for (int g0 = 0; g0 < S; g0 += G) {
                    const int gs = min(G, S - g0);
                    mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwd_error, kSiteBwdConsumer);
                    uint32_t dep = 0;
                    uint32_t rowa = base;
                    // four rows at a time where the norm is fixed on (0.889 -> 0.877 ms
                    // on the long workload), two in the run-time form
#pragma unroll(NORM > 0 ? 4 : 2)
                    for (int r = 0; r < gs; ++r) {
                        const float al = tk[g0 + r];
                        const float2 al2 = make_float2(al, al);
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            if (FULL || col[i] >= 0) {
                                const uint4 xv = lds128(rowa + i * vstep);
                                dep ^= xv.x;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) o[i][kk] = ffma2(al2, bf2_to_f2(u4_get(xv, kk)), o[i][kk]);
                            }
                        }
                        rowa += sb;
                    }
                    if (!a.resident) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                    }
                    next_chunk(k, ph, base);
                }
                if (!a.resident) {  // the streamed o-pass chunks are consumed
                    ck = k;
                    cphase = ph;
                    cbase = base;
                }
            }
            const float rho = tk[3 * s_pad];
            const float2 rho2 = make_float2(rho, rho);
            float2 gy2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float2 yh = fmul2(o[i][kk], rho2);
                    const float2 g = bf2_to_f2(u4_get(dyv[i], kk));
                    o[i][kk] = yh;
                    dw_acc[i][kk] = ffma2(g, yh, dw_acc[i][kk]);
                    const float2 gw = fmul2(g, bf2_to_f2(u4_get(wb[i], kk)));
                    gy2 = ffma2(gw, yh, gy2);
                    dout[i][kk] = gw;
                }
            }
            const float gy = warp_sum(gy2.x + gy2.y);
            if (lane == 0) red[(rbuf * red_rows) * kRedPitch + warp] = gy;
            named_bar_sync(1, nct);
            const float tot = red_sum(rbuf, 0);
            rbuf ^= 1;
            const float ncg = -tot * inv_d;
            const float2 ncg2 = make_float2(ncg, ncg);
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) dout[i][kk] = fmul2(rho2, ffma2(o[i][kk], ncg2, dout[i][kk]));
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) dout[i][kk] = bf2_to_f2(u4_get(dyv[i], kk));
        }

        // ---- dot pass: da_s = <do, v_s>, four rows at a time per chunk
        {
            int k = a.resident ? tk_ck : ck;
            uint32_t ph = a.resident ? tk_phase : cphase;
            uint32_t base = a.resident ? tk_base : cbase;
            for (int g0 = 0; g0 < S; g0 += G) {
                const int gs = min(G, S - g0);
                mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwd_error, kSiteBwdConsumer);
                uint32_t dep = 0;
                for (int c0 = 0; c0 < gs; c0 += 4) {
                    float part[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float2 d2 = make_float2(0.0f, 0.0f);
                        if (c0 + r < gs) {
                            const uint32_t rowa = base + static_cast<uint32_t>(c0 + r) * sb;
#pragma unroll
                            for (int i = 0; i < VPT; ++i) {
                                if (FULL || col[i] >= 0) {
                                    const uint4 xv = lds128(rowa + i * vstep);
                                    dep ^= xv.x;
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk) d2 = ffma2(dout[i][kk], bf2_to_f2(u4_get(xv, kk)), d2);
                                }
                            }
                        }
                        part[r] = d2.x + d2.y;
                    }
                    warp_reduce_scatter<4>(part, lane);
                    // lane l holds element l >> 3
                    if ((lane & 7) == 0 && c0 + (lane >> 3) < gs)
                        red[(rbuf * red_rows + g0 + c0 + (lane >> 3)) * kRedPitch + warp] = part[0];
                }
                if (!a.resident) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                }
                next_chunk(k, ph, base);
            }
            if (!a.resident) {
                ck = k;
                cphase = ph;
                cbase = base;
            }
        }
        named_bar_sync(1, nct);

        // ---- per-source coefficients, computed by every warp (identically)
        // and kept in registers: lane l holds sources l, l+32, ... (NJ of them).
        float cal[NJ], ck1[NJ], ck2[NJ];
        {
            float dav[NJ];
            float part_delta = 0.0f;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int s = lane + 32 * j;
                float d = 0.0f;
                if (s < S) {
                    d = red_sum(rbuf, s);
                    part_delta = fmaf(tk[s], d, part_delta);
                }
                dav[j] = d;
            }
            const float delta = warp_sum(part_delta);
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int s = lane + 32 * j;
                cal[j] = ck1[j] = ck2[j] = 0.0f;
                if (s < S) {
                    const float al = tk[s];
                    const float r = tk[s_pad + s];
                    const float z = tk[2 * s_pad + s];
                    const float dz = al * (dav[j] - delta);
                    cal[j] = al;
                    ck1[j] = r * dz;  // qs carries `scale`, so ck1 * qs = rstd * scale * dz * q
                    ck2[j] = -(r * r) * dz * z * inv_r;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_s(tempty_s + 8u * ts);  // this warp is done with tok[ts]
        }
        rbuf ^= 1;
        if (++ts == kTokSlots) {
            ts = 0;
            tphase ^= 1u;
        }

        // ---- write pass: dv_s rows and dq contributions
        uint32_t gdep = 0;  // data dependency of the added gradient's loads
        {
            int k = a.resident ? tk_ck : ck;
            uint32_t ph = a.resident ? tk_phase : cphase;
            uint32_t base = a.resident ? tk_base : cbase;
            const long long row_off = n * dld_b + d_off;
            const long long dstride = a.dsrc_stride;
            char* dnext = static_cast<char*>(a.dsrc[0]) + row_off;  // used when evenly spaced
            for (int g0 = 0; g0 < S; g0 += G) {
                const int gs = min(G, S - g0);
                if (!a.resident) mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwd_error, kSiteBwdConsumer);
                uint32_t dep = 0;
                uint32_t rowa = base;
#pragma unroll 2
                for (int r = 0; r < gs; ++r) {
                    const int s = g0 + r;
                    float al, k1, k2;
                    if constexpr (NJ == 1) {
                        al = __shfl_sync(0xffffffffu, cal[0], s);
                        k1 = __shfl_sync(0xffffffffu, ck1[0], s);
                        k2 = __shfl_sync(0xffffffffu, ck2[0], s);
                    } else {
                        static_assert(NJ == 4, "one or four groups of 32 sources");
                        if (S <= 32) {
                            al = __shfl_sync(0xffffffffu, cal[0], s);
                            k1 = __shfl_sync(0xffffffffu, ck1[0], s);
                            k2 = __shfl_sync(0xffffffffu, ck2[0], s);
                        } else {
                            const int j = s >> 5;
                            al = __shfl_sync(0xffffffffu, j == 0 ? cal[0] : j == 1 ? cal[1] : j == 2 ? cal[2] : cal[3], s & 31);
                            k1 = __shfl_sync(0xffffffffu, j == 0 ? ck1[0] : j == 1 ? ck1[1] : j == 2 ? ck1[2] : ck1[3], s & 31);
                            k2 = __shfl_sync(0xffffffffu, j == 0 ? ck2[0] : j == 1 ? ck2[1] : j == 2 ? ck2[2] : ck2[3], s & 31);
                        }
                    }
                    const float2 al2 = make_float2(al, al), k12 = make_float2(k1, k1), k22 = make_float2(k2, k2);
                    char* drow = dstride ? dnext : static_cast<char*>(a.dsrc[s]) + row_off;
                    dnext += dstride;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (FULL || col[i] >= 0) {
                            float2 dv[4];
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) dv[kk] = fmul2(al2, dout[i][kk]);
                            if (KEYALL || kmask[i] != 0u) {
                                const uint4 xv = lds128(rowa + i * vstep);
                                dep ^= xv.x;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    float2 x = bf2_to_f2(u4_get(xv, kk));
                                    if (!KEYALL && kmask[i] != 0xffu) {
                                        if (!((kmask[i] >> (2 * kk)) & 1u)) x.x = 0.0f;
                                        if (!((kmask[i] >> (2 * kk + 1)) & 1u)) x.y = 0.0f;
                                    }
                                    dv[kk] = ffma2(k12, qs[i][kk], ffma2(k22, x, dv[kk]));
                                    dq_acc[i][kk] = ffma2(k12, x, dq_acc[i][kk]);
                                }
                            }
                            if (ADDLAST && s == S - 1) {
                                // gradient reaching the last source from elsewhere (a fused
                                // block-partial sum's later uses), added before rounding
                                const uint4 gv = lds128(dy_lo + gk * sb + i * vstep);
                                gdep ^= gv.x;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    dv[kk] = ffma2(make_float2(1.0f, 1.0f), bf2_to_f2(u4_get(gv, kk)), dv[kk]);
                            }
                            if (ATTNRES_IN_BOUNDS(n < N && s < S && 8 * col[i] + 8 <= D, &g_bwd_error))
                            st_global_cs_v4(drow + static_cast<long long>(i) * vstep,
                                            make_uint4(pack_f2(dv[0]), pack_f2(dv[1]), pack_f2(dv[2]), pack_f2(dv[3])));
                        }
                    }
                    rowa += sb;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                next_chunk(k, ph, base);
            }
            ck = k;
            cphase = ph;
            cbase = base;
        }
        if constexpr (ADDLAST) {
            __syncwarp();
            if (lane == 0) mbar_arrive_after(dyempty_s + 8u * gk, gdep);
        }
    }

    // ---------------------------------------------- per-CTA partial sums
    const int R = a.R;
    const int Dw = norm_on ? D : 0;
    const int W = R + Dw;
    float* my_part = a.part + static_cast<size_t>(blockIdx.x) * W;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        if (col[i] >= 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * col[i] + e;
                const float dqv = (e & 1) ? dq_acc[i][e >> 1].y : dq_acc[i][e >> 1].x;
                const float dwv = (e & 1) ? dw_acc[i][e >> 1].y : dw_acc[i][e >> 1].x;
                // dq = scale * sum_s dz_s k_s = scale * sum_s c1_s t_s
                if (!ATTNRES_IN_BOUNDS(static_cast<int>(blockIdx.x) < a.part_rows && j < D &&
                                           (!((kmask[i] >> e) & 1u) || (j >= ko && j - ko < R)),
                                       &g_bwd_error))
                    continue;
                if ((kmask[i] >> e) & 1u) my_part[j - ko] = a.scale * dqv;
                if (norm_on) my_part[R + j] = dwv;
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
    // four columns at a time, every load of them in flight before the adds
    // (which keep the CTA order)
    for (int c0 = threadIdx.x; c0 < W; c0 += 4 * nct) {
        float v[4][kGroupTicket];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * nct;
#pragma unroll
            for (int b = 0; b < kGroupTicket; ++b)
                v[u][b] = (c < W && b < g_size) ? ldcg_f32(a.part + static_cast<size_t>(g_first + b) * W + c) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float acc = 0.0f;
#pragma unroll
            for (int b = 0; b < kGroupTicket; ++b)
                if (b < g_size) acc += v[u][b];
            if (c0 + u * nct < W) gsum[c0 + u * nct] = acc;
        }
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
    for (int c0 = threadIdx.x; c0 < W; c0 += 4 * nct) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int g0 = 0; g0 < a.ngroups; g0 += 8) {
            float v[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * nct;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[u][k] = (c < W && g0 + k < a.ngroups)
                                  ? ldcg_f32(a.gpart + static_cast<size_t>(g0 + k) * W + c) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (g0 + k < a.ngroups) acc[u] += v[u][k];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * nct;
            if (c >= W) continue;
            const uint16_t h = static_cast<uint16_t>(pack_bf16x2(acc[u], 0.0f) & 0xffffu);
            if (c < R) {
                a.dq[c] = h;
                if (a.dq_f32) a.dq_f32[c] = acc[u];
            } else {
                a.dw_o[c - R] = h;
                if (a.dw_o_f32) a.dw_o_f32[c - R] = acc[u];
            }
        }
    }
}

// Finalize for the split-N path: column c of dq/dw_o is the sum of the P
// partial rows.  A block takes kFinCols columns; its kFinSlices warps each
// add one contiguous range of rows for them (eight loads in flight per
// thread: one or two rounds for up to 512 rows), then the ranges' sums are
// added in range order -- a fixed order, so the result does not depend on
// timing.
constexpr int kFinCols = 32, kFinSlices = 32;

__global__ void __launch_bounds__(kFinCols * kFinSlices) attnres_finalize_kernel(
    const float* __restrict__ part, int P, int R, int W, uint16_t* dq, float* dq_f32, uint16_t* dw_o,
    float* dw_o_f32) {
    __shared__ float sums[kFinSlices][kFinCols];
    pdl_wait();  // the partial rows are complete and visible
    const int lane = threadIdx.x % kFinCols, sl = threadIdx.x / kFinCols;
    const int c = blockIdx.x * kFinCols + lane;
    const int per = (P + kFinSlices - 1) / kFinSlices;
    const int b0 = sl * per, b1 = min(P, b0 + per);
    float acc = 0.0f;
    if (c < W) {
        for (int b = b0; b < b1; b += 8) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = b + k < b1 ? __ldcg(part + static_cast<size_t>(b + k) * W + c) : 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (b + k < b1) acc += v[k];
        }
    }
    sums[sl][lane] = acc;
    __syncthreads();
    if (sl != 0 || c >= W) return;
    acc = sums[0][lane];
#pragma unroll
    for (int k = 1; k < kFinSlices; ++k) acc += sums[k][lane];
    const uint16_t h = static_cast<uint16_t>(pack_bf16x2(acc, 0.0f) & 0xffffu);
    if (c < R) {
        dq[c] = h;
        if (dq_f32) dq_f32[c] = acc;
    } else {
        dw_o[c - R] = h;
        if (dw_o_f32) dw_o_f32[c - R] = acc;
    }
}

template <int VPT, bool KEYALL, bool FULL, bool ADDLAST, int NORM, int NJ = 1>
cudaError_t launch_bwd_t(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_bwd_kernel<VPT, KEYALL, FULL, ADDLAST, NORM, NJ>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_bwd));
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(plan.grid), dim3((plan.b_ncw + 1) * 32), plan.smem_bwd, stream, a);
    if (err != cudaSuccess || !plan.split) return err;
    const int W = a.R + (a.out_norm ? a.D : 0);
    return launch_pdl(attnres_finalize_kernel, dim3((W + kFinCols - 1) / kFinCols), dim3(kFinCols * kFinSlices), 0,
                      stream, static_cast<const float*>(a.part), plan.grid, a.R, W, a.dq, a.dq_f32, a.dw_o,
                      a.dw_o_f32);
}

template <int VPT, int NORM, int NJ>
cudaError_t dispatch_cols(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    const bool full = (a.D / 8) == VPT * 32 * plan.b_ncw;
    if (a.dlast_add) {
        // with an added gradient: whole-vector ownership compiled in for rows
        // of up to 4096 channels (the block schedule's widths), else the
        // general column form
        if constexpr (VPT <= 2) {
            if (full)
                return a.R == a.D ? launch_bwd_t<VPT, true, true, true, NORM, NJ>(plan, a, stream)
                                  : launch_bwd_t<VPT, false, true, true, NORM, NJ>(plan, a, stream);
        }
        return a.R == a.D ? launch_bwd_t<VPT, true, false, true, NORM, NJ>(plan, a, stream)
                          : launch_bwd_t<VPT, false, false, true, NORM, NJ>(plan, a, stream);
    }
    if (a.R == a.D)
        return full ? launch_bwd_t<VPT, true, true, false, NORM, NJ>(plan, a, stream)
                    : launch_bwd_t<VPT, true, false, false, NORM, NJ>(plan, a, stream);
    if constexpr (NORM < 0 && NJ == 1) {
        return cudaErrorInvalidConfiguration;  // not dispatched (dispatch_key)
    } else {
        return full ? launch_bwd_t<VPT, false, true, false, NORM, NJ>(plan, a, stream)
                    : launch_bwd_t<VPT, false, false, false, NORM, NJ>(plan, a, stream);
    }
}

// One group of 32 sources per lane when S <= 32, four otherwise -- except the
// sliced-key launches without the norm and without an added gradient, whose
// four-group form measured faster (sliced block shape: 0.394 against 0.415
// ms; the full-key short shape ran 0.131 against 0.147 ms with one group).
template <int VPT, int NORM>
cudaError_t dispatch_key(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    const bool one_group = a.S <= 32 && (NORM >= 0 || a.dlast_add || a.R == a.D);
    return one_group ? dispatch_cols<VPT, NORM, 1>(plan, a, stream) : dispatch_cols<VPT, NORM, 4>(plan, a, stream);
}

// Every kernel of this unit's output-norm mode.
template <int NORM>
cudaError_t launch_bwd_mode(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    switch (plan.b_vpt) {
        case 1: return dispatch_key<1, NORM>(plan, a, stream);
        case 2: return dispatch_key<2, NORM>(plan, a, stream);
        case 4: return dispatch_key<4, NORM>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

// This unit's first recorded wait failure (then cleared).
inline unsigned take_unit_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof zero);
    return v;
}

}  // namespace
}  // namespace attnres
