// attnres_bwd_cluster.cu -- backward of the Attention Residuals read for
// tokens whose S source rows do not fit in one SM's shared memory (the deep
// shapes: 64 rows of 8192 channels are 1 MB per token).  A thread-block
// cluster of `cl` CTAs shares each token: CTA r of the cluster owns columns
// [r*D/cl, (r+1)*D/cl) of all S rows (and of dy).  Either a token's column
// slices stay in shared memory for all passes ("resident"), or they stream
// through the chunk ring once per pass ("streaming": o rebuild when the
// output norm needs it, dot pass, write pass).  Streaming one token at a
// time per CTA, the rows a CTA reads again in a later pass were read
// S * D * 2 / cl bytes earlier; over the whole grid that reuse distance is
// (clusters) x (one token's rows), cl times shorter than with one CTA per
// token, so the second and third reads of a row hit L2 and each row crosses
// HBM once either way.
//
// Per token (chain rule through "Fast Attention Residuals", section
// "Equation", with the output RMSNorm of "[Perf] Parallelize AttnRes
// long-sequence reduction", Summary; the same formulas as
// attnres_bwd_kernel.cuh):
//   out-norm:  o = sum_s alpha_s v_s (this CTA's columns), yhat = o * o_rstd,
//              dw_o += dy * yhat, g = dy * w_o,
//              do = o_rstd * (g - yhat * <g, yhat> / D);   else do = dy
//   da_s  = <do, v_s>,   delta = sum_s alpha_s da_s,  dz_s = alpha_s (da_s - delta)
//   dv_s  = alpha_s do  +  on key channels: c1_s q + c2_s t_s
//           with c1_s = rstd_s scale dz_s,  c2_s = -rstd_s^2 dz_s z_s / R
//   dq   += sum_s c1_s t_s
// Two of these are sums over all D channels: <g, yhat> and the S dots da_s.
// Each CTA forms its slice's partial sums and the cluster exchanges them
// through distributed shared memory: one warp writes the CTA's values into
// every peer's exchange buffer (st.shared::cluster) and arrives on the
// peer's exchange mbarrier with release at cluster scope; every CTA waits on
// its own barrier (acquire at cluster scope, bounded) and adds the cl
// partial sums in rank order -- the same order in every CTA, so all CTAs
// derive bitwise identical coefficients, and the result is reproducible run
// to run.  Exchange buffers alternate between two sets per round; a CTA can
// run at most one round ahead of a peer (it cannot finish round k+1 before
// that peer has sent it, which the peer does only after reading round k),
// so two sets suffice.
//
// dq and dw_o: each CTA accumulates its columns over all of the cluster's
// tokens in registers and writes them into its cluster's FP32 partial row;
// the finalize kernel adds the rows in cluster order.
#include "device_utils.cuh"
#include "kernels.cuh"

#include <cstdlib>
#include <mutex>

namespace attnres {
namespace {

// First failed wait of any cluster-backward launch (0 = none).
__device__ unsigned int g_bwdc_error = 0;

// L2 policy for rows that a later pass of the same token reads again.
__device__ __forceinline__ uint64_t policy_keep_in_l2() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// KEYALL: R == D (no per-channel key masks).  NORM: 0 no output norm, 1 o
// rebuilt from the rows, 2 the caller's FP32 o (a.o_pre).  NJ: groups of 32
// sources whose coefficients each lane holds (1: S <= 32, 4: up to 128
// sources).  FULL: every consumer thread owns whole 16-byte vectors of the
// slice.  a.resident selects resident or streaming rows at run time.
template <int VPT, bool KEYALL, int NORM, int NJ, bool FULL>
__global__ void __launch_bounds__(kMaxThreads, 1) attnres_bwd_cluster_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = a.chunks;   // ring depth in chunks
    const int G = a.rows;     // rows per chunk
    const int DS = a.dy_slots;
    const int s_pad = a.s_pad;
    const int CL = a.cl;
    const ClusterLayout XL = make_cluster_layout(K, G, a.slot_bytes, DS, s_pad, CL);
    const SmemLayout& L = XL.base;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* dyfull = reinterpret_cast<uint64_t*>(smem + L.dyfull);
    uint64_t* dyempty = reinterpret_cast<uint64_t*>(smem + L.dyempty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + XL.xbar);
    float* red = reinterpret_cast<float*>(smem + L.red);  // [2][red_rows][kRedPitch]
    float* tok = reinterpret_cast<float*>(smem + L.tok);  // [kTokSlots][3*s_pad + 4]
    const float* xbuf = reinterpret_cast<const float*>(smem + XL.xbuf);  // [2][CL][s_pad]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int tstride = 3 * s_pad + 4;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const long long cid = cluster_index_x();
    const long long ncl = cluster_count_x();
    const long long N = a.N;
    const int S = a.S;
    const int D = a.D;
    const int slice = a.slice;  // columns of every row this CTA holds
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
        mbar_init(xbar + 0, kExchangeArrivals);
        mbar_init(xbar + 1, kExchangeArrivals);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // every CTA's exchange barriers are initialised before any peer arrives on them
    cluster_sync_all();
    // set-up above overlaps the previous kernel's tail; global memory only after it
    pdl_wait();
    pdl_launch_dependents();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        const uint64_t pol_keep = policy_keep_in_l2();
        const uint32_t row_bytes = static_cast<uint32_t>(slice) * 2u;
        const long long col0 = static_cast<long long>(rank) * slice;  // first column of the slice
        unsigned char* ring = smem + L.ring;
        unsigned char* dyring = smem + L.dyring;
        // passes over a token's row slices: resident -> one; streaming -> (o
        // rebuild when o is not the caller's), dot pass, write pass
        const int npass = a.resident ? 1 : (NORM == 1 ? 3 : 2);
        int k = 0;
        uint32_t phase = 0;
        int dk = 0;
        uint32_t dphase = 0;
        int ts = 0;
        uint32_t tphase = 0;
        long long issued = 0, dy_issued = 0;
        for (long long n = cid; n < N; n += ncl) {
            // one decision for the whole warp (lane 0's view of the flag): every
            // lane leaves the loop together and meets the same __syncwarp and
            // cluster barrier below
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            // token statistics -> tok[ts] (all 32 lanes arrive on tfull)
            mbar_wait(tempty + ts, tphase ^ 1u, abort_flag, &g_bwdc_error, kSiteBwdProducer);
            float* dst = tok + ts * tstride;
            for (int e = lane; e < S; e += 32) {
                cp_async_4(dst + e, a.alpha + n * S + e);
                cp_async_4(dst + s_pad + e, a.rstd + n * S + e);
                cp_async_4(dst + 2 * s_pad + e, a.logit + n * S + e);
            }
            if (NORM != 0 && lane == 0) cp_async_4(dst + 3 * s_pad, a.o_rstd + n);
            cp_async_arrive_noinc(tfull + ts);
            if (++ts == kTokSlots) {
                ts = 0;
                tphase ^= 1u;
            }
            if (lane == 0) {
                // the caller's FP32 o of this token's slice: into L2 while the
                // consumers finish the previous token, so their loads of it hit
                if (NORM == 2 && !a.resident) prefetch_l2_bulk(a.o_pre + n * D + col0, row_bytes * 2u);
                if (mbar_wait(dyempty + dk, dphase ^ 1u, abort_flag, &g_bwdc_error, kSiteBwdProducer)) {
                    mbar_arrive_expect_tx(dyfull + dk, row_bytes);
                    tma_load_1d(dyring + dk * sb, a.dy + n * D + col0, row_bytes, dyfull + dk, pol);
                    ++dy_issued;
                    if (++dk == DS) {
                        dk = 0;
                        dphase ^= 1u;
                    }
                }
                bool stop = false;
                for (int pass = 0; pass < npass && !stop; ++pass) {
                    // the last pass's reads are the token's last: evict them first
                    const uint64_t cp = pass + 1 == npass ? pol : pol_keep;
                    for (int g0 = 0; g0 < S; g0 += G) {
                        const int gs = min(G, S - g0);
                        if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_bwdc_error, kSiteBwdProducer)) {
                            stop = true;
                            break;
                        }
                        mbar_arrive_expect_tx(full + k, row_bytes * static_cast<uint32_t>(gs));
                        for (int r = 0; r < gs; ++r) {
                            const unsigned char* src =
                                static_cast<const unsigned char*>(a.src[g0 + r]) + (n * a.src_ld + col0) * 2;
                            tma_load_1d(ring + k * cb + r * sb, src, row_bytes, full + k, cp);
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
            // copies still in flight land before the CTA may leave
            for (int c = 0; c < K && c < issued; ++c) {
                const long long fills = (issued - 1 - c) / K + 1;
                volatile int no_abort = 0;
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_bwdc_error, kSiteDrain);
            }
            for (int c = 0; c < DS && c < dy_issued; ++c) {
                const long long fills = (dy_issued - 1 - c) / DS + 1;
                volatile int no_abort = 0;
                mbar_wait(dyfull + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_bwdc_error, kSiteDrain);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- consumers
        const int ncv = slice >> 3;  // 16-byte vectors of the slice
        const int v0 = static_cast<int>(rank) * ncv;  // first global vector of the slice
        const int ko = a.ko, kend = a.ko + a.R;
        int lcol[VPT];         // local vector index inside the slice, -1 = none
        unsigned kmask[VPT];
        float2 qs[VPT][4];     // scale * q at the owned key channels, 0 elsewhere
        uint4 wb[VPT];         // output-norm weight bits
        float2 dq_acc[VPT][4];
        float2 dw_acc[VPT][4];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = threadIdx.x + i * nct;
            lcol[i] = c < ncv ? c : -1;
            unsigned m = 0;
            uint32_t ww[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float qv[2];
                uint32_t wv = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = 8 * (v0 + c) + 2 * kk + h;
                    const bool in_key = lcol[i] >= 0 && j >= ko && j < kend;
                    m |= in_key ? (1u << (2 * kk + h)) : 0u;
                    qv[h] = in_key ? a.scale * bf16_bits_to_float(a.q[j - ko]) : 0.0f;
                    const uint32_t wh = (NORM != 0 && lcol[i] >= 0) ? a.w_o[j] : 0x3f80u;
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

        const uint32_t sbase = smem_u32(smem);
        const uint32_t voff = static_cast<uint32_t>(lcol[0] < 0 ? 0 : lcol[0]) * 16u;
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
        const uint32_t xbar_s = sbase + XL.xbar;
        const uint32_t xbuf_s = sbase + XL.xbuf;
        const uint32_t ctab_s = sbase + XL.ctab + static_cast<uint32_t>(warp * s_pad) * 16u;  // this warp's table
        const int red_rows = L.red_rows;
        const int nq = (ncw + 3) >> 2;
        const long long dld_b = a.dsrc_ld * 2;
        const long long d_off = static_cast<long long>(v0 + (lcol[0] < 0 ? 0 : lcol[0])) * 16;

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

        // One exchange round: warp 0 sends this CTA's `nval` values (value_of(s))
        // to every CTA of the cluster -- lane l writes values l / CL, l / CL +
        // 32 / CL, ... into CTA (l % CL)'s buffer row of this rank, then arrives
        // on that CTA's barrier (32 arrivals per CTA and round) -- and every
        // consumer waits until all peers' values are in.  Returns the round's
        // [CL][s_pad] buffer.
        int xround = 0;
        auto exchange = [&](int nval, auto&& value_of) -> const float* {
            const int b = xround & 1;
            const uint32_t par = static_cast<uint32_t>(xround >> 1) & 1u;
            if (warp == 0) {
                const uint32_t dst = static_cast<uint32_t>(lane % CL);
                const uint32_t row = xbuf_s + static_cast<uint32_t>(((b * CL + static_cast<int>(rank)) * s_pad) * 4);
                const uint32_t rrow = cluster_map(row, dst);
                for (int s = lane / CL; s < nval; s += 32 / CL) st_cluster_f32(rrow + 4u * s, value_of(s));
                mbar_arrive_remote(cluster_map(xbar_s + 8u * b, dst));
            }
            mbar_wait_cluster_s(xbar_s + 8u * b, par, abort_flag, &g_bwdc_error, kSiteBwdExchange);
            ++xround;
            return xbuf + b * CL * s_pad;
        };
        auto cluster_total = [&](const float* xb, int s) -> float {
            float t = 0.0f;
            for (int r = 0; r < CL; ++r) t += xb[r * s_pad + s];  // rank order: identical in every CTA
            return t;
        };

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

        for (long long n = cid; n < N; n += ncl) {
            mbar_wait_s(tfull_s + 8u * ts, tphase, abort_flag, &g_bwdc_error, kSiteBwdTokStat);
            const float* tk = tok + ts * tstride;

            // ---- dy slice into registers; its slot is free again at once
            uint4 dyv[VPT];
            {
                mbar_wait_s(dyfull_s + 8u * dk, dphase, abort_flag, &g_bwdc_error, kSiteBwdConsumer);
                uint32_t dep = 0;
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    dyv[i] = (FULL || lcol[i] >= 0) ? lds128(dy_lo + dk * sb + i * vstep) : make_uint4(0u, 0u, 0u, 0u);
                    dep ^= dyv[i].x;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_after(dyempty_s + 8u * dk, dep);
                if (++dk == DS) {
                    dk = 0;
                    dphase ^= 1u;
                }
            }
            // first chunk of this token's rows (resident: used by every pass)
            const bool res = a.resident != 0;
            const int tk_ck = ck;
            const uint32_t tk_phase = cphase, tk_base = cbase;

            // ---- gradient wrt the mixture o (kept in registers)
            float2 dout[VPT][4];
            if constexpr (NORM != 0) {
                float2 o[VPT][4];
                if constexpr (NORM == 2) {
                    // the caller's FP32 o, this slice's columns
                    const float* prow = a.o_pre + n * static_cast<long long>(D);
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (FULL || lcol[i] >= 0) {
                            const int gc = v0 + lcol[i];
                            const uint4 lo = ld_global_nc_v4(prow + 8 * gc);
                            const uint4 hi = ld_global_nc_v4(prow + 8 * gc + 4);
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
                        mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwdc_error, kSiteBwdConsumer);
                        uint32_t dep = 0;
                        uint32_t rowa = base;
#pragma unroll 4
                        for (int r = 0; r < gs; ++r) {
                            const float al = tk[g0 + r];
                            const float2 al2 = make_float2(al, al);
#pragma unroll
                            for (int i = 0; i < VPT; ++i) {
                                if (FULL || lcol[i] >= 0) {
                                    const uint4 xv = lds128(rowa + i * vstep);
                                    dep ^= xv.x;
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        o[i][kk] = ffma2(al2, bf2_to_f2(u4_get(xv, kk)), o[i][kk]);
                                }
                            }
                            rowa += sb;
                        }
                        if (!res) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                        }
                        next_chunk(k, ph, base);
                    }
                    if (!res) {  // the streamed o-pass chunks are consumed
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
                const float part_gy = red_sum(rbuf, 0);
                rbuf ^= 1;
                // <g, yhat> over all D channels: the cluster's partial sums
                const float* xb = exchange(1, [&](int) { return part_gy; });
                const float tot = cluster_total(xb, 0);
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

            // ---- dot pass: this slice's part of da_s = <do, v_s>
            {
                int k = res ? tk_ck : ck;
                uint32_t ph = res ? tk_phase : cphase;
                uint32_t base = res ? tk_base : cbase;
                // one quad of rows: its four partial dots into p[0..3]
                auto quad = [&](uint32_t rowa0, int nrow, float* p, uint32_t& dep) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float2 d2 = make_float2(0.0f, 0.0f);
                        if (r < nrow) {
                            const uint32_t rowa = rowa0 + static_cast<uint32_t>(r) * sb;
#pragma unroll
                            for (int i = 0; i < VPT; ++i) {
                                if (FULL || lcol[i] >= 0) {
                                    const uint4 xv = lds128(rowa + i * vstep);
                                    dep ^= xv.x;
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        d2 = ffma2(dout[i][kk], bf2_to_f2(u4_get(xv, kk)), d2);
                                }
                            }
                        }
                        p[r] = d2.x + d2.y;
                    }
                };
                if (G % 4 == 0) {
                    // Streamed chunks of whole quads: two quads (eight rows,
                    // across chunk boundaries) per warp reduce-scatter, which
                    // halves the shuffle latency per row; each chunk is released
                    // as soon as its rows are read.
                    int crow = 0;  // rows of the current chunk already read
                    uint32_t dep = 0;
                    for (int b0 = 0; b0 < S; b0 += 8) {
                        float part[8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int q0 = b0 + 4 * h;
                            if (q0 < S) {
                                if (crow == 0) mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwdc_error, kSiteBwdConsumer);
                                quad(base + static_cast<uint32_t>(crow) * sb, S - q0, part + 4 * h, dep);
                                crow += 4;
                                if (crow == G || q0 + 4 >= S) {
                                    if (!res) {
                                        __syncwarp();
                                        if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                                    }
                                    dep = 0;
                                    crow = 0;
                                    next_chunk(k, ph, base);
                                }
                            } else {
#pragma unroll
                                for (int r = 0; r < 4; ++r) part[4 * h + r] = 0.0f;
                            }
                        }
                        warp_reduce_scatter<8>(part, lane);
                        if ((lane & 3) == 0 && b0 + (lane >> 2) < S)
                            red[(rbuf * red_rows + b0 + (lane >> 2)) * kRedPitch + warp] = part[0];
                    }
                } else {
                    for (int g0 = 0; g0 < S; g0 += G) {
                        const int gs = min(G, S - g0);
                        mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwdc_error, kSiteBwdConsumer);
                        uint32_t dep = 0;
                        for (int c0 = 0; c0 < gs; c0 += 4) {
                            float part[4];
                            quad(base + static_cast<uint32_t>(c0) * sb, gs - c0, part, dep);
                            warp_reduce_scatter<4>(part, lane);
                            if ((lane & 7) == 0 && c0 + (lane >> 3) < gs)
                                red[(rbuf * red_rows + g0 + c0 + (lane >> 3)) * kRedPitch + warp] = part[0];
                        }
                        if (!res) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
                        }
                        next_chunk(k, ph, base);
                    }
                }
                if (!res) {
                    ck = k;
                    cphase = ph;
                    cbase = base;
                }
            }
            named_bar_sync(1, nct);

            // ---- the cluster's da_s, then the per-source coefficients (every
            // warp computes them identically; lane l holds sources l, l+32, ...,
            // and writes them to the warp's own table for the write pass)
            {
                const int rb = rbuf;
                const float* xb = exchange(S, [&](int s) { return red_sum(rb, s); });
                float dav[NJ];
                float part_delta = 0.0f;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int s = lane + 32 * j;
                    float d = 0.0f;
                    if (s < S) {
                        d = cluster_total(xb, s);
                        part_delta = fmaf(tk[s], d, part_delta);
                    }
                    dav[j] = d;
                }
                const float delta = warp_sum(part_delta);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int s = lane + 32 * j;
                    if (s < S) {
                        const float al = tk[s];
                        const float r = tk[s_pad + s];
                        const float z = tk[2 * s_pad + s];
                        const float dz = al * (dav[j] - delta);
                        const float k1 = r * dz;  // qs carries `scale`
                        const float k2 = -(r * r) * dz * z * inv_r;
                        sts128(ctab_s + 16u * static_cast<uint32_t>(s),
                               make_uint4(__float_as_uint(al), __float_as_uint(k1), __float_as_uint(k2), 0u));
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

            // ---- write pass: dv_s slices and dq contributions; releases the chunks
            {
                // the gradient rows are not read again here: first out of L2,
                // so the rows this pass re-reads stay
                const uint64_t st_pol = policy_evict_first();
                int k = res ? tk_ck : ck;
                uint32_t ph = res ? tk_phase : cphase;
                uint32_t base = res ? tk_base : cbase;
                const long long row_off = n * dld_b + d_off;
                const long long dstride = a.dsrc_stride;
                char* dnext = static_cast<char*>(a.dsrc[0]) + row_off;  // used when evenly spaced
                for (int g0 = 0; g0 < S; g0 += G) {
                    const int gs = min(G, S - g0);
                    if (!res) mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_bwdc_error, kSiteBwdConsumer);
                    uint32_t dep = 0;
                    uint32_t rowa = base;
#pragma unroll 2
                    for (int r = 0; r < gs; ++r) {
                        const int s = g0 + r;
                        // one broadcast load of the source's three coefficients
                        const float4 cf = lds128f(ctab_s + 16u * static_cast<uint32_t>(s));
                        const float2 al2 = make_float2(cf.x, cf.x), k12 = make_float2(cf.y, cf.y),
                                     k22 = make_float2(cf.z, cf.z);
                        char* drow = dstride ? dnext : static_cast<char*>(a.dsrc[s]) + row_off;
                        dnext += dstride;
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            if (FULL || lcol[i] >= 0) {
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
                                if (ATTNRES_IN_BOUNDS(n < N && s < S && 8 * (v0 + lcol[i]) + 8 <= D, &g_bwdc_error))
                                st_global_v4_policy(drow + static_cast<long long>(i) * vstep,
                                                    make_uint4(pack_f2(dv[0]), pack_f2(dv[1]), pack_f2(dv[2]), pack_f2(dv[3])),
                                                    st_pol);
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
        }

        // ------------------------------ this CTA's columns of the cluster's partial row
        const int R = a.R;
        const int W = R + (NORM != 0 ? D : 0);
        float* my_part = a.part + static_cast<size_t>(cid) * W;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (FULL || lcol[i] >= 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 8 * (v0 + lcol[i]) + e;
                    const float dqv = (e & 1) ? dq_acc[i][e >> 1].y : dq_acc[i][e >> 1].x;
                    const float dwv = (e & 1) ? dw_acc[i][e >> 1].y : dw_acc[i][e >> 1].x;
                    if (!ATTNRES_IN_BOUNDS(cid < a.part_rows && j < D && (!((kmask[i] >> e) & 1u) || (j >= ko && j - ko < R)),
                                           &g_bwdc_error))
                        continue;
                    if ((kmask[i] >> e) & 1u) my_part[j - ko] = a.scale * dqv;  // dq = scale * sum_s c1_s t_s
                    if (NORM != 0) my_part[R + j] = dwv;
                }
            }
        }
        __syncwarp();
    }
    // no CTA leaves while a peer may still write into its exchange buffers
    cluster_sync_all();
}

template <int VPT, bool KEYALL, int NORM, int NJ, bool FULL>
cudaLaunchConfig_t cluster_config(const Plan& plan, int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>((plan.b_ncw + 1) * 32));
    cfg.dynamicSmemBytes = plan.smem_bwd;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(plan.cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int VPT, bool KEYALL, int NORM, int NJ, bool FULL>
struct LaunchFn {
    static cudaError_t run(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
        auto kern = attnres_bwd_cluster_kernel<VPT, KEYALL, NORM, NJ, FULL>;
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(plan.smem_bwd));
        if (err != cudaSuccess) return err;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = cluster_config<VPT, KEYALL, NORM, NJ, FULL>(plan, plan.grid, stream, attr);
        // may start during the previous kernel's tail (it waits before any global access)
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, kern, a);
        if (err != cudaSuccess) return err;
        const int W = a.R + (a.out_norm ? a.D : 0);
        return launch_finalize(a.part, plan.nparts, a.R, W, a.dq, a.dq_f32, a.dw_o, a.dw_o_f32, stream);
    }
    static cudaError_t fail() { return cudaErrorInvalidConfiguration; }
};

template <int VPT, bool KEYALL, int NORM, int NJ, bool FULL>
struct OccupancyFn {
    static int run(const Plan& plan) {
        auto kern = attnres_bwd_cluster_kernel<VPT, KEYALL, NORM, NJ, FULL>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(plan.smem_bwd)) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = cluster_config<VPT, KEYALL, NORM, NJ, FULL>(plan, plan.cl, nullptr, attr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return n;
    }
    static int fail() { return 0; }
};

// One instantiation per (vectors per thread, all channels keys, output-norm
// mode, source groups); `Fn` launches or queries occupancy.
template <template <int, bool, int, int, bool> class Fn, int VPT, bool KA, int NM, typename... Args>
auto pick_nj(bool one, bool full, Args&&... args) {
    if (full) return one ? Fn<VPT, KA, NM, 1, true>::run(args...) : Fn<VPT, KA, NM, 4, true>::run(args...);
    return one ? Fn<VPT, KA, NM, 1, false>::run(args...) : Fn<VPT, KA, NM, 4, false>::run(args...);
}

template <template <int, bool, int, int, bool> class Fn, int VPT, bool KA, typename... Args>
auto pick_norm(int norm, bool one, bool full, Args&&... args) {
    switch (norm) {
        case 0: return pick_nj<Fn, VPT, KA, 0>(one, full, args...);
        case 1: return pick_nj<Fn, VPT, KA, 1>(one, full, args...);
        case 2: return pick_nj<Fn, VPT, KA, 2>(one, full, args...);
        default: return Fn<VPT, KA, 0, 1, false>::fail();
    }
}

// full: every consumer thread owns whole 16-byte vectors of the slice (no
// per-vector ownership checks compiled in).
template <template <int, bool, int, int, bool> class Fn, typename... Args>
auto dispatch(int vpt, bool keyall, int norm, int S, bool full, Args&&... args) {
    const bool one = S <= 32;
    if (vpt == 1)
        return keyall ? pick_norm<Fn, 1, true>(norm, one, full, args...) : pick_norm<Fn, 1, false>(norm, one, full, args...);
    if (vpt == 2)
        return keyall ? pick_norm<Fn, 2, true>(norm, one, full, args...) : pick_norm<Fn, 2, false>(norm, one, full, args...);
    return Fn<1, true, 0, 1, false>::fail();
}

}  // namespace

cudaError_t launch_bwd_cluster(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    // output norm: o rebuilt from the rows when they are resident (free) or no
    // saved copy was passed; the caller's FP32 o saves a streamed pass otherwise
    const int norm = !a.out_norm ? 0 : ((a.resident || !a.o_pre) ? 1 : 2);
    const bool full = plan.slice / 8 == plan.b_vpt * 32 * plan.b_ncw;
    return dispatch<LaunchFn>(plan.b_vpt, a.R == a.D, norm, a.S, full, plan, a, stream);
}

int bwd_cluster_max_active(const Plan& plan, bool keyall, bool norm, int S) {
    // cached per device and launch shape (an occupancy query per call would
    // add host time to every backward)
    struct Entry {
        int dev, vpt, ncw, cl, smem, keyall, norm, one, full, n;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool full = plan.slice / 8 == plan.b_vpt * 32 * plan.b_ncw;
    const Entry key{dev, plan.b_vpt, plan.b_ncw, plan.cl, static_cast<int>(plan.smem_bwd), keyall, norm, S <= 32, full, 0};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        const Entry& e = cache[i];
        if (e.dev == key.dev && e.vpt == key.vpt && e.ncw == key.ncw && e.cl == key.cl && e.smem == key.smem &&
            e.keyall == key.keyall && e.norm == key.norm && e.one == key.one && e.full == key.full)
            return e.n;
    }
    const int n = dispatch<OccupancyFn>(plan.b_vpt, keyall, norm ? 1 : 0, S, full, plan);
    if (used < 64) {
        cache[used] = key;
        cache[used].n = n;
        ++used;
    }
    return n;
}

unsigned take_bwd_error_cluster() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwdc_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_bwdc_error, &zero, sizeof zero);
    return v;
}

}  // namespace attnres
