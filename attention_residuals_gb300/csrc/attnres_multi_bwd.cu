// attnres_multi_bwd.cu -- backward kernel of the multi-query read.
//
// Each query m is an independent read of the same sources ("Fast Attention
// Residuals", section "Multi-query AttnRes"), so with the forward's saved
// alpha_ms, logit z_ms and key statistics r_s (chain rule through section
// "Equation", per query):
//   da_ms  = <dy_m, v_s>,  delta_m = sum_s alpha_ms da_ms,
//   dz_ms  = alpha_ms (da_ms - delta_m)
//   b_ms   = scale r_s dz_ms,   c_s = -(r_s^2 / R) sum_m dz_ms z_ms
//   dv_s   = sum_m alpha_ms dy_m  +  on key channels: sum_m b_ms q_m + c_s t_s
//   dq_m  += sum_s b_ms t_s                      (summed over tokens)
// The sources feed every query, so their gradient is the sum over queries.
//
// GB300 mapping.  One persistent CTA per SM with up to 16 consumer warps
// (the passes below are latency-bound: more warps hide it).  A producer warp streams each
// token's S source rows (1-D TMA into a chunk ring), its M dy rows (one TMA
// group per token into a dy ring) and its saved statistics (cp.async into a
// two-slot ring).  The token stays resident for all passes:
//   dot pass: one warp per source row, lanes over the row's vectors, mixed-
//             precision bf16 FMAs against every dy row, reduce-scatter per
//             four queries;
//   coefficients: after a CTA barrier, one warp per query forms delta_m,
//             b_ms and its share of c_s into shared tables;
//   write pass: after a second barrier, thread t owns fixed 16-byte column
//             vectors; it forms dv_s for every source with the dy rows and
//             query vectors held in registers (queries in register blocks of
//             MB when M > MB), stores each row once, and accumulates its dq
//             columns.
// dq: with one register block the per-thread dq sums stay in registers for
// all of the CTA's tokens; with several they accumulate in shared memory.
// Each CTA writes one FP32 partial row [M * R]; a finalize kernel adds the
// rows in CTA order (bitwise reproducible).
// Selected queries (SEL: per-token rows of an [E, R] bank chosen by ids): the
// bank stays in shared memory when it fits (rows addressed by id, ids loaded
// one token ahead); with one register block each token's dq is added into
// the CTA's FP32 partial rows [E * R] in the workspace by vector reductions
// (every address has one writer thread, so the sums are reproducible), with
// several blocks it goes through the shared-memory table as for fixed queries.
// MQ > 0 fixes the query count at compile time (M = 1, 2, 4).
#include <cfloat>

#include "device_utils.cuh"
#include "kernels.cuh"
#include "launch_pdl.cuh"

namespace attnres {
namespace {

// First failed wait of any multi-query backward launch (0 = none).
__device__ unsigned int g_multi_bwd_error = 0;

__device__ __forceinline__ float2 key_part(const float2 x, unsigned mask, int kk) {
    return make_float2((mask >> (2 * kk)) & 1u ? x.x : 0.0f, (mask >> (2 * kk + 1)) & 1u ? x.y : 0.0f);
}

template <int VPT, int MB, bool SEL, int MQ, bool FULL>
__global__ void __launch_bounds__(kMultiBwdThreads, 1) attnres_multi_bwd_kernel(const __grid_constant__ MultiBwdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int ncw = a.ncw;
    const int nct = ncw * 32;
    const int K = a.chunks;
    const int G = a.rows;
    const int S = a.S;
    const int M = MQ > 0 ? MQ : a.M;  // MQ > 0: the query count is fixed at compile time
    const int DS = a.dy_slots;
    const int s_pad = a.s_pad, m_pad = a.m_pad;
    const int nmb = (M + MB - 1) / MB;
    const bool selected = SEL;         // per-token queries from a bank (a.ids set)
    // one register block: q and the token's dq live in registers (fixed
    // queries: dq for the whole launch; selected queries: q reloaded and dq
    // added to the bank row's shared-memory sums per token); several blocks:
    // q comes from shared memory per row and dq sums go to shared memory
    const bool regblock = nmb == 1;
    // selected queries with one register block add each token's dq straight
    // into this CTA's workspace row (vector reductions to L2, no return value)
    const bool dq_in_smem = !regblock;
    const int QR = selected ? a.E : M;       // rows of dq (queries or bank rows)
    // selected queries with one register block: the whole bank (and a zero
    // row, index E) stays in shared memory, addressed by the token's ids
    const bool bank_res = selected && regblock && a.bank_rows > 0;
    const MultiLayout L = make_multi_layout(K, G, a.slot_bytes, M, DS, s_pad, m_pad, a.nkv, dq_in_smem ? a.nkv : 0,
                                            true, QR, a.bank_rows > 0 ? max(a.bank_rows, m_pad) : -1);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* dyfull = reinterpret_cast<uint64_t*>(smem + L.dyfull);
    uint64_t* dyempty = reinterpret_cast<uint64_t*>(smem + L.dyempty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    float* tok = reinterpret_cast<float*>(smem + L.tok);
    float* da_t = reinterpret_cast<float*>(smem + L.tab);  // [m_pad][s_pad]
    float* al_t = da_t + m_pad * s_pad;                    // [s_pad][m_pad]
    float* b_t = al_t + s_pad * m_pad;                     // [s_pad][m_pad]
    float* zr_t = b_t + s_pad * m_pad;                     // [m_pad][s_pad]
    // dq sums (several blocks, or bank rows): row m, key vector v, channel e at
    // dqsm[m * nkv * 8 + (e / 4) * nkv * 4 + v * 4 + e % 4] -- two planes of
    // four channels, so a warp's 16-byte accesses to consecutive vectors are
    // free of bank conflicts
    float* dqsm = reinterpret_cast<float*>(smem + L.dqsm);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int tstride = static_cast<int>(L.tstride);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int D = a.D;
    const int MS = M * S;
    const uint32_t sb = static_cast<uint32_t>(a.slot_bytes);
    const uint32_t cb = static_cast<uint32_t>(G) * sb;
    const int cpt = (S + G - 1) / G;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, ncw);
        }
        for (int k = 0; k < DS; ++k) {
            mbar_init(dyfull + k, 1);
            mbar_init(dyempty + k, ncw);
        }
        for (int k = 0; k < kMultiTokSlots; ++k) {
            mbar_init(tfull + k, 32);
            mbar_init(tempty + k, ncw);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    // coefficients of padded queries stay zero; dq sums start at zero
    for (int i = threadIdx.x; i < 2 * s_pad * m_pad; i += blockDim.x) al_t[i] = 0.0f;
    if (dq_in_smem)
        for (int i = threadIdx.x; i < QR * a.nkv * 8; i += blockDim.x) dqsm[i] = 0.0f;
    __syncthreads();
    // set-up above overlaps the previous kernel's tail; global memory only after it
    pdl_wait();
    pdl_launch_dependents();

    if (warp == ncw) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
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
            // saved statistics -> tok[ts] (all 32 lanes arrive on tfull)
            mbar_wait(tempty + ts, tphase ^ 1u, abort_flag, &g_multi_bwd_error, kSiteBwdProducer);
            float* dst = tok + ts * tstride;
            for (int e = lane; e < MS; e += 32) {
                cp_async_4(dst + e, a.alpha + n * MS + e);
                cp_async_4(dst + MS + e, a.logit + n * MS + e);
            }
            for (int e = lane; e < S; e += 32) cp_async_4(dst + 2 * MS + e, a.rstd + n * S + e);
            cp_async_arrive_noinc(tfull + ts);
            if (++ts == kMultiTokSlots) {
                ts = 0;
                tphase ^= 1u;
            }
            if (lane == 0) {
                if (mbar_wait(dyempty + dk, dphase ^ 1u, abort_flag, &g_multi_bwd_error, kSiteBwdProducer)) {
                    mbar_arrive_expect_tx(dyfull + dk, row_bytes * static_cast<uint32_t>(M));
                    for (int m = 0; m < M; ++m)
                        tma_load_1d(dyring + (dk * M + m) * sb, a.dy + m * a.dy_ms + n * a.dy_ns, row_bytes,
                                    dyfull + dk, pol);
                    ++dy_issued;
                    if (++dk == DS) {
                        dk = 0;
                        dphase ^= 1u;
                    }
                }
                for (int g0 = 0; g0 < S && !*abort_flag; g0 += G) {
                    const int gs = min(G, S - g0);
                    if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_multi_bwd_error, kSiteBwdProducer)) break;
                    mbar_arrive_expect_tx(full + k, row_bytes * static_cast<uint32_t>(gs));
                    for (int r = 0; r < gs; ++r) {
                        const unsigned char* src =
                            static_cast<const unsigned char*>(a.src[g0 + r]) + (n * a.src_ld) * 2;
                        tma_load_1d(ring + k * cb + r * sb, src, row_bytes, full + k, pol);
                    }
                    ++issued;
                    if (++k == K) {
                        k = 0;
                        phase ^= 1u;
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
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_bwd_error, kSiteDrain);
            }
            for (int c = 0; c < DS && c < dy_issued; ++c) {
                const long long fills = (dy_issued - 1 - c) / DS + 1;
                volatile int no_abort = 0;
                mbar_wait(dyfull + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_bwd_error, kSiteDrain);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ncv = D >> 3;
    const int ko = a.ko, kend = a.ko + a.R;
    const int kv0 = a.kv0, nkv = a.nkv;
    const int kw = nkv * 8;
    // this CTA's FP32 partial rows: part[cta][m * R + (c - ko)], m < QR
    float* prow = a.part + static_cast<long long>(blockIdx.x) * QR * a.R;
    // 16-byte reductions need the vector's first key channel 4-aligned in the row
    const bool red_vec = ((ko & 3) == 0) && ((a.R & 3) == 0);
    // dq of one owned key vector into bank row m of this CTA's partial rows
    auto dq_red = [&](int m, int c, unsigned msk, const float2 (&d)[4]) {
        float* p = prow + static_cast<long long>(m) * a.R + (8 * c - ko);
        if (red_vec && msk == 0xffu) {
            red_add_v4(p, d[0].x, d[0].y, d[1].x, d[1].y);
            red_add_v4(p + 4, d[2].x, d[2].y, d[3].x, d[3].y);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if ((msk >> e) & 1u) red_add_f32(p + e, (e & 1) ? d[e >> 1].y : d[e >> 1].x);
        }
    };
    // dq sums of one owned key vector (eight channels as four pairs) into row m
    auto dq_add = [&](int m, int v, const float2 (&d)[4]) {
        float4* p0 = reinterpret_cast<float4*>(dqsm + m * kw + 4 * v);
        float4* p1 = reinterpret_cast<float4*>(dqsm + m * kw + (kw >> 1) + 4 * v);
        float4 x = *p0, y = *p1;
        x.x += d[0].x; x.y += d[0].y; x.z += d[1].x; x.w += d[1].y;
        y.x += d[2].x; y.y += d[2].y; y.z += d[3].x; y.w += d[3].y;
        *p0 = x;
        *p1 = y;
    };
    const uint32_t kwb = static_cast<uint32_t>(nkv) * 16u;
    int col[VPT];
    int kvi[VPT];        // key vector index within the key window, -1 outside
    unsigned kmask[VPT];  // key channels of the vector (bit e = channel 8*col + e)
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * nct;
        col[i] = (FULL || c < ncv) ? c : -1;
        kvi[i] = (col[i] >= kv0 && col[i] < kv0 + nkv) ? col[i] - kv0 : -1;
        unsigned m = 0;
        for (int e = 0; e < 8; ++e) {
            const int j = 8 * c + e;
            if (kvi[i] >= 0 && j >= ko && j < kend) m |= 1u << e;
        }
        kmask[i] = m;
    }
    if (regblock && selected) {
        // this thread's key channels of the CTA's partial rows start at zero
        // (the same thread adds to them later, so program order suffices)
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (kvi[i] < 0) continue;
            for (int m = 0; m < QR; ++m)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if ((kmask[i] >> e) & 1u) prow[static_cast<long long>(m) * a.R + (8 * col[i] + e - ko)] = 0.0f;
        }
    }
    const float inv_r = 1.0f / static_cast<float>(a.R);
    const float scale = a.scale;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t voff = static_cast<uint32_t>(col[0] < 0 ? 0 : col[0]) * 16u;
    const uint32_t vstep = static_cast<uint32_t>(nct) * 16u;
    const uint32_t ring_raw = sbase + L.ring;
    const uint32_t ring_lo = ring_raw + voff;
    const uint32_t dy_raw = sbase + L.dyring;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    const uint32_t dyfull_s = sbase + L.dyfull;
    const uint32_t dyempty_s = sbase + L.dyempty;
    const uint32_t tfull_s = sbase + L.tfull;
    const uint32_t tempty_s = sbase + L.tempty;
    const uint32_t qsm_s = sbase + L.qsm;
    // Bank row of slot m of token n (selected queries); -1 for an id outside
    // [0, E), which is recorded as an error and contributes nothing.
    auto bank_row = [&](long long n, int m) -> int {
        const long long id = a.ids[n * M + m];
        if (id < 0 || id >= a.E) {
            atomicCAS(&g_multi_bwd_error, 0u, static_cast<unsigned>(kSiteBadId));
            return -1;
        }
        return static_cast<int>(id);
    };
    // queries by key channel into shared memory (token n's bank rows when selected)
    const bool q_vec = ((ko | kend) & 7) == 0 && (reinterpret_cast<uintptr_t>(a.q) & 15u) == 0;
    auto load_q = [&](long long n) {
        uint16_t* qsm = reinterpret_cast<uint16_t*>(smem + L.qsm);
        if (q_vec) {
            // aligned key: whole 16-byte vectors of each query (bank) row
#pragma unroll 4
            for (int i = threadIdx.x; i < m_pad * nkv; i += nct) {
                const int m = i / nkv;
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (m < M) {
                    const int row = selected ? bank_row(n, m) : m;
                    if (row >= 0) w = ld_global_nc_v4(a.q + static_cast<long long>(row) * a.R + 8 * (i - m * nkv));
                }
                *reinterpret_cast<uint4*>(qsm + 8 * i) = w;
            }
            return;
        }
        for (int i = threadIdx.x; i < m_pad * kw; i += nct) {
            const int m = i / kw;
            const int c = 8 * kv0 + (i - m * kw);
            uint16_t v = 0;
            if (m < M && c >= ko && c < kend) {
                const int row = selected ? bank_row(n, m) : m;
                if (row >= 0) v = a.q[static_cast<long long>(row) * a.R + (c - ko)];
            }
            qsm[i] = v;
        }
    };
    if (!selected) load_q(0);
    if (bank_res) {
        uint16_t* qsm = reinterpret_cast<uint16_t*>(smem + L.qsm);
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
    // Resident bank: lane m < M of every warp holds the bank row of slot m,
    // loaded one token ahead; an id outside [0, E) is recorded and reads the
    // zero row (and adds to no dq row).
    auto row_of = [&](long long id) -> int {
        if (id < 0 || id >= a.E) {
            atomicCAS(&g_multi_bwd_error, 0u, static_cast<unsigned>(kSiteBadId));
            return a.E;
        }
        return static_cast<int>(id);
    };
    long long id_next = (bank_res && lane < M) ? a.ids[static_cast<long long>(blockIdx.x) * M + lane] : 0;
    // One register block: the query values at the owned key vectors and the
    // dq sums live in registers for the whole launch.
    float2 qf[MB][VPT][4];
    float2 dqa[MB][VPT][4];
#pragma unroll
    for (int j = 0; j < MB; ++j)
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float qv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = 2 * kk + h;
                    const bool in = regblock && !selected && j < M && ((kmask[i] >> e) & 1u);
                    qv[h] = in ? bf16_bits_to_float(a.q[static_cast<long long>(j) * a.R + (8 * col[i] + e - ko)])
                               : 0.0f;
                }
                qf[j][i][kk] = make_float2(qv[0], qv[1]);
                dqa[j][i][kk] = make_float2(0.0f, 0.0f);
            }
    named_bar_sync(1, nct);

    int ck = 0;
    uint32_t cphase = 0;
    int dk = 0;
    uint32_t dphase = 0;
    int ts = 0;
    uint32_t tphase = 0;
    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        int my_row = 0;
        if (bank_res) {
            my_row = lane < M ? row_of(id_next) : a.E;
            const long long nn = n + gridDim.x;
            id_next = (lane < M && nn < N) ? a.ids[nn * M + lane] : 0;
        }
        {
            int k = ck;
            uint32_t ph = cphase;
            for (int c = 0; c < cpt; ++c) {
                mbar_wait_s(full_s + 8u * k, ph, abort_flag, &g_multi_bwd_error, kSiteBwdConsumer);
                if (++k == K) {
                    k = 0;
                    ph ^= 1u;
                }
            }
            mbar_wait_s(dyfull_s + 8u * dk, dphase, abort_flag, &g_multi_bwd_error, kSiteBwdConsumer);
            mbar_wait_s(tfull_s + 8u * ts, tphase, abort_flag, &g_multi_bwd_error, kSiteBwdTokStat);
        }
        const uint32_t dyb = dy_raw + static_cast<uint32_t>(dk * M) * sb;
        // dot pass: da_ms = <dy_m, v_s>, one warp per source row
        for (int r = warp; r < S; r += ncw) {
            int kc = ck + r / G;
            if (kc >= K) kc -= K;
            const uint32_t row = ring_raw + static_cast<uint32_t>(kc) * cb + static_cast<uint32_t>(r % G) * sb;
            for (int m4 = 0; m4 < M; m4 += 4) {
                // two vectors per step into separate sums: half the FMA chain
                float t[4][2], u[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) t[j][0] = t[j][1] = u[j][0] = u[j][1] = 0.0f;
                int v = lane;
                for (; v + 32 < ncv; v += 64) {
                    const uint4 x0 = lds128(row + 16u * v);
                    const uint4 x1 = lds128(row + 16u * (v + 32));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (m4 + j < M) {
                            const uint32_t yrow = dyb + static_cast<uint32_t>(m4 + j) * sb;
                            const uint4 y0 = lds128(yrow + 16u * v);
                            const uint4 y1 = lds128(yrow + 16u * (v + 32));
                            bf16_dot8(x0, y0, t[j][0], t[j][1]);
                            bf16_dot8(x1, y1, u[j][0], u[j][1]);
                        }
                    }
                }
                if (v < ncv) {
                    const uint4 x0 = lds128(row + 16u * v);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (m4 + j < M) {
                            const uint4 y0 = lds128(dyb + static_cast<uint32_t>(m4 + j) * sb + 16u * v);
                            bf16_dot8(x0, y0, t[j][0], t[j][1]);
                        }
                    }
                }
                float part[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) part[j] = (t[j][0] + t[j][1]) + (u[j][0] + u[j][1]);
                warp_reduce_scatter<4>(part, lane);
                if ((lane & 7) == 0) {
                    const int e = lane >> 3;
                    if (m4 + e < M) da_t[(m4 + e) * s_pad + r] = part[0];
                }
            }
        }
        named_bar_sync(1, nct);
        // every warp is past the previous token's write and dq passes: the
        // token's bank rows can replace the queries in shared memory
        if (selected && !bank_res) load_q(n);
        // coefficients.  M <= 4: warp 0 forms every query's and also
        // c_s = sum_m zr_ms (into zr_t[s]); otherwise one warp per query and
        // the write pass adds the zr rows itself.
        const bool one_warp_coef = M <= 4;
        if (one_warp_coef) {
            if (warp == 0) {
                const float* tk = tok + ts * tstride;
                float cs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int m = 0; m < M; ++m) {
                    float al[4], da[4], z[4], rs[4];
                    float p = 0.0f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = lane + 32 * i;
                        al[i] = da[i] = z[i] = rs[i] = 0.0f;
                        if (s < S) {
                            al[i] = tk[m * S + s];
                            z[i] = tk[MS + m * S + s];
                            rs[i] = tk[2 * MS + s];
                            da[i] = da_t[m * s_pad + s];
                            p = fmaf(al[i], da[i], p);
                        }
                    }
                    const float delta = warp_sum(p);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = lane + 32 * i;
                        if (s < S) {
                            const float dz = al[i] * (da[i] - delta);
                            al_t[s * m_pad + m] = al[i];
                            b_t[s * m_pad + m] = scale * rs[i] * dz;
                            cs[i] += -(dz * z[i]) * (rs[i] * rs[i]) * inv_r;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (lane + 32 * i < S) zr_t[lane + 32 * i] = cs[i];
            }
        } else {
            const float* tk = tok + ts * tstride;
            for (int m = warp; m < M; m += ncw) {
                float al[4], da[4], z[4], rs[4];
                float p = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int s = lane + 32 * i;
                    al[i] = da[i] = z[i] = rs[i] = 0.0f;
                    if (s < S) {
                        al[i] = tk[m * S + s];
                        z[i] = tk[MS + m * S + s];
                        rs[i] = tk[2 * MS + s];
                        da[i] = da_t[m * s_pad + s];
                        p = fmaf(al[i], da[i], p);
                    }
                }
                const float delta = warp_sum(p);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int s = lane + 32 * i;
                    if (s < S) {
                        const float dz = al[i] * (da[i] - delta);
                        al_t[s * m_pad + m] = al[i];
                        b_t[s * m_pad + m] = scale * rs[i] * dz;
                        zr_t[m * s_pad + s] = -(dz * z[i]) * (rs[i] * rs[i]) * inv_r;
                    }
                }
            }
        }
        named_bar_sync(1, nct);
        if (lane == 0) mbar_arrive_s(tempty_s + 8u * ts);

        // write pass: dv_s for every source row, one store per row
        if (regblock) {
            if (selected) {
                // this token's bank rows: query values at the owned key vectors
                // from shared memory, and a fresh dq sum
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    uint32_t qrow = qsm_s + static_cast<uint32_t>(j) * kwb;
                    if (bank_res) {
                        const int r = __shfl_sync(0xffffffffu, my_row, j);
                        qrow = qsm_s + static_cast<uint32_t>(j < M ? r : a.E) * kwb;
                    }
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        uint4 qv = make_uint4(0u, 0u, 0u, 0u);
                        if (kvi[i] >= 0) qv = lds128(qrow + 16u * kvi[i]);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            qf[j][i][kk] = key_part(bf2_to_f2(u4_get(qv, kk)), kmask[i], kk);
                            dqa[j][i][kk] = make_float2(0.0f, 0.0f);
                        }
                    }
                }
            }
            float2 dyf[MB][VPT][4];
            uint32_t ddep = 0;
#pragma unroll
            for (int j = 0; j < MB; ++j)
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    uint4 yv = make_uint4(0u, 0u, 0u, 0u);
                    if (j < M && (FULL || col[i] >= 0)) {
                        yv = lds128(dyb + static_cast<uint32_t>(j) * sb + voff + i * vstep);
                        ddep ^= yv.x;
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) dyf[j][i][kk] = bf2_to_f2(u4_get(yv, kk));
                }
            __syncwarp();
            if (lane == 0) mbar_arrive_after(dyempty_s + 8u * dk, ddep);
            int kc = ck;
            for (int r0 = 0; r0 < S; r0 += G) {
                const int rn = min(G, S - r0);
                uint32_t dep = 0;
                uint32_t rowa = ring_lo + static_cast<uint32_t>(kc) * cb;
#pragma unroll 2
                for (int r = 0; r < rn; ++r) {
                    const int s = r0 + r;
                    float2 al2[MB], bl2[MB];
                    {
                        // the row's first four weights / b coefficients in one 16-byte load each
                        const float4 a4 = *reinterpret_cast<const float4*>(al_t + s * m_pad);
                        const float4 b4 = *reinterpret_cast<const float4*>(b_t + s * m_pad);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
                        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                        for (int j = 0; j < MB; ++j) {
                            al2[j] = make_float2(av[j], av[j]);
                            bl2[j] = make_float2(bv[j], bv[j]);
                        }
                    }
                    float cs = zr_t[s];
                    if (!one_warp_coef)
                        for (int m = 1; m < M; ++m) cs += zr_t[m * s_pad + s];
                    const float2 cs2 = make_float2(cs, cs);
                    uint16_t* drow = static_cast<uint16_t*>(a.dsrc[s]) + n * a.dsrc_ld;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        if (FULL || col[i] >= 0) {
                            const uint4 xv = lds128(rowa + i * vstep);
                            dep ^= xv.x;
                            float2 o[4];
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                o[kk] = fmul2(al2[0], dyf[0][i][kk]);
#pragma unroll
                                for (int j = 1; j < MB; ++j) o[kk] = ffma2(al2[j], dyf[j][i][kk], o[kk]);
                            }
                            if (kvi[i] >= 0) {
                                const bool whole = kmask[i] == 0xffu;  // every channel a key channel
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const float2 x2 = bf2_to_f2(u4_get(xv, kk));
                                    const float2 xk = whole ? x2 : key_part(x2, kmask[i], kk);
                                    o[kk] = ffma2(cs2, xk, o[kk]);
#pragma unroll
                                    for (int j = 0; j < MB; ++j) {
                                        o[kk] = ffma2(bl2[j], qf[j][i][kk], o[kk]);
                                        dqa[j][i][kk] = ffma2(bl2[j], xk, dqa[j][i][kk]);
                                    }
                                }
                            }
                            if (ATTNRES_IN_BOUNDS(n < a.N && s < a.S && 8 * col[i] + 8 <= a.D, &g_multi_bwd_error))
                            st_global_cs_v4(drow + 8 * col[i], make_uint4(pack_f2(o[0]), pack_f2(o[1]),
                                                                          pack_f2(o[2]), pack_f2(o[3])));
                        }
                    }
                    rowa += sb;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_after(empty_s + 8u * kc, dep);
                if (++kc == K) kc = 0;
            }
            if (selected) {
                // the token's dq into its bank rows' sums (own columns only)
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    if (j >= M) continue;
                    int row;
                    if (bank_res) {
                        row = __shfl_sync(0xffffffffu, my_row, j);
                        if (row >= a.E) row = -1;
                    } else {
                        row = bank_row(n, j);
                    }
                    if (row < 0) continue;
#pragma unroll
                    for (int i = 0; i < VPT; ++i)
                        if (kvi[i] >= 0) dq_red(row, col[i], kmask[i], dqa[j][i]);
                }
            }
        } else {
            // several register blocks: dy and query vectors come from shared
            // memory for every row, dq sums go to shared memory afterwards
            uint32_t ddep = 0;
            {
                int kc = ck;
                for (int r0 = 0; r0 < S; r0 += G) {
                    const int rn = min(G, S - r0);
                    uint32_t rowa = ring_lo + static_cast<uint32_t>(kc) * cb;
                    for (int r = 0; r < rn; ++r) {
                        const int s = r0 + r;
                        float cs = zr_t[s];
                        if (!one_warp_coef)
                            for (int m = 1; m < M; ++m) cs += zr_t[m * s_pad + s];
                        const float2 cs2 = make_float2(cs, cs);
                        uint16_t* drow = static_cast<uint16_t*>(a.dsrc[s]) + n * a.dsrc_ld;
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            if (!FULL && col[i] < 0) continue;
                            float2 o[4];
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) o[kk] = make_float2(0.0f, 0.0f);
                            for (int mb = 0; mb < M; mb += MB) {
#pragma unroll
                                for (int j = 0; j < MB; ++j) {
                                    if (mb + j < M) {
                                        const float av = al_t[s * m_pad + mb + j];
                                        const float2 al2 = make_float2(av, av);
                                        const uint4 yv =
                                            lds128(dyb + static_cast<uint32_t>(mb + j) * sb + voff + i * vstep);
                                        ddep ^= yv.x;
#pragma unroll
                                        for (int kk = 0; kk < 4; ++kk)
                                            o[kk] = ffma2(al2, bf2_to_f2(u4_get(yv, kk)), o[kk]);
                                        if (kvi[i] >= 0) {
                                            const float bv = b_t[s * m_pad + mb + j];
                                            const float2 bl2 = make_float2(bv, bv);
                                            const uint4 qv = lds128(qsm_s + static_cast<uint32_t>(mb + j) * kwb +
                                                                    16u * static_cast<uint32_t>(kvi[i]));
#pragma unroll
                                            for (int kk = 0; kk < 4; ++kk)
                                                o[kk] = ffma2(bl2, bf2_to_f2(u4_get(qv, kk)), o[kk]);
                                        }
                                    }
                                }
                            }
                            if (kvi[i] >= 0) {
                                const uint4 xv = lds128(rowa + i * vstep);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    o[kk] = ffma2(cs2, key_part(bf2_to_f2(u4_get(xv, kk)), kmask[i], kk), o[kk]);
                            }
                            if (ATTNRES_IN_BOUNDS(n < a.N && s < a.S && 8 * col[i] + 8 <= a.D, &g_multi_bwd_error))
                            st_global_cs_v4(drow + 8 * col[i], make_uint4(pack_f2(o[0]), pack_f2(o[1]),
                                                                          pack_f2(o[2]), pack_f2(o[3])));
                        }
                        rowa += sb;
                    }
                    if (++kc == K) kc = 0;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_after(dyempty_s + 8u * dk, ddep);
            // dq pass: one register block of queries at a time
            uint32_t dep = 0;
            for (int mb = 0; mb < M; mb += MB) {
                float2 dqt[MB][VPT][4];
#pragma unroll
                for (int j = 0; j < MB; ++j)
#pragma unroll
                    for (int i = 0; i < VPT; ++i)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) dqt[j][i][kk] = make_float2(0.0f, 0.0f);
                int kc = ck;
                for (int r0 = 0; r0 < S; r0 += G) {
                    const int rn = min(G, S - r0);
                    uint32_t rowa = ring_lo + static_cast<uint32_t>(kc) * cb;
                    for (int r = 0; r < rn; ++r) {
                        const int s = r0 + r;
                        float2 bl2[MB];
#pragma unroll
                        for (int j = 0; j < MB; ++j) {
                            const float bv = b_t[s * m_pad + mb + j];
                            bl2[j] = make_float2(bv, bv);
                        }
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            if (kvi[i] >= 0) {
                                const uint4 xv = lds128(rowa + i * vstep);
                                dep ^= xv.x;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const float2 xk = key_part(bf2_to_f2(u4_get(xv, kk)), kmask[i], kk);
#pragma unroll
                                    for (int j = 0; j < MB; ++j) dqt[j][i][kk] = ffma2(bl2[j], xk, dqt[j][i][kk]);
                                }
                            }
                        }
                        rowa += sb;
                    }
                    if (++kc == K) kc = 0;
                }
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    if (mb + j >= M) continue;
                    const int row = selected ? bank_row(n, mb + j) : mb + j;
                    if (row < 0) continue;
#pragma unroll
                    for (int i = 0; i < VPT; ++i)
                        if (kvi[i] >= 0) dq_add(row, kvi[i], dqt[j][i]);
                }
            }
            // the chunks held every row until the dq pass
            int kc = ck;
            for (int c = 0; c < cpt; ++c) {
                __syncwarp();
                if (lane == 0) mbar_arrive_after(empty_s + 8u * kc, dep);
                if (++kc == K) kc = 0;
            }
        }
        for (int c = 0; c < cpt; ++c) {
            if (++ck == K) {
                ck = 0;
                cphase ^= 1u;
            }
        }
        if (++dk == DS) {
            dk = 0;
            dphase ^= 1u;
        }
        if (++ts == kMultiTokSlots) {
            ts = 0;
            tphase ^= 1u;
        }
    }

    // the partial rows already hold the reductions of selected queries with one block
    if (!(regblock && selected)) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (kvi[i] < 0) continue;
            for (int m = 0; m < QR; ++m) {
                float v8[8];
                if (regblock && !selected) {
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        if (j == m) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                v8[2 * kk] = dqa[j][i][kk].x;
                                v8[2 * kk + 1] = dqa[j][i][kk].y;
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v8[e] = dqsm[m * kw + (e >> 2) * (kw >> 1) + 4 * kvi[i] + (e & 3)];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if ((kmask[i] >> e) & 1u) prow[m * a.R + (8 * col[i] + e - ko)] = v8[e];
            }
        }
    }
}

template <int VPT, int MB, bool SEL, int MQ, bool FULL>
cudaError_t launch_t(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_multi_bwd_kernel<VPT, MB, SEL, MQ, FULL>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_bwd));
    if (err != cudaSuccess) return err;
    err = launch_pdl(kern, dim3(plan.grid), dim3((plan.b_ncw + 1) * 32), plan.smem_bwd, stream, a);
    if (err != cudaSuccess) return err;
    const int W = (a.ids ? a.E : a.M) * a.R;
    return launch_finalize(a.part, plan.grid, W, W, const_cast<uint16_t*>(a.dq), a.dq_f32, nullptr, nullptr,
                           stream);
}

template <int VPT, int MB, bool SEL, int MQ, bool FULL>
int occupancy_one(const MultiPlan& plan) {
    auto kern = attnres_multi_bwd_kernel<VPT, MB, SEL, MQ, FULL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(plan.smem_bwd)) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (plan.b_ncw + 1) * 32, plan.smem_bwd) != cudaSuccess)
        return 0;
    return n;
}

// CTAs per SM that both forms a launch may pick fit (selected queries have two)
template <int VPT, int MB, bool SEL, int MQ>
int occupancy_t(const MultiPlan& plan) {
    const int n = occupancy_one<VPT, MB, SEL, MQ, false>(plan);
    if constexpr (SEL) {
        const int f = occupancy_one<VPT, MB, SEL, MQ, true>(plan);
        return f < n ? f : n;
    }
    return n;
}

}  // namespace

unsigned take_multi_bwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_bwd_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_bwd_error, &zero, sizeof zero);
    return v;
}

namespace {
// With a fixed query count only the block size the planner derives from it
// (multi_bwd_mb) is instantiated.
template <int VPT, int MB, bool SEL, int MQ>
constexpr bool bwd_reachable() {
    return MQ == 0 || MB == multi_bwd_mb(MQ, VPT);
}

template <bool SEL, int MQ>
int bwd_occupancy_mq(const MultiPlan& plan) {
#define ATTNRES_OCC(V, B)                                                        \
    case V * 10 + B:                                                             \
        if constexpr (bwd_reachable<V, B, SEL, MQ>()) return occupancy_t<V, B, SEL, MQ>(plan); \
        return 0;
    switch (plan.b_vpt * 10 + plan.mb_b) {
        ATTNRES_OCC(1, 1)
        ATTNRES_OCC(1, 2)
        ATTNRES_OCC(2, 1)
        default: return 0;
    }
#undef ATTNRES_OCC
}

template <bool SEL, int MQ, bool FULL>
cudaError_t launch_bwd_mq(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream) {
#define ATTNRES_LAUNCH(V, B)                                                                  \
    case V * 10 + B:                                                                          \
        if constexpr (bwd_reachable<V, B, SEL, MQ>()) return launch_t<V, B, SEL, MQ, FULL>(plan, a, stream); \
        return cudaErrorInvalidConfiguration;
    switch (plan.b_vpt * 10 + plan.mb_b) {
        ATTNRES_LAUNCH(1, 1)
        ATTNRES_LAUNCH(1, 2)
        ATTNRES_LAUNCH(2, 1)
        default: return cudaErrorInvalidConfiguration;
    }
#undef ATTNRES_LAUNCH
}

template <bool SEL>
int bwd_occupancy_sel(const MultiPlan& plan) {
    switch (plan.mq) {
        case 1: return bwd_occupancy_mq<SEL, 1>(plan);
        case 2: return bwd_occupancy_mq<SEL, 2>(plan);
        case 4: return bwd_occupancy_mq<SEL, 4>(plan);
        default: return bwd_occupancy_mq<SEL, 0>(plan);
    }
}

template <bool SEL, bool FULL>
cudaError_t launch_bwd_full(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream) {
    switch (plan.mq) {
        case 1: return launch_bwd_mq<SEL, 1, FULL>(plan, a, stream);
        case 2: return launch_bwd_mq<SEL, 2, FULL>(plan, a, stream);
        case 4: return launch_bwd_mq<SEL, 4, FULL>(plan, a, stream);
        default: return launch_bwd_mq<SEL, 0, FULL>(plan, a, stream);
    }
}

// Selected queries: whole-vector ownership compiled in when every consumer
// thread owns whole 16-byte vectors of the row (measured 1.056 -> 0.977 ms
// on K=2 slots over S=10 N=32768 D=4096 rows; the same form measured 1.7%
// slower for fixed queries, which keep the general one).
template <bool SEL>
cudaError_t launch_bwd_sel(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream) {
    if constexpr (SEL) {
        if (a.D / 8 == plan.b_vpt * 32 * plan.b_ncw) return launch_bwd_full<SEL, true>(plan, a, stream);
    }
    return launch_bwd_full<SEL, false>(plan, a, stream);
}
}  // namespace

// plan.E > 0: the selected-query kernels (a query bank and per-token ids)
int multi_bwd_occupancy(const MultiPlan& plan) {
    return plan.E > 0 ? bwd_occupancy_sel<true>(plan) : bwd_occupancy_sel<false>(plan);
}

cudaError_t launch_multi_bwd(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream) {
    return a.ids ? launch_bwd_sel<true>(plan, a, stream) : launch_bwd_sel<false>(plan, a, stream);
}

}  // namespace attnres
