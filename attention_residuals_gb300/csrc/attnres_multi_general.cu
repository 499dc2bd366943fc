// attnres_multi_general.cu -- backward of the multi-query and selected-query
// reads for any shape (S <= 128 sources, D <= 8192 channels, M <= 16
// queries), as two kernels over column blocks.
//
// Per token, with the forward's saved alpha_ms, logit z_ms and key rstd r_s
// ("Fast Attention Residuals", sections "Multi-query AttnRes" and "Equation";
// the chain rule of attnres_multi_bwd.cu):
//   da_ms = <dy_m, v_s>,  delta_m = sum_s alpha_ms da_ms,  dz_ms = alpha_ms (da_ms - delta_m)
//   b_ms  = scale r_s dz_ms,   c_s = -(r_s^2 / R) sum_m dz_ms z_ms
//   dv_s  = sum_m alpha_ms dy_m  +  on key channels: sum_m b_ms q_m + c_s t_s
//   dq_m += sum_s b_ms t_s                       (summed over tokens)
//
// Kernel A (coefficients) walks a token's rows in blocks of columns: a
// producer warp copies the block of the M dy rows and the S source rows into
// a shared-memory ring (1-D TMA, one copy per row; rows padded so ldmatrix is
// conflict-free; queries past M and sources past S read one zero row), and
// the consumer warps form DA = DY[M x D] . V[S x D]^T, a contraction over the
// whole row, with bf16 tensor-core MMAs (mma.sync m16n8k16: the products of
// bf16 operands are exact, the sums FP32).  After the last block the partial
// tiles are added in a fixed order, every query's coefficients are formed in
// FP32 and the token's table [S][alpha_s0..alpha_sM-1, b_s0..b_sM-1, c_s]
// goes to the workspace.
//
// Kernel B (gradients) gives each CTA one block of columns for a group of
// tokens.  Here the SIMT form: thread t owns column pairs of the block and
// holds the queries in pairs -- for query pair i and column c, {q_2i,
// q_2i+1}, the token's dy values and the dq sums the same way -- so each
// 16-byte load of a coefficient row gives two aligned pairs that feed the
// packed FMAs directly (per source row and column pair: 3M/2 packed FMAs
// per column, one read of the row's pair, one 4-byte store).  dq: fixed
// queries keep the sums in registers for all of the CTA's tokens and write
// one partial row per token group; selected queries add each token's sums
// into the bank rows of the group's partial row with L2 reductions (every
// address has one writer thread, so the order and the result are fixed).
// The finalize kernel adds the groups' rows in order: bitwise reproducible.
// With fixed queries, at most 16 sources and nine or more queries the plan
// takes the tensor-core gradient kernel of attnres_multi_grad_mma.cu instead.
//
// The sources and dy are read twice (once per kernel); the resident one-CTA
// kernels of attnres_multi_bwd.cu read them once and serve one or two
// queries when a token fits.
#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {
namespace {

// First failed wait of any launch of this unit (0 = none).
__device__ unsigned int g_multi_gen_error = 0;
// Sixteen zero bytes: copied behind a row block whose width is 8 modulo 16,
// so the last MMA step reads zeros there.
__device__ __align__(16) unsigned char g_zero16[16];

constexpr int kGenWarps = 8;                     // consumer warps of the gradient kernel
constexpr int kGenThreads = (kGenWarps + 1) * 32;
constexpr int kGenTokSlots = 4;                  // statistics slots of the coefficient kernel (tokens the producer may run ahead)

// ---------------------------------------------------------------- kernel A
// Shared memory: ring of `bufs` row blocks ([M dy rows][S source rows] x
// pitch bytes), one zero row that the MMAs read for queries M..15 and
// sources S..s8-1, full/empty barriers, statistics ring
// [kGenTokSlots][2*M*S + S], partial tiles [kgroups][16][s8], per-warp
// parts of the c_s sums [kCoefWarps][s8], coefficient table [S][cs]
// (queries padded to M4 = M rounded up to 4, for 16-byte loads: alpha at 0,
// b at M4, c at 2 M4; the padding stays zero).
//
// Four consumer warps and a producer warp; two CTAs share an SM, so one
// CTA's per-token reductions overlap the other's MMAs and copies.
constexpr int kCoefWarps = kMultiCoefWarps;
constexpr int kCoefThreads = (kCoefWarps + 1) * 32;

struct GenALayout {
    uint32_t ring, zero, full, empty, tfull, tempty, tok, red, zr, coef, misc, total;
    uint32_t buf_bytes, tstride;
};

__host__ __device__ inline GenALayout gen_a_layout(int bufs, int s8, uint32_t pitch, int M, int S, int kgroups,
                                                   int cs) {
    GenALayout L;
    L.buf_bytes = static_cast<uint32_t>(M + S) * pitch;
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(bufs) * L.buf_bytes;
    off = align_up(off, 16);
    L.zero = off;
    off += pitch;
    off = align_up(off, 16);
    L.full = off;
    off += 8u * bufs;
    L.empty = off;
    off += 8u * bufs;
    L.tfull = off;
    off += 8u * kGenTokSlots;
    L.tempty = off;
    off += 8u * kGenTokSlots;
    off = align_up(off, 16);
    L.tstride = align_up(static_cast<uint32_t>(2 * M * S + S), 4u);
    L.tok = off;
    off += kGenTokSlots * L.tstride * 4u;
    L.red = off;
    off += static_cast<uint32_t>(kgroups) * 16u * static_cast<uint32_t>(s8) * 4u;
    L.zr = off;
    off += static_cast<uint32_t>(kCoefWarps) * static_cast<uint32_t>(s8) * 4u;
    off = align_up(off, 16);
    L.coef = off;
    off += static_cast<uint32_t>(S) * static_cast<uint32_t>(cs) * 4u;
    L.misc = off;
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

__global__ void __launch_bounds__(kCoefThreads, 2) attnres_multi_coef_kernel(const __grid_constant__ MultiGenArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = a.S, M = a.M, s8 = a.s8;
    const int M4 = (M + 3) & ~3;
    const int MS = M * S;
    const int ntiles = s8 / 8;
    const int kg = a.kgroups;
    const GenALayout L = gen_a_layout(a.bufs, s8, a.pitch, M, S, kg, a.cs);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    float* tok = reinterpret_cast<float*>(smem + L.tok);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* zr = reinterpret_cast<float*>(smem + L.zr);
    float* coef = reinterpret_cast<float*>(smem + L.coef);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = a.bufs;
    const int nb = a.nblocks;
    const int dc = a.dc;
    const long long N = a.N;
    const int D = a.D;
    const uint32_t pitch = a.pitch;
    const int tstride = static_cast<int>(L.tstride);
    const int cs = a.cs;
    constexpr int nct = kCoefWarps * 32;

    if (threadIdx.x == 0) {
        for (int b = 0; b < B; ++b) {
            mbar_init(full + b, 1);
            mbar_init(empty + b, kCoefWarps);
        }
        for (int k = 0; k < kGenTokSlots; ++k) {
            mbar_init(tfull + k, 32);
            mbar_init(tempty + k, kCoefWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    // the zero row and the coefficient table's padding stay zero
    for (int i = threadIdx.x; i < static_cast<int>(pitch) / 16; i += blockDim.x)
        *reinterpret_cast<uint4*>(smem + L.zero + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < S * cs; i += blockDim.x) coef[i] = 0.0f;
    __syncthreads();

    if (warp == kCoefWarps) {
        // ------------------------------------------------------ producer
        // lane 0 claims a buffer and announces its bytes; all lanes issue the
        // row copies (one 1-D TMA copy per row, rows spread over the lanes)
        const uint64_t pol = policy_evict_first();
        int b = 0;
        uint32_t phase = 0;
        int ts = 0;
        uint32_t tphase = 0;
        long long issued = 0;
        for (long long n = blockIdx.x; n < N; n += gridDim.x) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            // saved statistics -> tok[ts] (all 32 lanes arrive on tfull)
            mbar_wait(tempty + ts, tphase ^ 1u, abort_flag, &g_multi_gen_error, kSiteBwdProducer);
            float* dst = tok + ts * tstride;
            for (int e = lane; e < MS; e += 32) {
                cp_async_4(dst + e, a.alpha + n * MS + e);
                cp_async_4(dst + MS + e, a.logit + n * MS + e);
            }
            for (int e = lane; e < S; e += 32) cp_async_4(dst + 2 * MS + e, a.rstd + n * S + e);
            cp_async_arrive_noinc(tfull + ts);
            if (++ts == kGenTokSlots) {
                ts = 0;
                tphase ^= 1u;
            }
            bool stop = false;
            for (int c = 0; c < nb && !stop; ++c) {
                const int c0 = c * dc;
                const int wc = min(dc, D - c0);
                const uint32_t bytes = static_cast<uint32_t>(wc) * 2u;
                const bool tail = (wc & 15) != 0;  // width 8 mod 16: zeros behind the block
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(empty + b, phase ^ 1u, abort_flag, &g_multi_gen_error, kSiteBwdProducer) ? 1 : 0;
                    if (ok) mbar_arrive_expect_tx(full + b, (bytes + (tail ? 16u : 0u)) * static_cast<uint32_t>(M + S));
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    stop = true;
                    break;
                }
                unsigned char* buf = smem + L.ring + b * L.buf_bytes;
                for (int r = lane; r < M + S; r += 32) {
                    const bool dyrow = r < M;
                    const int row = r;
                    const void* src = dyrow ? static_cast<const void*>(a.dy + r * a.dy_ms + n * a.dy_ns + c0)
                                            : static_cast<const void*>(static_cast<const unsigned char*>(a.src[r - M]) +
                                                                       (n * a.src_ld + c0) * 2);
                    tma_load_1d(buf + row * pitch, src, bytes, full + b, pol);
                    if (tail) tma_load_1d(buf + row * pitch + bytes, g_zero16, 16u, full + b, pol);
                }
                ++issued;
                if (++b == B) {
                    b = 0;
                    phase ^= 1u;
                }
            }
            if (stop) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0 && *abort_flag) {
            for (int c = 0; c < B && c < issued; ++c) {
                const long long fills = (issued - 1 - c) / B + 1;
                volatile int no_abort = 0;
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_gen_error, kSiteDrain);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // warp -> (source tile group, k group): with fewer 8-source tiles than
    // warps the k steps of a block are split between warps (partial tiles
    // added afterwards in k-group order); otherwise every warp owns whole
    // tiles (tiles w, w + 4, w + 8, w + 12).
    const bool split_k = ntiles < kCoefWarps;
    const int my_tile = split_k ? warp % ntiles : warp;
    const int my_kg = split_k ? warp / ntiles : 0;
    const bool active = !split_k || warp < ntiles * kg;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring_s = sbase + L.ring;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    const uint32_t tfull_s = sbase + L.tfull;
    const uint32_t tempty_s = sbase + L.tempty;
    // ldmatrix row addresses of this lane, relative to a buffer (A: dy row
    // `ra`; B: source row `rb` of a tile), or absolute at the zero row for
    // queries past M and sources past S
    const uint32_t zero_s = sbase + L.zero;
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t a_col = static_cast<uint32_t>((lane >> 4) * 8) * 2u;
    const uint32_t b_col = static_cast<uint32_t>(((lane >> 3) & 1) * 8) * 2u;
    auto a_addr = [&](uint32_t buf) { return ra < M ? buf + static_cast<uint32_t>(ra) * pitch + a_col : zero_s + a_col; };
    auto b_addr = [&](uint32_t buf, int tile) {
        const int rb = tile * 8 + (lane & 7);
        return rb < S ? buf + static_cast<uint32_t>(M + rb) * pitch + b_col : zero_s + b_col;
    };
    const int g = lane >> 2, t4 = lane & 3;
    const float inv_r = 1.0f / static_cast<float>(a.R);

    int b = 0;
    uint32_t phase = 0;
    int ts = 0;
    uint32_t tphase = 0;
    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        float acc[4][4];  // up to four 8-source tiles per warp (s8 <= 128)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
        for (int c = 0; c < nb; ++c) {
            const int wc = min(dc, D - c * dc);
            const int ksteps = (wc + 15) >> 4;
            mbar_wait_s(full_s + 8u * b, phase, abort_flag, &g_multi_gen_error, kSiteBwdConsumer);
            const uint32_t buf = ring_s + static_cast<uint32_t>(b) * L.buf_bytes;
            const uint32_t abuf = a_addr(buf), bbuf = b_addr(buf, my_tile);
            uint32_t dep = 0;
            if (active && split_k) {
                // one tile: the fragments of four k steps are loaded before
                // their MMAs, which alternate between two accumulators (added
                // in a fixed order after the token)
                for (int ks = my_kg; ks < ksteps; ks += 4 * kg) {
                    uint32_t af[4][4], bf[4][2];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int kk = ks + u * kg;
                        if (kk < ksteps) {
                            ldsm_x4(abuf + static_cast<uint32_t>(kk) * 32u, af[u][0], af[u][1], af[u][2], af[u][3]);
                            ldsm_x2(bbuf + static_cast<uint32_t>(kk) * 32u, bf[u][0], bf[u][1]);
                            dep ^= af[u][0] ^ bf[u][0];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (ks + u * kg < ksteps)
                            mma_bf16_16816(acc[u & 1], af[u][0], af[u][1], af[u][2], af[u][3], bf[u][0], bf[u][1]);
                }
            } else if (active) {
                // whole tiles (up to four): the fragments of two k steps are
                // loaded before their MMAs
                for (int ks = my_kg; ks < ksteps; ks += 2 * kg) {
                    uint32_t af[2][4], bf[2][4][2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int kk = ks + u * kg;
                        if (kk < ksteps) {
                            ldsm_x4(abuf + static_cast<uint32_t>(kk) * 32u, af[u][0], af[u][1], af[u][2], af[u][3]);
                            dep ^= af[u][0];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int tile = my_tile + j * kCoefWarps;
                                if (tile < ntiles) {
                                    ldsm_x2(b_addr(buf, tile) + static_cast<uint32_t>(kk) * 32u, bf[u][j][0], bf[u][j][1]);
                                    dep ^= bf[u][j][0];
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (ks + u * kg < ksteps) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (my_tile + j * kCoefWarps < ntiles)
                                    mma_bf16_16816(acc[j], af[u][0], af[u][1], af[u][2], af[u][3], bf[u][j][0],
                                                   bf[u][j][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_after(empty_s + 8u * b, dep);
            if (++b == a.bufs) {
                b = 0;
                phase ^= 1u;
            }
        }
        if (split_k) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[0][e] += acc[1][e];
        }
        // partial tiles -> red[k group][query][source]; then DA = their sum in k-group order
        if (active) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tile = my_tile + j * kCoefWarps;
                if ((j == 0 || !split_k) && tile < ntiles) {
                    float* r = red + (my_kg * 16) * s8;
                    const int s0 = tile * 8 + 2 * t4;
                    r[g * s8 + s0] = acc[j][0];
                    r[g * s8 + s0 + 1] = acc[j][1];
                    r[(g + 8) * s8 + s0] = acc[j][2];
                    r[(g + 8) * s8 + s0 + 1] = acc[j][3];
                }
            }
        }
        named_bar_sync(1, nct);
        mbar_wait_s(tfull_s + 8u * ts, tphase, abort_flag, &g_multi_gen_error, kSiteBwdTokStat);
        // coefficients: warp w forms those of queries w, w + 4, w + 8, w + 12
        // together (lanes over sources; da_ms = the k-group partials added in
        // k-group order), and its part of sum_m dz_ms z_ms per source
        const float* tk = tok + ts * tstride;
        constexpr int kQW = 16 / kCoefWarps;  // queries per warp (M <= 16)
        auto da_of = [&](int m, int s) {
            float d = 0.0f;
            for (int k = 0; k < kg; ++k) d += red[(k * 16 + m) * s8 + s];
            return d;
        };
        if (S <= 32) {
            // one source per lane: every load of the warp's queries is issued
            // before the sums that use it
            const int s = lane;
            const bool sv = s < S;
            float al[kQW], lg[kQW], dd[kQW], delta[kQW];
#pragma unroll
            for (int i = 0; i < kQW; ++i) {
                const int m = warp + i * kCoefWarps;
                const bool v = sv && m < M;
                al[i] = v ? tk[m * S + s] : 0.0f;
                lg[i] = v ? tk[MS + m * S + s] : 0.0f;
                float d = 0.0f;
#pragma unroll
                for (int k = 0; k < kCoefWarps; ++k)
                    if (k < kg) d += v ? red[(k * 16 + m) * s8 + s] : 0.0f;
                dd[i] = d;
                delta[i] = al[i] * d;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < kQW; ++i) delta[i] += __shfl_xor_sync(0xffffffffu, delta[i], o);
            if (sv) {
                const float r = tk[2 * MS + s];
                float z = 0.0f;
#pragma unroll
                for (int i = 0; i < kQW; ++i) {
                    const int m = warp + i * kCoefWarps;
                    if (m < M) {
                        const float dz = al[i] * (dd[i] - delta[i]);
                        coef[s * cs + m] = al[i];
                        coef[s * cs + M4 + m] = a.scale * r * dz;
                        z = fmaf(dz, lg[i], z);
                    }
                }
                zr[warp * s8 + s] = z;
            }
        } else {
            float delta[kQW];
#pragma unroll
            for (int i = 0; i < kQW; ++i) {
                const int m = warp + i * kCoefWarps;
                float p = 0.0f;
                if (m < M)
                    for (int s = lane; s < S; s += 32) p = fmaf(tk[m * S + s], da_of(m, s), p);
                delta[i] = p;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < kQW; ++i) delta[i] += __shfl_xor_sync(0xffffffffu, delta[i], o);
            for (int s = lane; s < S; s += 32) {
                const float r = tk[2 * MS + s];
                float z = 0.0f;
#pragma unroll
                for (int i = 0; i < kQW; ++i) {
                    const int m = warp + i * kCoefWarps;
                    if (m < M) {
                        const float al = tk[m * S + s];
                        const float dz = al * (da_of(m, s) - delta[i]);
                        coef[s * cs + m] = al;
                        coef[s * cs + M4 + m] = a.scale * r * dz;
                        z = fmaf(dz, tk[MS + m * S + s], z);
                    }
                }
                zr[warp * s8 + s] = z;
            }
        }
        named_bar_sync(1, nct);
        // the token's table -> workspace (16-byte stores; cs is a multiple of 4);
        // the vector holding c_s = -(r_s^2 / R) sum_m dz_ms z_ms (the warps'
        // parts added in warp order) gets it on the way
        {
            float4* out = reinterpret_cast<float4*>(a.coef + n * static_cast<long long>(S) * cs);
            const float4* in = reinterpret_cast<const float4*>(coef);
            const int cs4 = cs / 4;
            for (int i = threadIdx.x; i < S * cs4; i += nct) {
                float4 v = in[i];
                const int s = i / cs4;
                if (4 * (i - s * cs4) == 2 * M4) {
                    float z = 0.0f;
#pragma unroll
                    for (int w = 0; w < kCoefWarps; ++w) z += zr[w * s8 + s];
                    const float r = tk[2 * MS + s];
                    v.x = -(r * r) * inv_r * z;
                }
                out[i] = v;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_s(tempty_s + 8u * ts);
        if (++ts == kGenTokSlots) {
            ts = 0;
            tphase ^= 1u;
        }
        named_bar_sync(1, nct);  // the table and DA are rewritten by the next token
    }
}

// ---------------------------------------------------------------- kernel B
// Shared memory: `tslots` token slots x {coefficient table [S][cs], dy block
// [M][dcb], ids [M] (selected)}, source chunk ring [chunks][rows][dcb],
// barriers, the selected bank's block [(E + 1) rows] when it is kept in
// shared memory.
struct GenBLayout {
    uint32_t slot, slot_bytes, coef_off, dy_off, ids_off, ring, chunk_bytes, full, empty, tfull, tempty, bank, misc,
        total;
};

__host__ __device__ inline GenBLayout gen_b_layout(int S, int cs, int M, int dcb, int rows, int chunks, int bank_rows,
                                                   int tslots) {
    GenBLayout L;
    const uint32_t row = static_cast<uint32_t>(dcb) * 2u;
    L.coef_off = 0;
    L.dy_off = align_up(static_cast<uint32_t>(S * cs) * 4u, 16);
    L.ids_off = L.dy_off + static_cast<uint32_t>(M) * row;
    L.slot_bytes = align_up(L.ids_off + static_cast<uint32_t>(M) * 8u, 128);
    uint32_t off = 0;
    L.slot = off;
    off += static_cast<uint32_t>(tslots) * L.slot_bytes;
    L.ring = off;
    L.chunk_bytes = static_cast<uint32_t>(rows) * row;
    off += static_cast<uint32_t>(chunks) * L.chunk_bytes;
    off = align_up(off, 16);
    L.full = off;
    off += 8u * chunks;
    L.empty = off;
    off += 8u * chunks;
    L.tfull = off;
    off += 8u * tslots;
    L.tempty = off;
    off += 8u * tslots;
    off = align_up(off, 16);
    L.bank = off;
    off += static_cast<uint32_t>(bank_rows) * row;
    L.misc = off;
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

// MQ: register arrays for up to MQ queries (the run-time M <= MQ).  P: column
// pairs per thread (the CTA's block is 512 * P columns; pair p of thread t is
// columns 2 (t + 256 p) and the next).  SEL: per-token queries from the bank
// rows a.ids selects.
template <int MQ, int P, bool SEL>
__global__ void __launch_bounds__(kGenThreads, 1) attnres_multi_grad_kernel(const __grid_constant__ MultiGenArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = a.S, M = a.M, cs = a.cs;
    const int M4 = (M + 3) & ~3;  // queries padded to 4 in the coefficient table
    const int dcb = a.dcb;        // == kMultiGenColumns * P
    const int G = a.rows_b;
    const int K = a.chunks_b;
    const int TS = a.tslots_b;
    const int E = SEL ? a.E : 0;
    const bool bank_smem = SEL && a.bank_rows > 0;
    const GenBLayout L = gen_b_layout(S, cs, M, dcb, G, K, a.bank_rows, TS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint64_t* tfull = reinterpret_cast<uint64_t*>(smem + L.tfull);
    uint64_t* tempty = reinterpret_cast<uint64_t*>(smem + L.tempty);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int D = a.D;
    const int nbb = (D + dcb - 1) / dcb;
    const int cblk = static_cast<int>(blockIdx.x) % nbb;   // this CTA's column block
    const int grp = static_cast<int>(blockIdx.x) / nbb;    // its token group
    const int ngrp = static_cast<int>(gridDim.x) / nbb;
    const int c0 = cblk * dcb;
    const int wc = min(dcb, D - c0);
    const uint32_t row_bytes = static_cast<uint32_t>(wc) * 2u;
    const uint32_t rowp = static_cast<uint32_t>(dcb) * 2u;  // smem row pitch
    const int QR = SEL ? E : M;
    float* prow = a.part + static_cast<long long>(grp) * QR * a.R;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, kGenWarps);
        }
        for (int k = 0; k < TS; ++k) {
            // the TMA copies (one arrival with their bytes); with selected
            // queries also the producer's cp.async copies of the ids
            mbar_init(tfull + k, SEL ? 2 : 1);
            mbar_init(tempty + k, kGenWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    // the thread's column pairs and their key channels
    const int ko = a.ko, kend = a.ko + a.R;
    int j0[P];
    bool own[P], kx[P], ky[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int pi = static_cast<int>(threadIdx.x) + p * kGenWarps * 32;  // pair index within the block
        j0[p] = c0 + 2 * pi;
        own[p] = threadIdx.x < kGenWarps * 32 && 2 * pi < wc;
        kx[p] = own[p] && j0[p] >= ko && j0[p] < kend;
        ky[p] = own[p] && j0[p] + 1 >= ko && j0[p] + 1 < kend;
    }
    if (bank_smem) {
        // the bank's key values at this block's columns, row e at L.bank + e * rowp
        // (row E stays zero: it serves an id outside [0, E))
        uint16_t* bk = reinterpret_cast<uint16_t*>(smem + L.bank);
        for (int i = threadIdx.x; i < (E + 1) * dcb; i += blockDim.x) {
            const int e = i / dcb, j = c0 + (i - e * dcb);
            bk[i] = (e < E && j < D && j >= ko && j < kend) ? a.q[static_cast<long long>(e) * a.R + (j - ko)]
                                                            : static_cast<uint16_t>(0);
        }
    }
    if (SEL) {
        // this thread's key channels of the group's partial rows start at zero
        // (the same thread adds to them later, so program order suffices)
#pragma unroll
        for (int p = 0; p < P; ++p)
            for (int e = 0; e < E; ++e) {
                if (kx[p]) prow[static_cast<long long>(e) * a.R + (j0[p] - ko)] = 0.0f;
                if (ky[p]) prow[static_cast<long long>(e) * a.R + (j0[p] + 1 - ko)] = 0.0f;
            }
    }
    __syncthreads();

    if (warp == kGenWarps) {
        // ------------------------------------------------------ producer
        // lane 0 claims a slot or chunk and announces its bytes; all lanes
        // issue the row copies
        const uint64_t pol = policy_evict_first();
        int k = 0;
        uint32_t phase = 0;
        int ts = 0;
        uint32_t tphase = 0;
        long long issued = 0, tissued = 0;
        for (long long n = grp; n < N; n += ngrp) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int ok = 1;
            const uint32_t cbytes = static_cast<uint32_t>(S * cs) * 4u;
            if (lane == 0) {
                ok = mbar_wait(tempty + ts, tphase ^ 1u, abort_flag, &g_multi_gen_error, kSiteBwdProducer) ? 1 : 0;
                if (ok) mbar_arrive_expect_tx(tfull + ts, cbytes + static_cast<uint32_t>(M) * row_bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            unsigned char* slot = smem + L.slot + ts * L.slot_bytes;
            if (lane == 0)
                tma_load_1d(slot + L.coef_off, a.coef + n * static_cast<long long>(S) * cs, cbytes, tfull + ts, pol);
            for (int m = lane; m < M; m += 32)
                tma_load_1d(slot + L.dy_off + m * rowp, a.dy + m * a.dy_ms + n * a.dy_ns + c0, row_bytes, tfull + ts,
                            pol);
            if (SEL && lane == 0) {
                // ids are 8-byte aligned only: small asynchronous copies
                for (int m = 0; m < M; ++m) cp_async_8(slot + L.ids_off + 8 * m, a.ids + n * M + m);
                cp_async_arrive_noinc(tfull + ts);
            }
            ++tissued;
            if (++ts == TS) {
                ts = 0;
                tphase ^= 1u;
            }
            bool stop = false;
            for (int s0 = 0; s0 < S; s0 += G) {
                const int gs = min(G, S - s0);
                if (lane == 0) {
                    ok = mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_multi_gen_error, kSiteBwdProducer) ? 1 : 0;
                    if (ok) mbar_arrive_expect_tx(full + k, row_bytes * static_cast<uint32_t>(gs));
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    stop = true;
                    break;
                }
                for (int r = lane; r < gs; r += 32) {
                    const unsigned char* src = static_cast<const unsigned char*>(a.src[s0 + r]) + (n * a.src_ld + c0) * 2;
                    tma_load_1d(smem + L.ring + k * L.chunk_bytes + r * rowp, src, row_bytes, full + k, pol);
                }
                ++issued;
                if (++k == K) {
                    k = 0;
                    phase ^= 1u;
                }
            }
            if (stop) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0 && *abort_flag) {
            for (int c = 0; c < K && c < issued; ++c) {
                const long long fills = (issued - 1 - c) / K + 1;
                volatile int no_abort = 0;
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_gen_error, kSiteDrain);
            }
            for (int c = 0; c < TS && c < tissued; ++c) {
                const long long fills = (tissued - 1 - c) / TS + 1;
                volatile int no_abort = 0;
                mbar_wait(tfull + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_gen_error, kSiteDrain);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // Registers hold the queries in pairs: for query pair i and column c of
    // the thread (c = 2 p + h over its P column pairs), qp[i][c] = {q_2i,
    // q_2i+1} at that column; dyp holds the token's dy values and dqp the dq
    // sums the same way.  A coefficient row stores the four alphas (and the
    // four b) of a query group contiguously, so each 16-byte load gives two
    // aligned pairs that enter the packed FMAs as they are: a source row
    // costs, per group of four queries, two loads and six packed FMAs per
    // column, and the even and odd queries' partial sums are added at the end.
    constexpr int MP = MQ / 2;
    constexpr int C = 2 * P;
    float2 qp[MP][C], dqp[MP][C];
#pragma unroll
    for (int i = 0; i < MP; ++i)
#pragma unroll
        for (int p = 0; p < P; ++p) {
            float q[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};  // [query 2i + e][column]
            if (!SEL) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int m = 2 * i + e;
                    if (m < M) {
                        if (kx[p]) q[e][0] = bf16_bits_to_float(a.q[static_cast<long long>(m) * a.R + (j0[p] - ko)]);
                        if (ky[p]) q[e][1] = bf16_bits_to_float(a.q[static_cast<long long>(m) * a.R + (j0[p] + 1 - ko)]);
                    }
                }
            }
            qp[i][2 * p] = make_float2(q[0][0], q[1][0]);
            qp[i][2 * p + 1] = make_float2(q[0][1], q[1][1]);
            dqp[i][2 * p] = dqp[i][2 * p + 1] = make_float2(0.0f, 0.0f);
        }
    const uint32_t sbase = smem_u32(smem);
    constexpr int kPairWords = kGenWarps * 32;  // 4-byte words between a thread's pairs in a row
    const int rowp_w = static_cast<int>(rowp / 4u);
    const uint32_t full_s = sbase + L.full, empty_s = sbase + L.empty;
    const uint32_t tfull_s = sbase + L.tfull, tempty_s = sbase + L.tempty;
    float2 keep[P];
#pragma unroll
    for (int p = 0; p < P; ++p) keep[p] = make_float2(kx[p] ? 1.0f : 0.0f, ky[p] ? 1.0f : 0.0f);
    const float2 one = make_float2(1.0f, 1.0f);
    int k = 0;
    uint32_t phase = 0;
    int ts = 0;
    uint32_t tphase = 0;
    for (long long n = grp; n < N; n += ngrp) {
        mbar_wait_s(tfull_s + 8u * ts, tphase, abort_flag, &g_multi_gen_error, kSiteBwdConsumer);
        const unsigned char* slot = smem + L.slot + ts * L.slot_bytes;
        const float* ctab = reinterpret_cast<const float*>(slot + L.coef_off);
        const uint32_t* dyw = reinterpret_cast<const uint32_t*>(slot + L.dy_off) + threadIdx.x;
        float2 dyp[MP][C];
#pragma unroll
        for (int i = 0; i < MP; ++i)
#pragma unroll
            for (int p = 0; p < P; ++p) {
                uint32_t w0 = 0, w1 = 0;
                if (2 * i < M && own[p]) w0 = dyw[(2 * i) * rowp_w + p * kPairWords];
                if (2 * i + 1 < M && own[p]) w1 = dyw[(2 * i + 1) * rowp_w + p * kPairWords];
                dyp[i][2 * p] = make_float2(__uint_as_float(w0 << 16), __uint_as_float(w1 << 16));
                dyp[i][2 * p + 1] = make_float2(__uint_as_float(w0 & 0xffff0000u), __uint_as_float(w1 & 0xffff0000u));
            }
        const long long* ids = reinterpret_cast<const long long*>(slot + L.ids_off);
        if constexpr (SEL) {
#pragma unroll
            for (int i = 0; i < MP; ++i) {
                float q[2][P][2];  // [query 2i + e][pair][column]: the token's query values
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int m = 2 * i + e;
                    long long id = -1;
                    if (m < M) {
                        id = ids[m];
                        if (id < 0 || id >= E) {
                            if (threadIdx.x == 0) atomicCAS(&g_multi_gen_error, 0u, static_cast<unsigned>(kSiteBadId));
                            id = -1;
                        }
                    }
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        float x = 0.0f, y = 0.0f;
                        if (id >= 0) {
                            if (bank_smem) {
                                uint32_t w = 0;
                                if (own[p])
                                    w = reinterpret_cast<const uint32_t*>(smem + L.bank)[static_cast<int>(id) * rowp_w +
                                                                                         threadIdx.x + p * kPairWords];
                                const float2 f = bf2_to_f2(w);
                                x = f.x;
                                y = f.y;
                            } else {
                                if (kx[p]) x = bf16_bits_to_float(a.q[id * a.R + (j0[p] - ko)]);
                                if (ky[p]) y = bf16_bits_to_float(a.q[id * a.R + (j0[p] + 1 - ko)]);
                            }
                        }
                        q[e][p][0] = x;
                        q[e][p][1] = y;
                    }
                }
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    qp[i][2 * p] = make_float2(q[0][p][0], q[1][p][0]);
                    qp[i][2 * p + 1] = make_float2(q[0][p][1], q[1][p][1]);
                    dqp[i][2 * p] = dqp[i][2 * p + 1] = make_float2(0.0f, 0.0f);
                }
            }
        }
        for (int s0 = 0; s0 < S; s0 += G) {
            const int gs = min(G, S - s0);
            mbar_wait_s(full_s + 8u * k, phase, abort_flag, &g_multi_gen_error, kSiteBwdConsumer);
            const uint32_t* chunk =
                reinterpret_cast<const uint32_t*>(smem + L.ring + static_cast<uint32_t>(k) * L.chunk_bytes) + threadIdx.x;
            uint32_t dep = 0;
#pragma unroll 1
            for (int r = 0; r < gs; ++r) {
                const int s = s0 + r;
                float2 t[P], tb[C];
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const uint32_t w = own[p] ? chunk[r * rowp_w + p * kPairWords] : 0u;
                    dep ^= w;
                    t[p] = fmul2(bf2_to_f2(w), keep[p]);  // key channels of the row
                    tb[2 * p] = make_float2(t[p].x, t[p].x);
                    tb[2 * p + 1] = make_float2(t[p].y, t[p].y);
                }
                // alpha_s., b_s. and c_s of the row (the table's padding queries are zero)
                const float* crow = ctab + s * cs;
                // two accumulators per column for the alpha and the b terms (one
                // when a thread owns two column pairs, to stay within its registers)
                constexpr int h1 = C > 2 ? 0 : 1;
                float2 oa[2][C], ob[2][C];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int c = 0; c < C; ++c) oa[h][c] = ob[h][c] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int g4 = 0; g4 < MQ / 4; ++g4) {
                    if (4 * g4 < M) {
                        const float4 av = *reinterpret_cast<const float4*>(crow + 4 * g4);
                        const float4 bv = *reinterpret_cast<const float4*>(crow + M4 + 4 * g4);
                        const float2 a01 = make_float2(av.x, av.y), a23 = make_float2(av.z, av.w);
                        const float2 b01 = make_float2(bv.x, bv.y), b23 = make_float2(bv.z, bv.w);
#pragma unroll
                        for (int c = 0; c < C; ++c) {
                            oa[0][c] = ffma2(a01, dyp[2 * g4][c], oa[0][c]);
                            oa[h1][c] = ffma2(a23, dyp[2 * g4 + 1][c], oa[h1][c]);
                            ob[0][c] = ffma2(b01, qp[2 * g4][c], ob[0][c]);
                            ob[h1][c] = ffma2(b23, qp[2 * g4 + 1][c], ob[h1][c]);
                            dqp[2 * g4][c] = ffma2(b01, tb[c], dqp[2 * g4][c]);
                            dqp[2 * g4 + 1][c] = ffma2(b23, tb[c], dqp[2 * g4 + 1][c]);
                        }
                    }
                }
                const float cv = crow[2 * M4];
                const float2 cv2 = make_float2(cv, cv);
                uint16_t* drow = static_cast<uint16_t*>(a.dsrc[s]) + n * a.dsrc_ld;
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    // {even, odd} query sums at the pair's two columns, then their totals
                    float2 e0 = ffma2(one, oa[0][2 * p], ob[0][2 * p]);
                    float2 e1 = ffma2(one, oa[0][2 * p + 1], ob[0][2 * p + 1]);
                    if constexpr (h1 == 1) {
                        e0 = ffma2(one, e0, ffma2(one, oa[1][2 * p], ob[1][2 * p]));
                        e1 = ffma2(one, e1, ffma2(one, oa[1][2 * p + 1], ob[1][2 * p + 1]));
                    }
                    const float2 o = ffma2(cv2, t[p], ffma2(one, make_float2(e0.x, e1.x), make_float2(e0.y, e1.y)));
                    // no memory clobber: the next row's shared-memory loads may be issued before it
                    if (own[p] && ATTNRES_IN_BOUNDS(n < a.N && s < a.S && j0[p] + 2 <= a.D, &g_multi_gen_error))
                        asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(drow + j0[p]), "r"(pack_f2(o)));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_after(empty_s + 8u * k, dep);
            if (++k == K) {
                k = 0;
                phase ^= 1u;
            }
        }
        if constexpr (SEL) {
            // the token's dq into its bank rows of the group's partial row (the
            // ids are read again from the slot, which is still held)
#pragma unroll
            for (int m = 0; m < MQ; ++m) {
                const long long id = m < M ? ids[m] : -1;
                if (id >= 0 && id < E) {
                    float* pq = prow + id * a.R;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        const float2 d0 = dqp[m >> 1][2 * p], d1 = dqp[m >> 1][2 * p + 1];
                        if (kx[p]) red_add_f32(pq + (j0[p] - ko), (m & 1) ? d0.y : d0.x);
                        if (ky[p]) red_add_f32(pq + (j0[p] + 1 - ko), (m & 1) ? d1.y : d1.x);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_s(tempty_s + 8u * ts);
        if (++ts == TS) {
            ts = 0;
            tphase ^= 1u;
        }
    }
    if constexpr (!SEL) {
        // this thread's key channels of the group's partial row
#pragma unroll
        for (int m = 0; m < MQ; ++m) {
            if (m < M) {
                float* pq = prow + static_cast<long long>(m) * a.R;
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const float2 d0 = dqp[m >> 1][2 * p], d1 = dqp[m >> 1][2 * p + 1];
                    if (kx[p]) pq[j0[p] - ko] = (m & 1) ? d0.y : d0.x;
                    if (ky[p]) pq[j0[p] + 1 - ko] = (m & 1) ? d1.y : d1.x;
                }
            }
        }
    }
}

template <int MQ, int P, bool SEL>
cudaError_t launch_grad_t(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream) {
    auto kern = attnres_multi_grad_kernel<MQ, P, SEL>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.gen_smem_b));
    if (err != cudaSuccess) return err;
    kern<<<plan.gen_grid_b, kGenThreads, plan.gen_smem_b, stream>>>(a);
    return cudaGetLastError();
}

template <bool SEL>
cudaError_t launch_grad_sel(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream) {
    const int P = a.dcb / kMultiGenColumns;
    if (a.M <= 4) return P == 2 ? launch_grad_t<4, 2, SEL>(plan, a, stream) : launch_grad_t<4, 1, SEL>(plan, a, stream);
    if (a.M <= 8) return P == 2 ? launch_grad_t<8, 2, SEL>(plan, a, stream) : launch_grad_t<8, 1, SEL>(plan, a, stream);
    return launch_grad_t<16, 1, SEL>(plan, a, stream);
}

}  // namespace

size_t multi_gen_smem_a(int bufs, int s8, int pitch, int M, int S, int kgroups, int cs) {
    return gen_a_layout(bufs, s8, static_cast<uint32_t>(pitch), M, S, kgroups, cs).total;
}

size_t multi_gen_smem_b(int S, int cs, int M, int dcb, int rows, int chunks, int bank_rows, int tslots) {
    return gen_b_layout(S, cs, M, dcb, rows, chunks, bank_rows, tslots).total;
}

cudaError_t launch_multi_bwd_general(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream) {
    cudaError_t err = cudaFuncSetAttribute(attnres_multi_coef_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.gen_smem_a));
    if (err != cudaSuccess) return err;
    attnres_multi_coef_kernel<<<plan.gen_grid_a, kCoefThreads, plan.gen_smem_a, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const bool sel = a.ids != nullptr;
    err = sel ? launch_grad_sel<true>(plan, a, stream)
              : (plan.gen_grad_mma ? launch_multi_grad_mma(plan, a, stream) : launch_grad_sel<false>(plan, a, stream));
    if (err != cudaSuccess) return err;
    const int W = (sel ? a.E : a.M) * a.R;
    return launch_finalize(a.part, plan.gen_groups, W, W, a.dq, a.dq_f32, nullptr, nullptr, stream);
}

unsigned take_multi_gen_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_gen_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_gen_error, &zero, sizeof zero);
    return v;
}

}  // namespace attnres
