// attnres_multi_grad_mma.cu -- the gradient kernel of the general multi-query
// backward on the tensor cores: fixed queries, at most 16 sources.
//
// Per token, with the coefficient kernel's table (alpha_ms, b_ms and c_s;
// attnres_multi_general.cu gives the chain rule, "Fast Attention
// Residuals", sections "Multi-query AttnRes" and "Equation"):
//   dV [S x D]  = A^T [S x M] . DY [M x D] + B^T [S x M] . Q [M x D]
//                 + C [S x S] . T [S x D]       (C = diag(c_s), key channels)
//   dQ [M x R] += B [M x S] . T [S x R]                 (summed over tokens)
// with Q zero off the key channels and T the sources' rows.  With S and M
// padded to 16 these are chains of mma.m16n8k16: sources (dV) or queries
// (dQ) are the A rows, queries or sources the K dimension, 8-channel column
// tiles the N dimension.  The FP32 coefficients enter as three bf16 terms
// (hi + mid + lo, the rest below 2^-26 relative; smallest term first); dy, q
// and t are bf16 and exact, the products exact in FP32 and the sums FP32.
// A column tile that holds a key boundary adds c_s t_s per element instead.
//
// GB300 mapping: one CTA per 512-column block of a token group, as the SIMT
// gradient kernel.  A producer warp streams each token's coefficient table,
// its M dy rows and its S source rows (the block's columns, rows padded to
// 1040 bytes so that ldmatrix reads of 8 consecutive rows fall in different
// banks) into a ring of token slots with 1-D bulk copies; dy rows past M and
// source rows past S read one zero row.  Per token the consumer threads
// split the table into bf16 fragment tables in the slot (one element each),
// and each of the sixteen consumer warps -- four per scheduler, to cover the
// MMA and shared-memory latencies -- takes its A fragments from them with
// ldmatrix and runs its four column tiles (32 columns) with their
// independent chains interleaved: the dV product (B from the slot's dy rows
// by ldmatrix.trans and from the queries, held in registers for the launch),
// C . T and the dQ product (B = the slot's source rows).  dV rows leave as
// bf16 pairs straight from the accumulators; the dQ accumulators stay in
// registers for all of the CTA's tokens and are written once, as the
// group's partial row (the finalize kernel adds the groups in order).
#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {
namespace {

// First failed wait of any launch of this unit (0 = none).
__device__ unsigned int g_multi_grad_mma_error = 0;

constexpr int kGmWarps = 16;                       // MMA warps
constexpr int kGmBuildWarps = 2;                   // warps that split each token's coefficients
constexpr int kGmThreads = (kGmWarps + kGmBuildWarps + 1) * 32;  // plus the producer warp
constexpr int kGmCols = kGmWarps * 32;             // columns per CTA
constexpr int kGmPitch = kGmCols * 2 + 16;         // bytes per row in a slot
constexpr int kGmFragPitch = 48;                   // bytes per row of a fragment table (16 bf16 + 16)
constexpr int kGmFragBytes = 16 * kGmFragPitch;    // one 16 x 16 bf16 table
constexpr int kGmTables = 9;                       // {A, B, C} x {hi, mid, lo}
static_assert(kGmCols == kMultiGenColumns, "the MMA gradient kernel keeps the SIMT kernel's column blocks");

// Shared memory: `slots` token slots {coefficient table [S][cs] FP32, rows
// [M + S][kGmPitch] bytes: dy rows then source rows (both filled by the
// copies), fragment tables [kGmTables][16][kGmFragPitch] (written by the
// consumers)}, the zero row, barriers.
struct GmLayout {
    uint32_t ring, slot_bytes, rows_off, frag_off, zero, full, ready, empty, misc, total;
};

__host__ __device__ inline GmLayout gm_layout(int S, int cs, int M, int slots) {
    GmLayout L;
    L.rows_off = align_up(static_cast<uint32_t>(S * cs) * 4u, 16);
    L.frag_off = L.rows_off + static_cast<uint32_t>(M + S) * kGmPitch;
    L.slot_bytes = align_up(L.frag_off + kGmTables * kGmFragBytes, 128);
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(slots) * L.slot_bytes;
    L.zero = off;
    off += kGmPitch;
    off = align_up(off, 8);
    L.full = off;
    off += 8u * static_cast<uint32_t>(slots);
    L.ready = off;  // the slot's fragment tables are written
    off += 8u * static_cast<uint32_t>(slots);
    L.empty = off;
    off += 8u * static_cast<uint32_t>(slots);
    L.misc = off;  // abort flag
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

// An FP32 value as three bf16 terms x = hi + mid + lo (each difference is
// exact in FP32), as bf16 bits.
__device__ __forceinline__ void split3(float x, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
    const uint32_t h = pack_bf16x2(x, 0.0f) & 0xffffu;
    const float r = x - __uint_as_float(h << 16);
    const uint32_t md = pack_bf16x2(r, 0.0f) & 0xffffu;
    hi = static_cast<uint16_t>(h);
    mid = static_cast<uint16_t>(md);
    lo = static_cast<uint16_t>(pack_bf16x2(r - __uint_as_float(md << 16), 0.0f) & 0xffffu);
}

// M8: at most eight queries, so alpha and b share one 16-wide K step of the
// dV product (A = [alpha | b], B = [dy rows 0..7 ; query rows 0..7]).
template <bool M8>
__global__ void __launch_bounds__(kGmThreads, 1) attnres_multi_grad_mma_kernel(const __grid_constant__ MultiGenArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = a.S, M = a.M, cs = a.cs, D = a.D, R = a.R, ko = a.ko;
    const int M4 = (M + 3) & ~3;
    const int K = a.tslots_b;
    const GmLayout L = gm_layout(S, cs, M, K);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    const int nbb = (D + kGmCols - 1) / kGmCols;
    const int cblk = static_cast<int>(blockIdx.x) % nbb;  // this CTA's column block
    const int grp = static_cast<int>(blockIdx.x) / nbb;   // its token group
    const int ngrp = static_cast<int>(gridDim.x) / nbb;
    const int c0 = cblk * kGmCols;
    const int wc = min(kGmCols, D - c0);
    const uint32_t row_bytes = static_cast<uint32_t>(wc) * 2u;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(reinterpret_cast<uint64_t*>(smem + L.ready) + k, kGmBuildWarps);
            mbar_init(empty + k, kGmWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    for (int i = threadIdx.x; i < kGmPitch / 16; i += blockDim.x)
        *reinterpret_cast<uint4*>(smem + L.zero + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    // every slot's fragment tables start at zero: per token only the entries
    // of the S sources and the queries (or the diagonal) are rewritten
    for (int k = 0; k < K; ++k)
        for (int i = threadIdx.x; i < kGmTables * kGmFragBytes / 16; i += blockDim.x)
            *reinterpret_cast<uint4*>(smem + L.ring + k * L.slot_bytes + L.frag_off + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    if (warp == kGmWarps + kGmBuildWarps) {
        // ------------------------------------------------------ producer
        // lane 0 claims a slot and announces its bytes; the lanes issue the
        // row copies
        const uint64_t pol = policy_evict_first();
        const uint32_t cbytes = static_cast<uint32_t>(S * cs) * 4u;
        int k = 0;
        uint32_t phase = 0;
        long long issued = 0;
        for (long long n = grp; n < N; n += ngrp) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_multi_grad_mma_error, kSiteBwdProducer) ? 1 : 0;
                if (ok) mbar_arrive_expect_tx(full + k, cbytes + static_cast<uint32_t>(M + S) * row_bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            unsigned char* slot = smem + L.ring + k * L.slot_bytes;
            if (lane == 0) tma_load_1d(slot, a.coef + n * static_cast<long long>(S) * cs, cbytes, full + k, pol);
            for (int r = lane; r < M + S; r += 32) {
                const void* src = r < M ? static_cast<const void*>(a.dy + r * a.dy_ms + n * a.dy_ns + c0)
                                        : static_cast<const void*>(static_cast<const unsigned char*>(a.src[r - M]) +
                                                                   (n * a.src_ld + c0) * 2);
                tma_load_1d(slot + L.rows_off + r * kGmPitch, src, row_bytes, full + k, pol);
            }
            ++issued;
            if (++k == K) {
                k = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0 && *abort_flag) {
            // every copy this warp started lands before the CTA may exit
            for (int c = 0; c < K && c < issued; ++c) {
                const long long fills = (issued - 1 - c) / K + 1;
                volatile int no_abort = 0;
                mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_grad_mma_error,
                          kSiteDrain);
            }
        }
        return;
    }

    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_s = sbase + L.full, ready_s = sbase + L.ready, empty_s = sbase + L.empty;
    constexpr int tw = kGmFragBytes / 2;  // elements per fragment table

    if (warp >= kGmWarps) {
        // ------------------------------------------------------ builders
        // per token, once its copies have landed: the fragment tables in the
        // slot, [s][column] elements split over the builder threads (the
        // other entries stay zero): table A (terms at 0..2) the A of the dV
        // product, alpha_sk (M8: alpha_sk for k < 8, b_s,k-8 above); table B
        // (3..5) b_sm, the second K step of dV (not M8) and, read transposed,
        // the A of the dQ product; table C (6..8) diag(c_s).  The MMA warps
        // wait for them on the slot's `ready` barrier, so the builders run
        // ahead of them by up to the ring's depth.
        const int bt_id = static_cast<int>(threadIdx.x) - kGmWarps * 32;
        constexpr int nbt = kGmBuildWarps * 32;
        const int wa = M8 ? 8 + M4 : M4;  // live columns of table A
        const int na = S * wa, nb = S * M4;
        int k = 0;
        uint32_t phase = 0;
        for (long long n = grp; n < N; n += ngrp) {
            if (!mbar_wait_s(full_s + 8u * k, phase, abort_flag, &g_multi_grad_mma_error, kSiteBwdConsumer)) break;
            unsigned char* slot = smem + L.ring + k * L.slot_bytes;
            const float* ctab = reinterpret_cast<const float*>(slot);
            uint16_t* ft = reinterpret_cast<uint16_t*>(slot + L.frag_off);
            for (int i = bt_id; i < na + nb + S; i += nbt) {
                int tb, sr, c;
                float v;
                if (i < na) {
                    tb = 0;
                    sr = i / wa;
                    c = i - sr * wa;
                    if (M8)
                        v = c < 8 ? (c < M4 ? ctab[sr * cs + c] : 0.0f) : ctab[sr * cs + M4 + c - 8];
                    else
                        v = ctab[sr * cs + c];
                } else if (i < na + nb) {
                    tb = 1;
                    sr = (i - na) / M4;
                    c = (i - na) - sr * M4;
                    v = ctab[sr * cs + M4 + c];
                } else {
                    tb = 2;
                    sr = c = i - na - nb;
                    v = ctab[sr * cs + 2 * M4];
                }
                const int e = 3 * tb * tw + sr * (kGmFragPitch / 2) + c;
                split3(v, ft[e], ft[tw + e], ft[2 * tw + e]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_s(ready_s + 8u * k);
            if (++k == K) {
                k = 0;
                phase ^= 1u;
            }
        }
        return;
    }

    // ---------------------------------------------------------- MMA warps
    const uint32_t zero_s = sbase + L.zero;
    const int g = lane >> 2, t4 = lane & 3;
    const int wcol = warp * 32;   // the warp's first column within the block
    const bool wact = wcol < wc;  // a warp past the block's width only takes part in the waits
    auto is_key = [&](int col) { return col >= ko && col < ko + R; };

    // B fragments of the queries at the warp's column tiles:
    // {q[2 t4][col], q[2 t4 + 1][col]} and {q[2 t4 + 8][col], q[2 t4 + 9][col]}
    // at col = c0 + wcol + 8 j + g (zero off the key channels and past M);
    // per tile: wholly on the key (C . T by MMA), holding a key boundary
    // (c_s t_s per element), or off the key
    uint32_t bq[4][2];
    bool kall[4], kmix[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int col = c0 + wcol + 8 * j + g;
        const bool key = wact && col < D && is_key(col);
        auto qbits = [&](int m) -> uint32_t {
            return (key && m < M) ? static_cast<uint32_t>(a.q[static_cast<long long>(m) * R + (col - ko)]) : 0u;
        };
        bq[j][0] = qbits(2 * t4) | (qbits(2 * t4 + 1) << 16);
        bq[j][1] = qbits(2 * t4 + 8) | (qbits(2 * t4 + 9) << 16);
        const int t0 = c0 + wcol + 8 * j;
        kall[j] = t0 >= ko && t0 + 8 <= ko + R;
        kmix[j] = !kall[j] && t0 < ko + R && t0 + 8 > ko;
    }
    float dqa[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) dqa[j][e] = 0.0f;

    const int lr = lane & 15;  // the row this lane addresses for an ldmatrix.trans pair
    // ldmatrix addresses within a fragment table: A rows (non-transposed) and
    // the transposed read that gives A[m][s] from a table stored [s][m]
    const uint32_t fa_off = static_cast<uint32_t>((lane & 7) + ((lane >> 3) & 1) * 8) * kGmFragPitch +
                            static_cast<uint32_t>(lane >> 4) * 16u;
    const uint32_t ft_off = static_cast<uint32_t>((lane & 7) + ((lane >> 4) & 1) * 8) * kGmFragPitch +
                            static_cast<uint32_t>((lane >> 3) & 1) * 16u;
    int k = 0;
    uint32_t phase = 0;
    for (long long n = grp; n < N; n += ngrp) {
        // the tables are written (after the slot's copies landed)
        mbar_wait_s(ready_s + 8u * k, phase, abort_flag, &g_multi_grad_mma_error, kSiteBwdConsumer);
        mbar_wait_s(full_s + 8u * k, phase, abort_flag, &g_multi_grad_mma_error, kSiteBwdConsumer);
        unsigned char* slot = smem + L.ring + k * L.slot_bytes;
        const uint32_t rows_s = sbase + L.ring + static_cast<uint32_t>(k) * L.slot_bytes + L.rows_off;
        const uint32_t frag_s = sbase + L.ring + static_cast<uint32_t>(k) * L.slot_bytes + L.frag_off;
        const float* ctab = reinterpret_cast<const float*>(slot);
        if (wact) {
            const uint32_t dyrow = lr < M ? rows_s + static_cast<uint32_t>(lr) * kGmPitch : zero_s;
            const uint32_t trow = lr < S ? rows_s + static_cast<uint32_t>(M + lr) * kGmPitch : zero_s;
            // the B fragments of the warp's four tiles
            uint32_t bd[4][2], bt[4][2];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t coff = static_cast<uint32_t>(wcol + 8 * jj) * 2u;
                ldsm_x2_trans(dyrow + coff, bd[jj][0], bd[jj][1]);
                ldsm_x2_trans(trow + coff, bt[jj][0], bt[jj][1]);
            }
            float acc[4][4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[jj][e] = 0.0f;
            // dV: the four tiles' chains interleaved, smallest term first
            {
                uint32_t fa[3][4];
#pragma unroll
                for (int t = 0; t < 3; ++t) ldsm_x4(frag_s + t * kGmFragBytes + fa_off, fa[t][0], fa[t][1], fa[t][2], fa[t][3]);
#pragma unroll
                for (int t = 2; t >= 0; --t)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        mma_bf16_16816(acc[jj], fa[t][0], fa[t][1], fa[t][2], fa[t][3], bd[jj][0],
                                       M8 ? bq[jj][0] : bd[jj][1]);
            }
            if constexpr (!M8) {
                uint32_t fb[3][4];
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    ldsm_x4(frag_s + (3 + t) * kGmFragBytes + fa_off, fb[t][0], fb[t][1], fb[t][2], fb[t][3]);
#pragma unroll
                for (int t = 2; t >= 0; --t)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (kall[jj] || kmix[jj])
                            mma_bf16_16816(acc[jj], fb[t][0], fb[t][1], fb[t][2], fb[t][3], bq[jj][0], bq[jj][1]);
            }
            {
                // C . T on the tiles wholly on the key
                uint32_t fc[3][4];
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    ldsm_x4(frag_s + (6 + t) * kGmFragBytes + fa_off, fc[t][0], fc[t][1], fc[t][2], fc[t][3]);
#pragma unroll
                for (int t = 2; t >= 0; --t)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (kall[jj]) mma_bf16_16816(acc[jj], fc[t][0], fc[t][1], fc[t][2], fc[t][3], bt[jj][0], bt[jj][1]);
            }
            {
                // dQ (tiles with key channels): A = b_sm read transposed, B = the source rows
                uint32_t fq[3][4];
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    ldsm_x4_trans(frag_s + (3 + t) * kGmFragBytes + ft_off, fq[t][0], fq[t][1], fq[t][2], fq[t][3]);
#pragma unroll
                for (int t = 2; t >= 0; --t)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (kall[jj] || kmix[jj])
                            mma_bf16_16816(dqa[jj], fq[t][0], fq[t][1], fq[t][2], fq[t][3], bt[jj][0], bt[jj][1]);
            }
            // dV rows g and g + 8 of each tile as bf16 pairs; a tile holding a key
            // boundary adds c_s t_s per element first
            uint16_t* const d_g = g < S ? static_cast<uint16_t*>(a.dsrc[g]) + n * a.dsrc_ld + c0 : nullptr;
            uint16_t* const d_g8 = g + 8 < S ? static_cast<uint16_t*>(a.dsrc[g + 8]) + n * a.dsrc_ld + c0 : nullptr;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int cl = wcol + 8 * jj + 2 * t4;  // the pair's first column within the block
                if (cl >= wc) continue;
                float2 o0 = make_float2(acc[jj][0], acc[jj][1]), o1 = make_float2(acc[jj][2], acc[jj][3]);
                if (kmix[jj]) {
                    const float kx = is_key(c0 + cl) ? 1.0f : 0.0f, ky = is_key(c0 + cl + 1) ? 1.0f : 0.0f;
                    const uint32_t t_g = rows_s + static_cast<uint32_t>(M + g) * kGmPitch + static_cast<uint32_t>(cl) * 2u;
                    if (g < S) {
                        const float cg = ctab[g * cs + 2 * M4];
                        uint32_t w;
                        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(t_g));
                        const float2 t = bf2_to_f2(w);
                        o0 = make_float2(fmaf(cg * kx, t.x, o0.x), fmaf(cg * ky, t.y, o0.y));
                    }
                    if (g + 8 < S) {
                        const float cg8 = ctab[(g + 8) * cs + 2 * M4];
                        uint32_t w;
                        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(t_g + 8u * kGmPitch));
                        const float2 t = bf2_to_f2(w);
                        o1 = make_float2(fmaf(cg8 * kx, t.x, o1.x), fmaf(cg8 * ky, t.y, o1.y));
                    }
                }
                if (d_g && ATTNRES_IN_BOUNDS(n < a.N && c0 + cl + 2 <= D, &g_multi_grad_mma_error))
                    asm volatile("st.global.b32 [%0], %1;" ::"l"(d_g + cl), "r"(pack_f2(o0)) : "memory");
                if (d_g8 && ATTNRES_IN_BOUNDS(n < a.N && c0 + cl + 2 <= D, &g_multi_grad_mma_error))
                    asm volatile("st.global.b32 [%0], %1;" ::"l"(d_g8 + cl), "r"(pack_f2(o1)) : "memory");
            }
        }
        // this warp is done with the slot
        __syncwarp();
        if (lane == 0) mbar_arrive_s(empty_s + 8u * k);
        if (++k == K) {
            k = 0;
            phase ^= 1u;
        }
    }
    // the group's partial row: dq at the warp's key columns, rows m = g, g + 8
    if (wact) {
        float* prow = a.part + static_cast<long long>(grp) * M * R;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = c0 + wcol + 8 * j + 2 * t4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = g + 8 * (e >> 1), cc = col + (e & 1);
                if (m < M && cc < D && is_key(cc)) prow[static_cast<long long>(m) * R + (cc - ko)] = dqa[j][e];
            }
        }
    }
}

}  // namespace

size_t multi_grad_mma_smem(int S, int cs, int M, int slots) { return gm_layout(S, cs, M, slots).total; }

cudaError_t launch_multi_grad_mma(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream) {
    auto kern = a.M <= 8 ? attnres_multi_grad_mma_kernel<true> : attnres_multi_grad_mma_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.gen_smem_b));
    if (err != cudaSuccess) return err;
    kern<<<plan.gen_grid_b, kGmThreads, plan.gen_smem_b, stream>>>(a);
    return cudaGetLastError();
}

unsigned take_multi_grad_mma_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_grad_mma_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_grad_mma_error, &zero, sizeof zero);
    return v;
}

}  // namespace attnres
