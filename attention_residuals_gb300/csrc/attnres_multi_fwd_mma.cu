// attnres_multi_fwd_mma.cu -- multi-query forward on the tensor cores, for
// reads with several queries whose token stays in shared memory.
//
// "Fast Attention Residuals", section "Multi-query AttnRes": M queries (up
// to 16) read the same S sources of a token; per query m (section
// "Equation"): r_s = 1/sqrt(mean(t_s^2) + eps), z_ms = scale * r_s *
// <t_s, q_m>, alpha_m = softmax_s(z_m), y_m = sum_s alpha_ms v_s.  Per token
// both products are dense contractions with M as one dimension:
//   Z = Q [M x R] . T^T [R x S]        (logits before scaling)
//   Y = A [M x S] . V [S x D]          (outputs)
// With M padded to 16 each maps onto mma.m16n8k16: queries are the A rows,
// sources the B columns (logits) or the K dimension (outputs).  The products
// of bf16 operands are exact in FP32 and the sums are FP32.  The FP32 weights
// alpha enter the output MMA as three bf16 terms, alpha = hi + mid + lo (the
// rest below 2^-26 relative), so the outputs carry the FP32 weights, not
// bf16 ones (two terms leave 2^-17, which shows on outputs that cancel to
// near zero).
//
// GB300 mapping: persistent CTAs; one producer thread streams each token's
// S rows into a ring of token slots with 1-D TMA bulk copies, row pitch D*2+16
// bytes so the ldmatrix row addresses of 8 rows fall in different banks; rows
// past S (and queries past M) read a shared zero row.  Eight consumer warps
// per token: key statistics (one warp per source), the logit MMA split over
// the key's 16-channel steps (each warp a share of them, partial 16 x 32
// tiles added in warp order), the softmax (one warp per two queries, one lane
// per source), then the output MMA split over 8-channel column tiles.
#include <cfloat>
#include <cstdlib>
#include <cstring>

#include "device_utils.cuh"
#include "kernels.cuh"

namespace attnres {
namespace {

// First failed wait of any launch of this unit (0 = none).
__device__ unsigned int g_multi_mma_error = 0;

constexpr int kMmaWarps = 8;                       // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;  // plus the producer warp
constexpr int kMmaMaxS = 32;                       // sources per token (two 16-source K tiles)
constexpr int kMmaAPitch = (kMmaMaxS + 8) * 2;     // bytes per row of the bf16 weight tables
constexpr int kPartPitch = kMmaMaxS + 4;           // floats per row of a partial logit tile
constexpr int kStagePitch = 80;                    // bytes per row of a warp's output staging tile (64 + 16)
constexpr int kMmaMaxSlots = 8;                    // token slots in the ring
// Fewer queries: the other kernel, whose cost grows with the query count while
// this one's is nearly flat (measured, S=10 N=32768: D=1024 M=16 0.58 against
// 1.32 ms, D=4096 M=16 1.96 against 4.43 ms, but D=2048 M=8 0.99 against
// 0.83 ms and D=4096 M=4 1.68 against 0.91 ms).
constexpr int kMmaMinQueries = 9;

// Shared memory of one CTA.
struct MmaLayout {
    uint32_t ring, qtab, zero, part, atab, rtab, full, empty, misc, total;
};
// A warp's output staging tile (16 rows x kStagePitch bytes) lies in its own
// partial-logit tile: the warp writes it only after the softmax has read all
// the partial tiles and before it forms its next token's partials.
static_assert(16 * kStagePitch <= 16 * kPartPitch * 4, "staging tile larger than the partial tile");

__host__ __device__ inline MmaLayout mma_layout(int slots, int S, int pitch, int qrows, int qpitch) {
    MmaLayout L;
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(slots) * static_cast<uint32_t>(S) * static_cast<uint32_t>(pitch);
    L.qtab = off;  // query rows (key channels only), qpitch bytes each
    off += static_cast<uint32_t>(qrows) * static_cast<uint32_t>(qpitch);
    L.zero = off;  // one zero row, as wide as the widest row read
    off += static_cast<uint32_t>(pitch > qpitch ? pitch : qpitch);
    off = align_up(off, 16);
    L.part = off;  // [kMmaWarps][16][kPartPitch] partial logits
    off += static_cast<uint32_t>(kMmaWarps) * 16u * kPartPitch * 4u;
    L.atab = off;  // [3][16][kMmaAPitch / 2] bf16 weights: hi, mid, lo
    off += 3u * 16u * static_cast<uint32_t>(kMmaAPitch);
    L.rtab = off;  // [kMmaMaxS] key rstd of the token
    off += kMmaMaxS * 4u;
    off = align_up(off, 8);
    L.full = off;
    off += 8u * static_cast<uint32_t>(slots);
    L.empty = off;
    off += 8u * static_cast<uint32_t>(slots);
    L.misc = off;  // abort flag
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}


// Launch arguments: the multi-query forward's, plus the ring of token slots.
struct MmaFwdArgs {
    MultiFwdArgs f;
    int slots;   // token slots in the ring
    int pitch;   // bytes per source row in a slot (D * 2 + 16)
    int qpitch;  // bytes per query row (R * 2 + 16)
    int qrows;   // query rows in shared memory: M, or the bank's E rows
};

template <bool SEL>
__global__ void __launch_bounds__(kMmaThreads, 2) attnres_multi_fwd_mma_kernel(const __grid_constant__ MmaFwdArgs g) {
    const MultiFwdArgs& a = g.f;
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = a.S, D = a.D, R = a.R, M = a.M;
    const int K = g.slots;
    const uint32_t pitch = static_cast<uint32_t>(g.pitch), qpitch = static_cast<uint32_t>(g.qpitch);
    const uint32_t slot_bytes = static_cast<uint32_t>(S) * pitch;
    const MmaLayout L = mma_layout(K, S, g.pitch, g.qrows, g.qpitch);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long N = a.N;
    constexpr int nct = kMmaWarps * 32;

    if (threadIdx.x == 0) {
        for (int k = 0; k < K; ++k) {
            mbar_init(full + k, 1);
            mbar_init(empty + k, kMmaWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    // the zero row and the weight tables (rows past M stay zero)
    {
        const uint32_t zbytes = L.part - L.zero;
        for (uint32_t i = threadIdx.x * 16u; i < zbytes; i += blockDim.x * 16u)
            *reinterpret_cast<uint4*>(smem + L.zero + i) = make_uint4(0u, 0u, 0u, 0u);
        for (uint32_t i = threadIdx.x * 16u; i < 3u * 16u * kMmaAPitch; i += blockDim.x * 16u)
            *reinterpret_cast<uint4*>(smem + L.atab + i) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kMmaWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = static_cast<uint32_t>(D) * 2u;
            int k = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (long long n = blockIdx.x; n < N && !*abort_flag; n += gridDim.x) {
                if (!mbar_wait(empty + k, phase ^ 1u, abort_flag, &g_multi_mma_error, kSiteFwdProducer)) break;
                mbar_arrive_expect_tx(full + k, bytes * static_cast<uint32_t>(S));
                for (int s = 0; s < S; ++s) {
                    const unsigned char* src = static_cast<const unsigned char*>(a.src[s]) + (n * a.src_ld) * 2;
                    tma_load_1d(smem + L.ring + k * slot_bytes + s * pitch, src, bytes, full + k, pol);
                }
                ++issued;
                if (++k == K) {
                    k = 0;
                    phase ^= 1u;
                }
            }
            if (*abort_flag) {
                // every copy this thread started lands before the CTA may exit
                for (int c = 0; c < K && c < issued; ++c) {
                    const long long fills = (issued - 1 - c) / K + 1;
                    volatile int no_abort = 0;
                    mbar_wait(full + c, static_cast<uint32_t>((fills - 1) & 1), &no_abort, &g_multi_mma_error,
                              kSiteDrain);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring_s = sbase + L.ring;
    const uint32_t qtab_s = sbase + L.qtab;
    const uint32_t zero_s = sbase + L.zero;
    const uint32_t atab_s = sbase + L.atab;
    const uint32_t full_s = sbase + L.full;
    const uint32_t empty_s = sbase + L.empty;
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* rtab = reinterpret_cast<float*>(smem + L.rtab);
    uint16_t* atab = reinterpret_cast<uint16_t*>(smem + L.atab);
    const int ko = a.ko;
    const float inv_r = 1.0f / static_cast<float>(R);
    const int ksteps = R >> 4;           // 16-channel steps of the key
    const int ntile = (S + 7) >> 3;      // 8-source column tiles of the logits
    const int nkt = (S + 15) >> 4;       // 16-source K tiles of the outputs
    const int g8 = lane >> 2, t4 = lane & 3;
    // ldmatrix row of this lane for an A operand (16 rows x 16 columns)
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t acol = static_cast<uint32_t>(lane >> 4) * 16u;
    // ... and for a B operand (8 rows x 16 columns; lanes 16-31 mirror 0-15)
    const int brow = lane & 7;
    const uint32_t bcol = static_cast<uint32_t>((lane >> 3) & 1) * 16u;

    // query rows by key channel (the bank's rows for selected queries)
    {
        const int rows = SEL ? g.qrows : M;
        uint16_t* qt = reinterpret_cast<uint16_t*>(smem + L.qtab);
        const int rw = static_cast<int>(qpitch / 2);
        for (int i = threadIdx.x; i < rows * R; i += nct) {
            const int r = i / R, c = i - r * R;
            qt[r * rw + c] = a.q[static_cast<long long>(r) * R + c];
        }
    }
    named_bar_sync(1, nct);

    // the A row this lane addresses for the logits: query `arow` of the token
    auto query_row = [&](long long n) -> uint32_t {
        if (arow >= M) return zero_s;
        if constexpr (SEL) {
            const long long id = a.ids[n * M + arow];
            if (id < 0 || id >= a.E) {
                atomicCAS(&g_multi_mma_error, 0u, static_cast<unsigned>(kSiteBadId));
                return zero_s;  // reads as a zero query
            }
            return qtab_s + static_cast<uint32_t>(id) * qpitch;
        } else {
            return qtab_s + static_cast<uint32_t>(arow) * qpitch;
        }
    };

    int k = 0;
    uint32_t phase = 0;
    uint32_t qnext = SEL ? query_row(blockIdx.x < N ? static_cast<long long>(blockIdx.x) : 0) : query_row(0);
    for (long long n = blockIdx.x; n < N; n += gridDim.x) {
        const uint32_t qrow = qnext;
        if constexpr (SEL) {
            const long long nn = n + gridDim.x;
            if (nn < N) qnext = query_row(nn);  // one token ahead
        }
        mbar_wait_s(full_s + 8u * k, phase, abort_flag, &g_multi_mma_error, kSiteFwdConsumer);
        const uint32_t slot = ring_s + static_cast<uint32_t>(k) * slot_bytes;

        // ---- key statistics: one warp per source
        for (int s = warp; s < S; s += kMmaWarps) {
            const uint32_t row = slot + static_cast<uint32_t>(s) * pitch + static_cast<uint32_t>(ko) * 2u;
            float2 acc = make_float2(0.0f, 0.0f);
            for (int v = lane; v < (R >> 3); v += 32) {
                const uint4 x = lds128(row + 16u * static_cast<uint32_t>(v));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float2 f = bf2_to_f2(u4_get(x, kk));
                    acc = ffma2(f, f, acc);
                }
            }
            const float ss = warp_sum(acc.x + acc.y);
            if (lane == 0) {
                const float r = rsqrtf(fmaf(ss, inv_r, a.eps));
                rtab[s] = r;
                a.rstd[n * S + s] = r;
            }
        }

        // ---- logits: this warp's share of the key's 16-channel steps
        {
            float c[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) c[j][e] = 0.0f;
            uint32_t brows[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int src = 8 * j + brow;
                brows[j] = src < S ? slot + static_cast<uint32_t>(src) * pitch + static_cast<uint32_t>(ko) * 2u
                                   : zero_s;
            }
            for (int kk = warp; kk < ksteps; kk += kMmaWarps) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(qrow + 32u * static_cast<uint32_t>(kk) + acol, a0, a1, a2, a3);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j < ntile) {
                        uint32_t b0, b1;
                        ldsm_x2(brows[j] + 32u * static_cast<uint32_t>(kk) + bcol, b0, b1);
                        mma_bf16_16816(c[j], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
            float* pw = part + warp * 16 * kPartPitch;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < ntile) {
                    *reinterpret_cast<float2*>(pw + g8 * kPartPitch + 8 * j + 2 * t4) = make_float2(c[j][0], c[j][1]);
                    *reinterpret_cast<float2*>(pw + (g8 + 8) * kPartPitch + 8 * j + 2 * t4) =
                        make_float2(c[j][2], c[j][3]);
                }
            }
        }
        named_bar_sync(1, nct);

        // ---- softmax: one warp per two queries, one lane per source
        for (int m = warp; m < M; m += kMmaWarps) {
            float z = -FLT_MAX;
            if (lane < S) {
                float dot = 0.0f;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) dot += part[(w * 16 + m) * kPartPitch + lane];
                z = a.scale * rtab[lane] * dot;
                a.logit[(n * M + m) * S + lane] = z;
            }
            const float mx = warp_max(z);
            const float e = lane < S ? __expf(z - mx) : 0.0f;
            const float al = e / warp_sum(e);
            if (lane < S) a.alpha[(n * M + m) * S + lane] = al;
            // the weight as three bf16 terms for the output MMA (each
            // difference is exact in FP32)
            const uint32_t hb = pack_bf16x2(al, 0.0f) & 0xffffu;
            const float r1 = al - __uint_as_float(hb << 16);
            const uint32_t mb = pack_bf16x2(r1, 0.0f) & 0xffffu;
            const uint32_t lb = pack_bf16x2(r1 - __uint_as_float(mb << 16), 0.0f) & 0xffffu;
            constexpr int tw = 16 * (kMmaAPitch / 2);  // elements per table
            atab[m * (kMmaAPitch / 2) + lane] = static_cast<uint16_t>(hb);
            atab[tw + m * (kMmaAPitch / 2) + lane] = static_cast<uint16_t>(mb);
            atab[2 * tw + m * (kMmaAPitch / 2) + lane] = static_cast<uint16_t>(lb);
        }
        named_bar_sync(1, nct);

        // ---- outputs: this warp's 8-channel column tiles
        {
            uint32_t af[3][2][4];  // [term][K tile][fragment]
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                if (kt < nkt) {
                    const uint32_t ra = atab_s + static_cast<uint32_t>(arow) * kMmaAPitch + 32u * kt + acol;
#pragma unroll
                    for (int h = 0; h < 3; ++h)
                        ldsm_x4(ra + 16u * kMmaAPitch * h, af[h][kt][0], af[h][kt][1], af[h][kt][2], af[h][kt][3]);
                }
            }
            uint32_t vrows[2];
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                const int src = 16 * kt + (lane & 7) + ((lane >> 3) & 1) * 8;
                vrows[kt] = src < S ? slot + static_cast<uint32_t>(src) * pitch : zero_s;
            }
            // groups of four 8-channel column tiles (32 channels); the tile is
            // staged in shared memory so each query row leaves as 16-byte stores
            const int ntot = D >> 3;
            const uint32_t stage_s = sbase + L.part + static_cast<uint32_t>(warp) * 16u * kPartPitch * 4u;
            uint16_t* const ybase = a.y + n * a.y_ns;
            for (int grp = warp; grp * 4 < ntot; grp += kMmaWarps) {
                float acc[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    if (kt < nkt) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int t = 4 * grp + j;
                            if (t < ntot) {
                                uint32_t b0, b1;
                                ldsm_x2_trans(vrows[kt] + 16u * static_cast<uint32_t>(t), b0, b1);
                                // smallest term first
#pragma unroll
                                for (int h = 2; h >= 0; --h)
                                    mma_bf16_16816(acc[j], af[h][kt][0], af[h][kt][1], af[h][kt][2], af[h][kt][3],
                                                   b0, b1);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t c = static_cast<uint32_t>(j * 8 + 2 * t4) * 2u;
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage_s + g8 * kStagePitch + c),
                                 "r"(pack_f2(make_float2(acc[j][0], acc[j][1]))));
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage_s + (g8 + 8) * kStagePitch + c),
                                 "r"(pack_f2(make_float2(acc[j][2], acc[j][3]))));
                }
                __syncwarp();
                for (int cix = lane; cix < 64; cix += 32) {
                    const int row = cix >> 2, ch = cix & 3;
                    const int col = 32 * grp + 8 * ch;
                    if (row < M && col + 8 <= D &&
                        ATTNRES_IN_BOUNDS(col + 8 <= D && row < M, &g_multi_mma_error)) {
                        const uint4 v = lds128(stage_s + static_cast<uint32_t>(row) * kStagePitch + 16u * ch);
                        st_global_cs_v4(ybase + static_cast<long long>(row) * a.y_ms + col, v);
                    }
                }
                __syncwarp();
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
}

template <bool SEL>
int mma_occupancy(int smem) {
    auto kern = attnres_multi_fwd_mma_kernel<SEL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kMmaThreads, static_cast<size_t>(smem)) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// ATTNRES_MULTI_FWD (read on every call): "mma" the tensor-core form whenever
// the shape qualifies, "simt" never; unset: from kMmaMinQueries queries up.
int mma_choice() {
    const char* v = std::getenv("ATTNRES_MULTI_FWD");
    if (!v || !v[0]) return -1;
    if (std::strcmp(v, "mma") == 0) return 1;
    if (std::strcmp(v, "simt") == 0) return 0;
    return -1;
}

}  // namespace

bool plan_multi_fwd_mma(const attnres_multi_params* p, int E, int sm_count, long long smem_optin, MmaPlan* out) {
    const attnres_params& b = p->base;
    const int choice = mma_choice();
    if (choice == 0) return false;
    if (choice < 0 && p->M < kMmaMinQueries) return false;
    if (b.S > kMmaMaxS || b.R % 16 != 0 || b.key_offset % 8 != 0 || b.N < 1) return false;
    MmaPlan pl{};
    pl.pitch = b.D * 2 + 16;
    pl.qpitch = b.R * 2 + 16;
    pl.qrows = E > 0 ? E : p->M;
    auto fit = [&](long long budget) {
        int k = 0;
        while (k < kMmaMaxSlots &&
               mma_layout(k + 1, b.S, pl.pitch, pl.qrows, pl.qpitch).total <= static_cast<uint32_t>(budget))
            ++k;
        return k;
    };
    int per_sm = 2;
    int slots = fit(smem_optin / 2 - 1024);
    if (slots < 2) {
        per_sm = 1;
        slots = fit(smem_optin);
    }
    if (slots < 2) return false;
    pl.slots = slots;
    pl.smem = mma_layout(slots, b.S, pl.pitch, pl.qrows, pl.qpitch).total;
    const int occ = E > 0 ? mma_occupancy<true>(static_cast<int>(pl.smem))
                          : mma_occupancy<false>(static_cast<int>(pl.smem));
    if (occ < 1) return false;
    if (per_sm > occ) per_sm = occ;
    long long grid = static_cast<long long>(per_sm) * sm_count;
    if (b.N < grid) grid = b.N;
    pl.grid = static_cast<int>(grid);
    *out = pl;
    return true;
}

cudaError_t launch_multi_fwd_mma(const MmaPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    MmaFwdArgs g;
    g.f = a;
    g.slots = plan.slots;
    g.pitch = plan.pitch;
    g.qpitch = plan.qpitch;
    g.qrows = plan.qrows;
    auto kern = a.ids ? attnres_multi_fwd_mma_kernel<true> : attnres_multi_fwd_mma_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem));
    if (err != cudaSuccess) return err;
    kern<<<plan.grid, kMmaThreads, plan.smem, stream>>>(g);
    return cudaGetLastError();
}

unsigned take_multi_mma_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_mma_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_mma_error, &zero, sizeof zero);
    return v;
}

}  // namespace attnres
