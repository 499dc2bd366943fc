// kernels.cuh -- kernel arguments, shared-memory layout and launch plan of
// the AttnRes forward/backward kernels (internal to the library).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "attnres.h"

namespace attnres {

constexpr int kMaxConsumerWarps = 8;
// Threads per CTA: up to 8 consumer warps and one producer warp.
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
// Forward CTAs per SM: with at most two 16-byte vectors per thread two CTAs
// fit (registers <= 96, half the shared memory each) and each CTA's barrier
// and softmax phases overlap the other's streaming work; wider rows run one.
__host__ __device__ constexpr int fwd_ctas_per_sm(int vpt) { return vpt <= 2 ? 2 : 1; }
constexpr int kMaxChunks = 32;
constexpr int kTokSlots = 4;      // token-statistics ring depth (backward)
constexpr int kGroupTicket = 12;  // CTAs per first-level group of the in-kernel reduction
constexpr int kMaxGroup = 32;     // forward rows reduced together

// Where a bounded wait gave up (value recorded in g_device_error).
enum WaitSite : unsigned {
    kSiteFwdProducer = 1,
    kSiteFwdConsumer = 2,
    kSiteBwdProducer = 3,
    kSiteBwdConsumer = 4,
    kSiteBwdTokStat = 5,
    kSiteDrain = 6,
    kSiteBadId = 7,  // a selected-query id outside [0, E)
    kSiteBwdExchange = 8,  // a cluster peer's partial sums did not arrive
    kSiteBounds = 9,       // debug build: a store's indices fell outside the call's sizes
};

// Debug build (-DATTNRES_DEBUG, a stand-in for a memory checker): a global
// store whose row, source or column index falls outside the call's sizes is
// recorded (site kSiteBounds, read by attnres_check_device_error) and skipped
// instead of made.  The release build evaluates nothing.
#ifdef ATTNRES_DEBUG
#define ATTNRES_IN_BOUNDS(cond, errp) \
    ((cond) ? true : (atomicCAS((errp), 0u, static_cast<unsigned>(::attnres::kSiteBounds)), false))
#else
#define ATTNRES_IN_BOUNDS(cond, errp) true
#endif

// Launch plan: one persistent CTA per SM.  `ncw` consumer warps each own
// `vpt` 16-byte column vectors of every row.  Source rows stream through a
// ring of `chunks` chunks; a chunk holds up to `rows` source rows of
// `slot_bytes` each and has one "full" and one "empty" mbarrier, so waits
// and releases are per chunk, not per row.  The backward also has a ring of
// `dy_slots` single-row slots for dy.
struct Plan {
    int grid;                // backward CTAs (b_per_sm per SM, or clusters of cl)
    int b_per_sm;            // backward CTAs that share an SM
    int fgrid;               // forward CTAs (fwd_ctas_per_sm per SM)
    int ncw, vpt;            // forward: consumer warps, 16-byte vectors per thread
    int b_ncw, b_vpt;        // backward
    int slot_bytes;          // forward ring slot (one whole row)
    int b_slot_bytes;        // backward ring slot (a row, or a cluster CTA's column slice)
    int s_pad;
    int f_rows, f_chunks;    // forward: rows per chunk, ring depth
    int f_group;             // forward softmax group rows (whole chunks)
    int b_rows, b_chunks;    // backward
    int dy_slots;
    int resident;            // backward keeps a token's rows between its passes
    int split;               // backward reduction via the finalize kernel
    int cl;                  // backward CTAs per token (a thread-block cluster; 1 = none)
    int slice;               // columns of a token each backward CTA holds (D / cl)
    int nparts;              // backward partial rows (CTAs, or clusters)
    size_t smem_fwd;
    size_t smem_bwd;
    size_t ws_bytes;         // backward workspace
    size_t ws_part_off, ws_gpart_off;
    int ngroups;
};

// Byte offsets inside the dynamic shared memory of one CTA.
struct SmemLayout {
    uint32_t ring, dyring, full, empty, dyfull, dyempty, tfull, tempty, red, tok, coef, qsm, misc, total;
    int red_rows;  // rows of the reduction scratch (per buffer)
};

// The reduction scratch is [2 buffers][red_rows][kRedPitch] floats: row =
// reduced quantity, column = consumer warp.  A pitch of 20 floats lets a lane
// read one row's 16 warp partials with four conflict-free 16-byte loads.
constexpr int kRedPitch = 20;

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Forward: chunk ring, z[s_pad] and rstd[s_pad] of the current token, and
// the query as bf16 indexed by channel (slot_bytes, zero outside the key);
// with the fused block-partial sum, `dy_slots` single-row slots for the
// added rows.  Backward: chunk ring, dy ring, token-statistics ring.
__host__ __device__ inline SmemLayout make_layout(int chunks, int rows, int slot_bytes, int dy_slots,
                                                  int s_pad, bool backward) {
    SmemLayout L;
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(chunks) * static_cast<uint32_t>(rows) * static_cast<uint32_t>(slot_bytes);
    L.dyring = off;
    off += static_cast<uint32_t>(dy_slots) * static_cast<uint32_t>(slot_bytes);
    off = align_up(off, 16);
    L.full = off;
    off += 8u * chunks;
    L.empty = off;
    off += 8u * chunks;
    L.dyfull = off;
    off += 8u * dy_slots;
    L.dyempty = off;
    off += 8u * dy_slots;
    L.tfull = off;
    off += backward ? 8u * kTokSlots : 0u;
    L.tempty = off;
    off += backward ? 8u * kTokSlots : 0u;
    off = align_up(off, 16);
    L.red = off;
    L.red_rows = s_pad > 64 ? s_pad : 64;
    off += 2u * static_cast<uint32_t>(L.red_rows) * kRedPitch * 4u;
    L.tok = off;
    off += backward ? static_cast<uint32_t>(kTokSlots) * (3u * s_pad + 4u) * 4u : 0u;
    L.coef = off;
    off += backward ? 0u : 2u * s_pad * 4u;
    off = align_up(off, 16);
    L.qsm = off;
    off += backward ? 0u : static_cast<uint32_t>(slot_bytes);
    L.misc = off;  // abort flag, ticket flags
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

struct FwdArgs {
    const void* src[ATTNRES_MAX_S];
    long long N;
    long long src_ld;
    int S, D, R, ko, out_norm;
    float eps, scale;
    int chunks, rows, slot_bytes, ncw, s_pad;
    int group;          // softmax group rows (a whole number of chunks, <= kMaxGroup)
    const uint16_t* q;
    const uint16_t* w_o;
    uint16_t* y;
    float* alpha;
    float* rstd;
    float* logit;
    float* o_rstd;
    float* o_pre;       // optional FP32 [N, D] pre-norm mixture
    // Fused block-partial sum: source S-1 is formed as src[S-1] + delta
    // (rounded to bf16) and written to partial_out; NULL = plain read.
    const uint16_t* delta;
    long long delta_ld;
    uint16_t* partial_out;
    long long partial_ld;
    // Test hooks (zero in every ordinary launch): with test_withhold = k > 0
    // the producer of CTA 0 never issues its k-th chunk fill (and stops), so
    // that CTA's consumers give up waiting for it after test_wait_ns
    // nanoseconds (0: the default limit) -- the bounded-wait recovery path.
    long long test_withhold;
    uint64_t test_wait_ns;
};
constexpr int kDeltaSlots = 2;

struct BwdArgs {
    const void* src[ATTNRES_MAX_S];
    void* dsrc[ATTNRES_MAX_S];
    long long N;
    long long src_ld, dsrc_ld;
    long long dsrc_stride;  // bytes between dsrc[s] and dsrc[s+1] when evenly spaced, else 0
    int S, D, R, ko, out_norm;
    float eps, scale;
    int chunks, rows, slot_bytes, dy_slots, ncw, s_pad, resident, split, ngroups;
    int cl, slice;      // cluster size and columns per CTA (cl == 1: slice == D)
    const uint16_t* q;
    const uint16_t* w_o;
    const uint16_t* dy;
    const float* alpha;
    const float* rstd;
    const float* logit;
    const float* o_rstd;
    const float* o_pre;  // optional FP32 [N, D]; NULL = recompute o from the sources
    float* part;        // [grid][R + Dw] per-CTA partial sums (Dw = out_norm ? D : 0)
    int part_rows;      // rows the workspace holds at part (the plan's partial rows)
    float* gpart;       // [ngroups][R + Dw] group sums (in-kernel reduction)
    unsigned* tickets;  // [ngroups + 1] zeroed before launch (in-kernel reduction)
    uint16_t* dq;
    float* dq_f32;
    uint16_t* dw_o;
    float* dw_o_f32;
    // optional gradient added to the last source's gradient before rounding
    // (the fused block-partial sum's later uses); NULL = none
    const uint16_t* dlast_add;
    long long dlast_add_ld;
};

// Backward over a thread-block cluster: the backward layout of one CTA's
// column slice plus the exchange area, [2 buffers][cl ranks][s_pad] floats
// that peers write their per-token partial sums into, two mbarriers (one per
// buffer) that count the peers' arrivals, and each consumer warp's table of
// the token's per-source coefficients, [warps][s_pad] x {alpha, k1, k2, 0}.
struct ClusterLayout {
    SmemLayout base;
    uint32_t xbar, xbuf, ctab, total;
};

constexpr int kClusterMax = 8;          // portable cluster size
constexpr int kExchangeArrivals = 32;   // arrivals per exchange (every lane of one warp in each CTA)

__host__ __device__ inline ClusterLayout make_cluster_layout(int chunks, int rows, int slot_bytes, int dy_slots,
                                                             int s_pad, int cl) {
    ClusterLayout L;
    L.base = make_layout(chunks, rows, slot_bytes, dy_slots, s_pad, true);
    uint32_t off = align_up(L.base.total, 16);
    L.xbar = off;
    off += 2u * 8u;
    L.xbuf = off;
    off += 2u * static_cast<uint32_t>(cl) * static_cast<uint32_t>(s_pad) * 4u;
    off = align_up(off, 16);
    L.ctab = off;
    off += static_cast<uint32_t>(kMaxConsumerWarps) * static_cast<uint32_t>(s_pad) * 16u;
    L.total = align_up(off, 128);
    return L;
}

// The cluster backward (attnres_bwd_cluster.cu): launch, the largest number
// of its clusters that fit on the device at once (0 when the shape cannot
// run as a cluster), and its wait-failure record.
cudaError_t launch_bwd_cluster(const Plan& plan, const BwdArgs& a, cudaStream_t stream);
int bwd_cluster_max_active(const Plan& plan, bool keyall, bool norm, int S);
unsigned take_bwd_error_cluster();

// ---------------------------------------------------------------------------
// Multi-query read: M queries share one read of the sources.  A token's S
// rows stay resident in the chunk ring while every query is served; the
// backward also keeps the token's M dy rows (a ring of `dy_slots` groups of
// M rows) and its saved statistics (two slots) in shared memory.
// ---------------------------------------------------------------------------
constexpr int kMultiTokSlots = 2;
// The multi-query backward runs up to 16 consumer warps (one 16-byte vector
// per thread up to D = 4096) so that more warps hide shared-memory and
// barrier latency; registers are then capped near 120 per thread.
constexpr int kMultiBwdWarps = 16;
constexpr int kMultiBwdThreads = (kMultiBwdWarps + 1) * 32;

struct MultiLayout {
    uint32_t ring, dyring, full, empty, dyfull, dyempty, tfull, tempty, tok, tab, qsm, dqsm, misc, total;
    uint32_t tstride;  // floats per statistics slot
};

// Backward layout.  Tables (floats): da[m_pad][s_pad], alpha[s_pad][m_pad],
// b[s_pad][m_pad], zr[m_pad][s_pad].  qsm: q_rows (default m_pad) query rows
// of nkv 16-byte vectors (bf16); a resident query bank takes E + 1 rows.
// dqsm (only when the queries take several register blocks): dq_rows rows
// (queries, or bank rows) of dq_nkv * 8 FP32 partial sums.
__host__ __device__ inline MultiLayout make_multi_layout(int chunks, int rows, int slot_bytes, int M,
                                                        int dy_slots, int s_pad, int m_pad, int nkv,
                                                        int dq_nkv, bool backward, int dq_rows = -1,
                                                        int q_rows = -1) {
    MultiLayout L;
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(chunks) * static_cast<uint32_t>(rows) * static_cast<uint32_t>(slot_bytes);
    L.dyring = off;
    off += backward ? static_cast<uint32_t>(dy_slots) * static_cast<uint32_t>(M) * static_cast<uint32_t>(slot_bytes) : 0u;
    off = align_up(off, 16);
    L.full = off;
    off += 8u * chunks;
    L.empty = off;
    off += 8u * chunks;
    L.dyfull = off;
    off += backward ? 8u * dy_slots : 0u;
    L.dyempty = off;
    off += backward ? 8u * dy_slots : 0u;
    L.tfull = off;
    off += backward ? 8u * kMultiTokSlots : 0u;
    L.tempty = off;
    off += backward ? 8u * kMultiTokSlots : 0u;
    off = align_up(off, 16);
    L.tstride = align_up(static_cast<uint32_t>(2 * M * s_pad + s_pad), 4u);
    L.tok = off;
    off += backward ? kMultiTokSlots * L.tstride * 4u : 0u;
    L.tab = off;
    off += 4u * m_pad * s_pad * 4u;
    off = align_up(off, 16);
    L.qsm = off;
    off += static_cast<uint32_t>(q_rows < 0 ? m_pad : q_rows) * static_cast<uint32_t>(nkv) * 16u;
    L.dqsm = off;
    off += backward ? static_cast<uint32_t>(dq_rows < 0 ? M : dq_rows) * static_cast<uint32_t>(dq_nkv) * 32u : 0u;
    L.misc = off;  // abort flag
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

// Forward of the multi-query read: streamed like the single-query forward
// (online softmax over groups of whole chunks), MB queries per pass over a
// token.  Layout: chunk ring, full/empty mbarriers, pass-1 results
// [2][1 + kMultiMaxMB][kMaxGroup], logits of the block's queries
// [kMultiMaxMB][s_pad], key rstd [s_pad], queries [qrows][nkv * 8] bf16.
constexpr int kMultiMaxMB = 4;
// Register budget of the forward: two CTAs of up to 288 threads per SM when a
// thread owns at most two vectors.  The planner may place more CTAs of
// narrower rows (fewer warps) on an SM when they fit.
__host__ __device__ constexpr int multi_fwd_ctas_per_sm(int vpt) { return vpt <= 2 ? 2 : 1; }
constexpr int kMultiMaxCtasPerSm = 4;
// Query counts with their own kernel instantiations (M a compile-time
// constant: no per-query predicates in the unrolled loops); other counts run
// the run-time-M kernels.
__host__ __device__ constexpr int multi_fixed_m(int M) { return (M == 1 || M == 2 || M == 4) ? M : 0; }
__host__ __device__ constexpr int multi_pow2_ceil(int x) { return x <= 1 ? 1 : 2 * multi_pow2_ceil((x + 1) / 2); }
// Queries per register block: forward 4 / VPT, backward 2 / VPT, at most the
// next power of two of M.
__host__ __device__ constexpr int multi_fwd_mb(int M, int vpt) {
    return multi_pow2_ceil(M) < kMultiMaxMB / vpt ? multi_pow2_ceil(M) : kMultiMaxMB / vpt;
}
__host__ __device__ constexpr int multi_bwd_mb(int M, int vpt) {
    return multi_pow2_ceil(M) < 2 / vpt ? multi_pow2_ceil(M) : 2 / vpt;
}

struct MultiFwdLayout {
    uint32_t ring, full, empty, red, zall, rall, qsm, misc, total;
};

__host__ __device__ inline MultiFwdLayout make_multi_fwd_layout(int chunks, int rows, int slot_bytes, int s_pad,
                                                               int qrows, int nkv) {
    MultiFwdLayout L;
    uint32_t off = 0;
    L.ring = off;
    off += static_cast<uint32_t>(chunks) * static_cast<uint32_t>(rows) * static_cast<uint32_t>(slot_bytes);
    off = align_up(off, 16);
    L.full = off;
    off += 8u * chunks;
    L.empty = off;
    off += 8u * chunks;
    off = align_up(off, 16);
    L.red = off;
    off += 2u * (1 + kMultiMaxMB) * kMaxGroup * 4u;
    L.zall = off;
    off += static_cast<uint32_t>(kMultiMaxMB) * s_pad * 4u;
    L.rall = off;
    off += static_cast<uint32_t>(s_pad) * 4u;
    off = align_up(off, 16);
    L.qsm = off;
    off += static_cast<uint32_t>(qrows) * static_cast<uint32_t>(nkv) * 16u;
    L.misc = off;
    off += 16u;
    L.total = align_up(off, 128);
    return L;
}

struct MultiPlan {
    // general two-kernel backward (attnres_multi_general.cu): used when the
    // resident layout does not fit or for more than kMultiResidentMaxM queries
    int gen;
    int gen_grid_a, gen_grid_b, gen_groups;   // CTAs of the two kernels, token groups of the second
    size_t gen_smem_a, gen_smem_b;
    int gen_s8, gen_kgroups, gen_bufs, gen_dc, gen_pitch, gen_cs;
    int gen_dcb, gen_rows_b, gen_chunks_b, gen_bank_rows, gen_tslots_b;
    int gen_grad_mma;                         // gradient kernel on the tensor cores (attnres_multi_grad_mma.cu)
    size_t gen_part_off;                      // workspace: coefficient tables, then partial rows
    int grid;
    int fgrid;             // forward CTAs (multi_fwd_ctas_per_sm per SM)
    int f_group;           // forward softmax group rows (whole chunks, <= kMaxGroup)
    int qrows;             // query rows held in shared memory by the forward
    int bwd_ok;            // the backward's resident layout fits
    int E;                 // query bank rows (selected-query read), 0 otherwise
    int bank_f, bank_b;    // E + 1 when the bank (plus a zero row) stays in the forward's /
                           // backward's shared memory for the whole launch, else 0
    int ncw, vpt;          // forward: consumer warps, 16-byte vectors per thread
    int b_ncw, b_vpt;      // backward
    int mb_f, mb_b;        // queries per register block (forward / backward)
    int mq;                // M when the kernels are instantiated for it (1, 2 or 4), else 0
    int slot_bytes, s_pad, m_pad;
    int kv0, nkv;          // key window in 16-byte vectors
    int f_rows, f_chunks;  // forward chunk ring
    int b_rows, b_chunks, dy_slots;
    size_t smem_fwd, smem_bwd;
    size_t ws_bytes;       // backward workspace: [grid][M * R] FP32 partials
};

struct MultiFwdArgs {
    const void* src[ATTNRES_MAX_S];
    long long N, src_ld;
    long long y_ms, y_ns;  // elements between queries / tokens of the output
    int S, D, R, ko, M;
    float eps, scale;
    int chunks, rows, slot_bytes, ncw, s_pad, kv0, nkv;
    int group;             // softmax group rows (whole chunks)
    int qrows;             // query rows in shared memory (M, or MB: reloaded per block)
    const uint16_t* q;     // [M][R], or the query bank [E][R] when ids is set
    const long long* ids;  // [N][M] bank row of every (token, slot), or NULL
    int E;                 // bank rows
    int bank_rows;         // E + 1: the bank and a zero row stay in qsm (rows as ids), else 0
    uint16_t* y;
    float* alpha;          // [N][M][S]
    float* rstd;           // [N][S]
    float* logit;          // [N][M][S]
};

// The tensor-core multi-query forward (attnres_multi_fwd_mma.cu): for reads
// with several queries whose token's rows fit in shared memory at least
// twice.  plan_multi_fwd_mma is false when the shape does not qualify (then
// the kernel of attnres_multi_fwd_kernel.cuh runs).
struct MmaPlan {
    int grid, slots, pitch, qpitch, qrows;
    size_t smem;
};
bool plan_multi_fwd_mma(const attnres_multi_params* p, int E, int sm_count, long long smem_optin, MmaPlan* out);
cudaError_t launch_multi_fwd_mma(const MmaPlan& plan, const MultiFwdArgs& a, cudaStream_t stream);
unsigned take_multi_mma_error();

struct MultiBwdArgs {
    const void* src[ATTNRES_MAX_S];
    void* dsrc[ATTNRES_MAX_S];
    long long N, src_ld, dsrc_ld;
    long long dy_ms, dy_ns;
    int S, D, R, ko, M;
    float eps, scale;
    int chunks, rows, slot_bytes, dy_slots, ncw, s_pad, m_pad, kv0, nkv;
    const uint16_t* q;
    const uint16_t* dy;
    const float* alpha;
    const float* rstd;
    const float* logit;
    float* part;           // [grid][Q * R], Q = M (or E with ids)
    uint16_t* dq;          // [Q][R]
    float* dq_f32;         // [Q][R] or NULL
    const long long* ids;  // [N][M] bank row of every (token, slot), or NULL
    int E;                 // bank rows
    int bank_rows;         // E + 1: the bank and a zero row stay in qsm (rows as ids), else 0
};

// Arguments of the general multi-query backward (attnres_multi_general.cu).
struct MultiGenArgs {
    const void* src[ATTNRES_MAX_S];
    void* dsrc[ATTNRES_MAX_S];
    long long N, src_ld, dsrc_ld, dy_ms, dy_ns;
    int S, D, R, ko, M, E;
    float scale;
    // coefficient kernel: sources padded to s8, k groups of warps, ring of
    // `bufs` row blocks of `dc` columns (`pitch` bytes per row), `nblocks`
    // blocks per row, `cs` floats per source in the coefficient table
    int s8, kgroups, bufs, nblocks, dc, pitch, cs;
    // gradient kernel: column blocks of `dcb`, source chunks of `rows_b` rows
    // in a ring of `chunks_b`, bank rows kept in shared memory (E + 1, or 0)
    int dcb, rows_b, chunks_b, bank_rows, tslots_b;
    const uint16_t* q;     // [M][R], or the bank [E][R] with ids
    const long long* ids;  // [N][M] or NULL
    const uint16_t* dy;
    const float* alpha;
    const float* rstd;
    const float* logit;
    float* coef;           // [N][S][cs] workspace
    float* part;           // [groups][Q * R] workspace
    uint16_t* dq;
    float* dq_f32;
};
// Queries up to which the resident one-CTA multi-query backward runs (when
// its layout fits); more queries take the general backward (measured, S=10
// N=32768: M=2 D=4096 0.91 ms resident against 2.29 general, but M=3 D=4096
// 2.85 against 2.29, M=4 D=1024 0.77 against 0.68, S=16 N=16384 D=2048 M=4
// 1.50 against 0.84).
constexpr int kMultiResidentMaxM = 2;
constexpr int kMultiGenColumns = 512;   // columns per CTA of the gradient kernel, per column pair of a thread
constexpr int kMultiGenMaxBufs = 12;    // row-block buffers of the coefficient kernel
constexpr int kMultiCoefWarps = 4;      // consumer warps of the coefficient kernel
constexpr int kMultiGenMaxSlots = 8;    // token slots of the gradient kernel
// Queries from which the general backward's gradient kernel runs on the
// tensor cores (measured, S=10 N=32768: M=16 D=1024 1.45 against 2.05 ms for
// the whole backward, M=16 D=4096 5.53 against 7.92 ms, but M=8 D=4096 4.94
// against 4.22 ms).
constexpr int kMultiGradMmaMinM = 9;
size_t multi_gen_smem_a(int bufs, int s8, int pitch, int M, int S, int kgroups, int cs);
size_t multi_gen_smem_b(int S, int cs, int M, int dcb, int rows, int chunks, int bank_rows, int tslots);
cudaError_t launch_multi_bwd_general(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream);
unsigned take_multi_gen_error();
// Gradient kernel of the general backward on the tensor cores (fixed
// queries, at most 16 sources): its shared memory with `slots` token slots,
// its launch (grid and shared memory from the plan's gen_grid_b,
// gen_smem_b; token slots in a.tslots_b) and its first failed wait.
size_t multi_grad_mma_smem(int S, int cs, int M, int slots);
cudaError_t launch_multi_grad_mma(const MultiPlan& plan, const MultiGenArgs& a, cudaStream_t stream);
unsigned take_multi_grad_mma_error();

unsigned take_multi_fwd_error();
unsigned take_multi_bwd_error();
cudaError_t launch_multi_fwd(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream);
// CTAs of the plan's kernel variant that fit on one SM (0 on error).
int multi_fwd_occupancy(const MultiPlan& plan);
int multi_bwd_occupancy(const MultiPlan& plan);
cudaError_t launch_multi_bwd(const MultiPlan& plan, const MultiBwdArgs& a, cudaStream_t stream);
// Column sums of a [P][W] FP32 partial matrix in row order; columns < R go to
// dq (bf16 + optional FP32), the rest to dw_o.
cudaError_t launch_finalize(const float* part, int P, int R, int W, uint16_t* dq, float* dq_f32,
                            uint16_t* dw_o, float* dw_o_f32, cudaStream_t stream);

// Host-side launchers (return a CUDA error code) and the per-kernel records
// of failed waits (read and cleared; 0 = none).
unsigned take_fwd_error();
unsigned take_bwd_error();
// backward kernels with the output norm, by where o comes from (the dispatch
// in launch_bwd picks them); each unit's wait-failure record
cudaError_t launch_bwd_norm_rebuild(const Plan& plan, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_norm_saved(const Plan& plan, const BwdArgs& a, cudaStream_t stream);
unsigned take_bwd_error_rebuild();
unsigned take_bwd_error_saved();
cudaError_t launch_fwd(const Plan& plan, const FwdArgs& a, cudaStream_t stream);
// The forwards compiled at run time for the plan's exact shape (S, rows per
// chunk, group rows, ring depth as constants); cudaErrorNotSupported when
// that path is off or unavailable (the caller then launches a precompiled
// instance).  Its modules' wait-failure records, and how many kernels it holds.
cudaError_t jit_launch_fwd(const Plan& plan, const FwdArgs& a, cudaStream_t stream);
cudaError_t jit_launch_multi_fwd(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream);
unsigned take_jit_error(int kind);  // 0: single-query forward, 1: multi-query forward
int jit_fwd_kernels();
// Tokens from which a forward launch uses the run-time-compiled kernel.
constexpr long long kJitMinTokens = 1024;
cudaError_t launch_bwd(const Plan& plan, const BwdArgs& a, cudaStream_t stream);

}  // namespace attnres
