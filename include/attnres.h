/*
 * attnres.h -- C ABI of the GB300 (sm_103a) Attention Residuals read operator.
 *
 * The operator ("Fast Attention Residuals", sections "Quickstart" and
 * "Equation"): for every token n and S ordered full-width residual sources
 * v_s[n, 0:D] (bf16),
 *
 *   t_s   = v_s[n, key_offset : key_offset + R]      implicit key slice
 *   r_s   = 1 / sqrt(mean(t_s^2) + eps)              key reciprocal RMS ("rstd")
 *   z_s   = scale * r_s * <t_s, q>                   routing logit
 *   a_s   = softmax_s(z)                             routing weight ("alpha")
 *   o     = sum_s a_s * v_s[n, 0:D]
 *   y     = o                                        (out_norm == 0)
 *   y     = o * o_rstd * w_o, o_rstd = 1/sqrt(mean(o^2) + eps)   (out_norm == 1)
 *
 * The optional output RMSNorm and the statistic saved for backward reuse
 * (the output reciprocal RMS o_rstd) follow "[Perf] Parallelize AttnRes
 * long-sequence reduction", Summary.  The page's canonical key slice
 * is the final R channels (key_offset = D - R); any 0 <= key_offset <= D - R
 * is accepted.  Standard AttnRes is R == D; sliced low-rank routing is R < D
 * ("Fast Attention Residuals", section "Sliced LR-AttnRes").
 *
 * The backward returns dvalues, dq and dw_o; dq and dw_o are sums over all N
 * tokens.  For N >= split_n_threshold the per-CTA FP32 partial sums are
 * combined by a separate finalize kernel; shorter inputs finish the
 * reduction inside the backward kernel (the last CTA of each group, then the
 * last group, add the partials).  The page splits at 16384 tokens; on this
 * GPU the finalize kernel measured as fast or faster at every N, so the
 * default threshold is 1 (always the finalize kernel) and the in-kernel form
 * is there for callers that set a larger one.  Both orders are fixed, so dq
 * and dw_o are bitwise reproducible run to run.
 *
 * A token whose S source rows do not fit in one SM's shared memory (e.g. 64
 * rows of 8192 channels, 1 MB) is shared by a thread-block cluster of 2, 4
 * or 8 CTAs in the backward, each holding D/size columns of every row: the
 * rows are streamed once per pass, and with size-times fewer tokens in flight
 * the later passes find them in L2 instead of HBM; the CTAs exchange their
 * partial sums of the two full-width reductions through distributed shared
 * memory.  Its partial rows (one per cluster) always go through the finalize
 * kernel.  ATTNRES_BWD_CLUSTER in the environment (read on every call)
 * overrides the choice: "0" one CTA per token for every shape, "2"/"4"/"8"
 * clusters holding their slices resident, "s2"/"s4"/"s8" clusters streaming
 * them, "h2"/"h4"/"h8" the same with two CTAs per SM; a form the shape cannot
 * take falls back to one CTA per token.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers of the current CUDA device,
 *    except the attnres_params struct and the dsrc pointer array, which live
 *    in host memory and are read during the call only.
 *  - The caller owns every buffer, including the backward workspace.  The
 *    library allocates no device memory for data.  One exception: the first
 *    forward of 1024 or more tokens with a new shape on a device compiles a
 *    kernel for that shape on the host (NVRTC, inside the call, typically a
 *    few hundred milliseconds) and loads it as a module, for which the
 *    driver allocates the module's code and a 4-byte error word; later calls
 *    of that shape reuse it.  A shape first seen while the stream is being
 *    captured into a CUDA graph runs a precompiled kernel instead (see
 *    attnres_jit_kernel_count; ATTNRES_JIT=0 turns the run-time path off).
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and never synchronise the host.  Stream order holds:
 *    the backward kernels are launched with programmatic dependent launch,
 *    so they may start their set-up during the previous kernel's tail, but
 *    they touch no global memory before that kernel has finished.
 *  - Arguments are validated before anything is enqueued; on any error
 *    nothing is launched and the status says why.
 *  - bf16 is IEEE bfloat16 stored as uint16_t bit patterns.
 *  - Rows: every source row, dy row, y row and dvalues row starts on a
 *    16-byte boundary and D is a multiple of 8.
 */
#ifndef ATTNRES_H_
#define ATTNRES_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTNRES_MAX_S 128      /* most sources one call accepts           */
#define ATTNRES_MAX_D 8192     /* widest row one call accepts             */
#define ATTNRES_DEFAULT_SPLIT_N 1

typedef enum {
    ATTNRES_OK = 0,
    ATTNRES_ERR_INVALID_ARG = 1,  /* a size, flag or pointer is out of range      */
    ATTNRES_ERR_ALIGNMENT = 2,    /* a pointer or row stride breaks 16-byte rows  */
    ATTNRES_ERR_UNSUPPORTED = 3,  /* legal shape this build does not handle       */
    ATTNRES_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than required      */
    ATTNRES_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed         */
    ATTNRES_ERR_DEVICE = 6        /* a kernel reported a failed wait or a bad id  */
} attnres_status;

/*
 * Shape and source description shared by forward and backward.
 *   S            number of sources, 1 <= S <= ATTNRES_MAX_S
 *   D            row width, 8 <= D <= ATTNRES_MAX_D, D % 8 == 0
 *   R            key rank, 1 <= R <= D
 *   key_offset   first key channel, 0 <= key_offset <= D - R
 *   N            tokens (B*T*H flattened), N >= 0; N == 0 is a no-op
 *   eps          added to the mean square inside the root (default 2^-23)
 *   scale        logit multiplier applied after key normalisation (default 1)
 *   out_norm     0 or 1: apply the output RMSNorm with weight w_o
 *   split_n_threshold  N at or above which the backward uses the finalize
 *                kernel; <= 0 selects ATTNRES_DEFAULT_SPLIT_N
 *   src_ld       element stride between consecutive token rows of each
 *                source, src_ld >= D, src_ld % 8 == 0
 *   src[s]       device pointer to source s, row n at src[s] + n * src_ld
 *                (bf16, 16-byte aligned).  The same pointer may appear more
 *                than once (a shared source read twice).
 */
typedef struct {
    int32_t S;
    int32_t D;
    int32_t R;
    int32_t key_offset;
    int64_t N;
    float eps;
    float scale;
    int32_t out_norm;
    int32_t split_n_threshold;
    int64_t src_ld;
    const void* src[ATTNRES_MAX_S];
} attnres_params;

/*
 * Forward.  Outputs (device, caller-allocated, fully overwritten):
 *   y       bf16 [N, D] contiguous
 *   alpha   f32  [N, S]  routing weights a_s
 *   rstd    f32  [N, S]  key reciprocal RMS r_s
 *   logit   f32  [N, S]  routing logits z_s
 *   o_rstd  f32  [N]     output reciprocal RMS; required iff out_norm, else ignored
 *   o_pre   f32  [N, D]  optional (NULL allowed; must be NULL without out_norm):
 *                        the pre-norm mixture o.  The backward rebuilds o from
 *                        the sources when it is NULL, which is free when the
 *                        backward keeps a token's rows in shared memory
 *                        (attnres_plan_info slot 5, which counts a cluster's
 *                        column slices) and costs one more pass over the
 *                        sources otherwise.  The cluster backward always
 *                        rebuilds o and does not read o_pre.
 *   q       bf16 [R]     query;  w_o bf16 [D], required iff out_norm
 * alpha, rstd, logit, o_rstd (and o_pre) are what attnres_bwd consumes.
 * Errors: INVALID_ARG (sizes, NULL pointers), ALIGNMENT (16-byte rows),
 * UNSUPPORTED (no kernel configuration fits), CUDA (launch failure).
 */
attnres_status attnres_fwd(const attnres_params* p, const void* q, const void* w_o,
                           void* y, float* alpha, float* rstd, float* logit,
                           float* o_rstd, float* o_pre, void* stream);

/*
 * Bytes of device workspace attnres_bwd needs for these params on the
 * current device (0 when N == 0).  Depends on S, D, R, N, out_norm,
 * split_n_threshold, the device's SM count and shared memory, and
 * ATTNRES_BWD_CLUSTER only.
 */
size_t attnres_bwd_workspace_bytes(const attnres_params* p);

/*
 * Backward.  Inputs: q, w_o (iff out_norm), dy bf16 [N, D] contiguous, and
 * the forward's alpha, rstd, logit, o_rstd and (optional, may be NULL) o_pre
 * for the same sources.
 * Outputs (written, never accumulated):
 *   dsrc       host array of S device pointers; dsrc[s] receives the
 *              gradient of source s, bf16 rows at dsrc[s] + n * dsrc_ld
 *              (dsrc_ld >= D, % 8 == 0, 16-byte aligned rows).  Entries must
 *              be distinct and must not overlap any source or each other.
 *              Shared (repeated) sources get one gradient per occurrence; the
 *              caller adds them.
 *   dq         bf16 [R];   dq_f32   f32 [R] (may be NULL)
 *   dw_o       bf16 [D];   dw_o_f32 f32 [D] (may be NULL); required iff out_norm
 *   workspace  device scratch of at least attnres_bwd_workspace_bytes(p)
 *              bytes, 16-byte aligned; contents on entry are ignored.
 * Errors: as attnres_fwd, plus WORKSPACE.
 */
attnres_status attnres_bwd(const attnres_params* p, const void* q, const void* w_o,
                           const void* dy, const float* alpha, const float* rstd,
                           const float* logit, const float* o_rstd, const float* o_pre,
                           void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                           void* dw_o, float* dw_o_f32, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Fused block-partial read ("Fast Attention Residuals", section "Full and
 * Block schedules": Block supplies the embedding, the completed block sums
 * and the current partial sum, which the caller sums before the read).
 * Instead of materialising partial_new = partial + delta in a separate pass
 * and reading it back, the forward takes the previous partial sum as the
 * last source (src[S-1]) and the newest writer output `delta`, forms
 *
 *   partial_new[n] = partial[n] + delta[n]     (FP32 add, one bf16 rounding:
 *                                               exactly a bf16 tensor add)
 *
 * in shared memory, writes it to `partial_out` and reads the sources
 * (src[0..S-2], partial_new) exactly as attnres_fwd does.  One [N, D] read
 * and one launch less per layer than summing first.
 *   delta         bf16 rows at delta + n * delta_ld (16-byte aligned)
 *   partial_out   bf16 rows at partial_out + n * partial_ld; may be the same
 *                 memory as src[S-1] (an in-place update: each row is read
 *                 before it is written), must not overlap anything else
 * Other arguments, outputs and errors as attnres_fwd.
 */
attnres_status attnres_fwd_partial(const attnres_params* p, const void* q, const void* w_o,
                                   const void* delta, int64_t delta_ld, void* partial_out,
                                   int64_t partial_ld, void* y, float* alpha, float* rstd,
                                   float* logit, float* o_rstd, float* o_pre, void* stream);

/*
 * Backward of the fused block-partial read.  The caller passes the sources
 * with src[S-1] = partial_new (the forward's partial_out).  `g_partial`
 * (bf16 rows at g_partial + n * g_ld, or NULL) is the gradient reaching
 * partial_new from its later uses; it is added, before rounding, to the
 * gradient of the last source, so dsrc[S-1] receives the full gradient of
 * partial_new -- which is the gradient of both `partial` and `delta` (they
 * feed partial_new with unit weight).  Other arguments, outputs and errors
 * as attnres_bwd.
 */
attnres_status attnres_bwd_partial(const attnres_params* p, const void* q, const void* w_o,
                                   const void* dy, const float* alpha, const float* rstd,
                                   const float* logit, const float* o_rstd, const float* o_pre,
                                   const void* g_partial, int64_t g_ld, void* const* dsrc,
                                   int64_t dsrc_ld, void* dq, float* dq_f32, void* dw_o,
                                   float* dw_o_f32, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * Backward without a caller-supplied workspace (no counterpart in the
 * papers; it exists for callers that cannot allocate device memory, such as
 * code running inside a region being captured into a CUDA graph, plugins
 * that must not touch the allocator of the process hosting them, or
 * latency-critical paths where cudaMalloc's implicit synchronisation is not
 * acceptable).  Same arguments and results as attnres_bwd minus the
 * workspace: the scratch lives in a fixed device array of the library of
 * ATTNRES_NOALLOC_SCRATCH_BYTES bytes (16 MiB), which every GPU that loads
 * the library holds until the process exits.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 *     call.  The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Shapes whose scratch (attnres_bwd_workspace_bytes) exceeds the array
 *     are rejected with ATTNRES_ERR_WORKSPACE before anything is enqueued.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race and give wrong results; serialise
 *     them, e.g. on one stream.  The parts of the array that must start at
 *     zero are cleared by every call on its stream.
 */
#define ATTNRES_NOALLOC_SCRATCH_BYTES (16u << 20)
attnres_status attnres_bwd_noalloc(const attnres_params* p, const void* q, const void* w_o,
                                   const void* dy, const float* alpha, const float* rstd,
                                   const float* logit, const float* o_rstd, const float* o_pre,
                                   void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                   void* dw_o, float* dw_o_f32, void* stream);

/*
 * Training step from host memory: attnres_fwd + attnres_bwd over all N
 * tokens with the sources and dy in HOST memory and every result written
 * back to HOST memory.  Tokens are independent ("Fast Attention Residuals",
 * section "Equation"), so the step runs over chunks of chunk_tokens tokens
 * with double-buffered device staging on three streams: streams[1] copies
 * chunk c+1 in, streams[0] runs chunk c's kernels, streams[2] copies chunk
 * c-1's y and dvalues out, so both copy directions and the kernels overlap.
 * dq and dw_o sum every chunk's FP32 sums in chunk order (reproducible).
 *   p          as for attnres_fwd, except src[s] are HOST pointers (pinned
 *              memory gives asynchronous full-speed copies; pageable memory
 *              works but each copy then blocks the host)
 *   q, w_o     HOST bf16 [R] and [D] (w_o iff out_norm)
 *   dy         HOST bf16 rows at dy + n * dy_ld
 *   y          HOST bf16 rows at y + n * y_ld (written)
 *   dsrc[s]    HOST bf16 rows at dsrc[s] + n * dsrc_ld (written)
 *   dq, dq_f32, dw_o, dw_o_f32   HOST, written (the FP32 copies may be NULL;
 *              dw_o required iff out_norm)
 *   workspace  DEVICE, at least attnres_step_host_workspace_bytes(p,
 *              chunk_tokens) bytes, 256-byte aligned
 *   streams    three cudaStream_t (entries may repeat; NULL = legacy default)
 * Asynchronous: returns once everything is enqueued; streams[0] waits for the
 * other two at its end, so synchronising streams[0] (or an event recorded on
 * it after the call) completes the step.  Host buffers must stay valid and
 * untouched until then.  The per-token statistics stay on the device.
 * Errors: as attnres_fwd and attnres_bwd, plus WORKSPACE.
 */
size_t attnres_step_host_workspace_bytes(const attnres_params* p, int64_t chunk_tokens);
attnres_status attnres_step_host(const attnres_params* p, const void* q, const void* w_o,
                                 const void* dy, int64_t dy_ld, void* y, int64_t y_ld,
                                 void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                 void* dw_o, float* dw_o_f32, int64_t chunk_tokens, void* workspace,
                                 size_t workspace_bytes, void* const* streams);

/*
 * Kernels bound every wait on a shared-memory barrier.  A wait that runs out
 * of time makes the kernel record a nonzero code here and finish without
 * further waiting (its outputs are then garbage); so does a selected-query
 * id outside [0, E) (that query then reads as zero and adds nothing to the
 * bank gradient), and, in a library built with -DATTNRES_DEBUG, a global
 * store of an output whose indices fall outside the call's sizes (skipped,
 * never made).  This call synchronises the device, returns
 * ATTNRES_ERR_DEVICE and clears the record if one was set, ATTNRES_OK
 * otherwise.
 */
attnres_status attnres_check_device_error(void);

/* Static description of a status code; never NULL. */
const char* attnres_status_string(attnres_status s);

/*
 * Launch plan the library would use for these params on the current device
 * (for tests and benchmarks; no launch happens).  Fills out[0..9] with:
 * backward CTAs, consumer warps (forward * 1000 + backward), 16-byte vectors
 * per thread (forward * 1000 + backward), the backward ring
 * (chunks * 1000 + rows per chunk), the forward ring (chunks * 1000 + rows
 * per chunk = softmax group), the backward resident flag (1 = a token's
 * source rows stay in shared memory for all backward passes), dynamic
 * shared memory bytes of the backward kernel, the backward reduction path
 * (0 = in-kernel, 1 = finalize kernel), the backward cluster size (CTAs
 * that share one token, each holding D / size columns of its rows; 1 = one
 * CTA per token) and the number of FP32 partial rows the finalize adds.
 */
attnres_status attnres_plan_info(const attnres_params* p, int64_t out[10]);

/*
 * Forward launches (single- and multi-query) of at least 1024 tokens run a
 * kernel compiled at run time (NVRTC) for the plan's exact shape -- the
 * source count, rows per chunk, softmax group rows and ring depth as
 * constants -- once per shape and device in a process; when NVRTC or the driver library cannot be opened, or
 * a compile fails, the precompiled kernels run instead.  ATTNRES_JIT=0 in
 * the environment turns the run-time path off.  This call returns how many
 * such kernels this process holds (a diagnostic; never fails).
 */
int attnres_jit_kernel_count(void);

/* ------------------------------------------------------------------------
 * Multi-query read ("Fast Attention Residuals", section "Multi-query
 * AttnRes"): the same sources are read with M queries q_m (bf16 [M][R],
 * 1 <= M <= ATTNRES_MAX_M); each query has its own routing weights and its
 * own full-width output,
 *
 *   z_ms = scale * r_s * <t_s, q_m>,  a_m = softmax_s(z_m),  y_m = sum_s a_ms v_s
 *
 * with the key slice t_s and its reciprocal RMS r_s exactly as above (r_s
 * does not depend on the query).  The multi-query read has no output norm.
 * Every source row is read from HBM once per call for all M outputs.  The
 * gradient of a source is the sum over queries; dq_m sums over tokens.
 *
 * The forward streams each token's rows once per block of queries it holds
 * in registers (one block for M <= 4 at D <= 2048, M <= 2 at D <= 4096;
 * later blocks re-read the token from L2), so any S and D are served.  The
 * backward has two forms, both serving every S, D and M the ABI accepts:
 *  - resident (up to two queries, when a token's S source rows, its M dy
 *    rows and the queries' key channels fit in shared memory): one kernel
 *    that reads each row once;
 *  - general (more queries, or tokens that do not fit): a coefficient kernel
 *    forms the per-token dots <dy_m, v_s> over blocks of columns with bf16
 *    tensor-core MMAs and writes every token's coefficients to the
 *    workspace, then a gradient kernel forms dvalues and dq block by block
 *    (on the tensor cores for nine or more fixed queries and at most 16
 *    sources); the sources and dy are read twice.
 * ATTNRES_MULTI_BWD=general or resident in the environment (read on every
 * call) forces one form where it fits; ATTNRES_MULTI_GRAD=mma or simt the
 * general form's gradient kernel.
 * ------------------------------------------------------------------------ */
#define ATTNRES_MAX_M 16

/*
 *   base        S, D, R, key_offset, N, eps, scale, src_ld, src as for
 *               attnres_params; base.out_norm must be 0; split_n_threshold
 *               is ignored (the multi-query backward always finalizes its
 *               per-CTA partial sums in a separate kernel, in CTA order).
 *   M           number of queries, 1 <= M <= ATTNRES_MAX_M
 *   out_ld_m    element stride between query m and m + 1 of one token, in
 *               the output y and in the upstream gradient dy
 *   out_ld_n    element stride between token n and n + 1 of one query
 *               (both multiples of 8).  Query-major [M, N, D]: out_ld_m =
 *               N * D, out_ld_n = D; token-major [N, M, D] (the page's
 *               output_layout="token_major"): out_ld_m = D, out_ld_n = M * D.
 */
typedef struct {
    attnres_params base;
    int32_t M;
    int64_t out_ld_m;
    int64_t out_ld_n;
} attnres_multi_params;

/*
 * Multi-query forward.  q bf16 [M][R] contiguous.  Outputs (fully
 * overwritten): y bf16 rows y + m * out_ld_m + n * out_ld_n (16-byte
 * aligned), alpha f32 [N][M][S], rstd f32 [N][S], logit f32 [N][M][S].
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (out_norm set, or the shape
 * does not fit), CUDA.
 */
attnres_status attnres_multi_fwd(const attnres_multi_params* p, const void* q, void* y,
                                 float* alpha, float* rstd, float* logit, void* stream);

/* Bytes of workspace attnres_multi_bwd needs (0 when N == 0): the per-CTA FP32
 * partial rows of dq, plus the general form's coefficient tables (N * S *
 * (2 * M rounded up to 8 + 4) floats). */
size_t attnres_multi_bwd_workspace_bytes(const attnres_multi_params* p);

/*
 * Multi-query backward.  Inputs: q, dy (bf16 rows at dy + m * out_ld_m +
 * n * out_ld_n, 16-byte aligned) and the forward's alpha, rstd, logit.
 * Outputs (written, never accumulated): dsrc[s] as for attnres_bwd (the
 * sum over all M queries), dq bf16 [M][R], dq_f32 f32 [M][R] (may be NULL).
 * workspace: at least attnres_multi_bwd_workspace_bytes(p) bytes, 16-byte
 * aligned.  Errors: as attnres_multi_fwd, plus WORKSPACE.
 */
attnres_status attnres_multi_bwd(const attnres_multi_params* p, const void* q, const void* dy,
                                 const float* alpha, const float* rstd, const float* logit,
                                 void* const* dsrc, int64_t dsrc_ld, void* dq, float* dq_f32,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Launch plan of the multi-query kernels (no launch).  out[0..9]: forward
 * CTAs * 1000 + backward CTAs, consumer warps (forward * 1000 + backward),
 * 16-byte vectors per thread (forward * 1000 + backward), queries per
 * register block (forward * 1000 + backward), forward ring (chunks * 1000 +
 * rows per chunk), backward ring (chunks * 1000 + rows per chunk), dy slots,
 * the backward dynamic shared memory bytes (of the gradient kernel in the
 * general form), the backward form (0 resident, 1 general, 2 general with
 * its gradient kernel on the tensor cores) and the general form's token
 * groups (0 otherwise).
 */
attnres_status attnres_multi_plan_info(const attnres_multi_params* p, int64_t out[10]);

/* ------------------------------------------------------------------------
 * Selected-query read ("Fast Attention Residuals", section "Multi-query
 * AttnRes": attnres_selected(sources, query_bank, ids) takes an [E, R] bank
 * and integer [..., K] ids and returns [..., K, D]).  Output (n, k) is the
 * single-query read of token n's sources with query bank[ids[n][k]]:
 *
 *   z_nks = scale * r_ns * <t_ns, bank[ids[n][k]]>,  a_nk = softmax_s(z_nk),
 *   y[n][k] = sum_s a_nks v_s[n]
 *
 * Gradients: dsrc sums over the K reads of each token; dbank[e] sums the
 * query gradients of every (n, k) with ids[n][k] == e (zero for rows no
 * token selects).  Same kernels, layouts and range as the multi-query read
 * with M = K slots per token.
 *   p        as for the multi-query read, M = K (1 <= K <= ATTNRES_MAX_M)
 *   bank     bf16 [E][R] contiguous, E >= 1
 *   ids      int64 [N][K] contiguous, 8-byte aligned; an id outside
 *            [0, E) is recorded for attnres_check_device_error and the
 *            slot reads as a zero query
 *   y, alpha, rstd, logit   as for attnres_multi_fwd (slot k in place of m)
 *   dbank    bf16 [E][R], dbank_f32 f32 [E][R] (may be NULL): written
 * ------------------------------------------------------------------------ */
attnres_status attnres_selected_fwd(const attnres_multi_params* p, const void* bank, int32_t E,
                                    const int64_t* ids, void* y, float* alpha, float* rstd,
                                    float* logit, void* stream);

/* Bytes of workspace attnres_selected_bwd needs (0 when N == 0): FP32
 * partial rows of dbank (E * R floats per CTA, or per token group in the
 * general form) plus, in the general form, the coefficient tables as for
 * attnres_multi_bwd_workspace_bytes. */
size_t attnres_selected_bwd_workspace_bytes(const attnres_multi_params* p, int32_t E);

attnres_status attnres_selected_bwd(const attnres_multi_params* p, const void* bank, int32_t E,
                                    const int64_t* ids, const void* dy, const float* alpha,
                                    const float* rstd, const float* logit, void* const* dsrc,
                                    int64_t dsrc_ld, void* dbank, float* dbank_f32, void* workspace,
                                    size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H_ */
