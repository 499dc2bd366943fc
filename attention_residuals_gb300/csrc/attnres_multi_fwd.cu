// attnres_multi_fwd.cu -- multi-query forward launches: the precompiled
// instances of the kernel (attnres_multi_fwd_kernel.cuh), the run-time
// compiled form for the plan's exact shape when available (attnres_jit.cu),
// and the error record.
#include "attnres_multi_fwd_kernel.cuh"

namespace attnres {

namespace {

template <int VPT, int MB, bool SEL, int MQ>
cudaError_t launch_t(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_multi_fwd_kernel<VPT, MB, SEL, MQ>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_fwd));
    if (err != cudaSuccess) return err;
    kern<<<plan.fgrid, (plan.ncw + 1) * 32, plan.smem_fwd, stream>>>(a);
    return cudaGetLastError();
}

template <int VPT, int MB, bool SEL, int MQ>
int occupancy_t(const MultiPlan& plan) {
    auto kern = attnres_multi_fwd_kernel<VPT, MB, SEL, MQ>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(plan.smem_fwd)) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (plan.ncw + 1) * 32, plan.smem_fwd) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

unsigned take_multi_fwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_multi_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_multi_error, &zero, sizeof zero);
    const unsigned j = take_jit_error(1);  // read (and cleared) either way
    return v ? v : j;
}

namespace {
// One (VPT, MB) pair per plan; with a fixed query count only the block size
// the planner derives from it (multi_fwd_mb) is instantiated.
template <int VPT, int MB, bool SEL, int MQ>
constexpr bool fwd_reachable() {
    return MQ == 0 || MB == multi_fwd_mb(MQ, VPT);
}

template <bool SEL, int MQ>
int fwd_occupancy_mq(const MultiPlan& plan) {
#define ATTNRES_OCC(V, B)                                                        \
    case V * 10 + B:                                                             \
        if constexpr (fwd_reachable<V, B, SEL, MQ>()) return occupancy_t<V, B, SEL, MQ>(plan); \
        return 0;
    switch (plan.vpt * 10 + plan.mb_f) {
        ATTNRES_OCC(1, 1)
        ATTNRES_OCC(1, 2)
        ATTNRES_OCC(1, 4)
        ATTNRES_OCC(2, 1)
        ATTNRES_OCC(2, 2)
        ATTNRES_OCC(4, 1)
        default: return 0;
    }
#undef ATTNRES_OCC
}

template <bool SEL, int MQ>
cudaError_t launch_fwd_mq(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
#define ATTNRES_LAUNCH(V, B)                                                                  \
    case V * 10 + B:                                                                          \
        if constexpr (fwd_reachable<V, B, SEL, MQ>()) return launch_t<V, B, SEL, MQ>(plan, a, stream); \
        return cudaErrorInvalidConfiguration;
    switch (plan.vpt * 10 + plan.mb_f) {
        ATTNRES_LAUNCH(1, 1)
        ATTNRES_LAUNCH(1, 2)
        ATTNRES_LAUNCH(1, 4)
        ATTNRES_LAUNCH(2, 1)
        ATTNRES_LAUNCH(2, 2)
        ATTNRES_LAUNCH(4, 1)
        default: return cudaErrorInvalidConfiguration;
    }
#undef ATTNRES_LAUNCH
}

template <bool SEL>
int fwd_occupancy_sel(const MultiPlan& plan) {
    switch (plan.mq) {
        case 1: return fwd_occupancy_mq<SEL, 1>(plan);
        case 2: return fwd_occupancy_mq<SEL, 2>(plan);
        case 4: return fwd_occupancy_mq<SEL, 4>(plan);
        default: return fwd_occupancy_mq<SEL, 0>(plan);
    }
}

template <bool SEL>
cudaError_t launch_fwd_sel(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    switch (plan.mq) {
        case 1: return launch_fwd_mq<SEL, 1>(plan, a, stream);
        case 2: return launch_fwd_mq<SEL, 2>(plan, a, stream);
        case 4: return launch_fwd_mq<SEL, 4>(plan, a, stream);
        default: return launch_fwd_mq<SEL, 0>(plan, a, stream);
    }
}
}  // namespace

// plan.E > 0: the selected-query kernels (a query bank and per-token ids)
int multi_fwd_occupancy(const MultiPlan& plan) {
    return plan.E > 0 ? fwd_occupancy_sel<true>(plan) : fwd_occupancy_sel<false>(plan);
}

cudaError_t launch_multi_fwd(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    if (a.N >= kJitMinTokens) {
        const cudaError_t e = jit_launch_multi_fwd(plan, a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    return a.ids ? launch_fwd_sel<true>(plan, a, stream) : launch_fwd_sel<false>(plan, a, stream);
}

}  // namespace attnres
