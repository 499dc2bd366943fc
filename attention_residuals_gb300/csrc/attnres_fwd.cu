// attnres_fwd.cu -- forward launches of the Attention Residuals read operator:
// the precompiled instances of the forward kernel (attnres_fwd_kernel.cuh),
// the run-time-compiled form for the plan's exact shape when available
// (attnres_jit.cu), and the error record.
#include "attnres_fwd_kernel.cuh"

namespace attnres {

namespace {

template <int VPT, bool FULL, bool FUSED, int NORM>
cudaError_t launch_fwd_t(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    auto kern = attnres_fwd_kernel<VPT, FULL, FUSED, NORM>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(plan.smem_fwd));
    if (err != cudaSuccess) return err;
    kern<<<plan.fgrid, (plan.ncw + 1) * 32, plan.smem_fwd, stream>>>(a);
    return cudaGetLastError();
}

template <int VPT, int NORM>
cudaError_t dispatch_key(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    if (a.delta) return launch_fwd_t<VPT, false, true, NORM>(plan, a, stream);  // the general column form
    const bool full = (a.D / 8) == VPT * 32 * plan.ncw;
    return full ? launch_fwd_t<VPT, true, false, NORM>(plan, a, stream)
                : launch_fwd_t<VPT, false, false, NORM>(plan, a, stream);
}

template <int VPT>
cudaError_t dispatch_norm(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    if (!a.out_norm) return dispatch_key<VPT, 0>(plan, a, stream);
    return a.o_pre ? dispatch_key<VPT, 2>(plan, a, stream) : dispatch_key<VPT, 1>(plan, a, stream);
}

}  // namespace

unsigned take_fwd_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fwd_error, sizeof v) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_fwd_error, &zero, sizeof zero);
    const unsigned j = take_jit_error(0);  // read (and cleared) either way
    return v ? v : j;
}

cudaError_t launch_fwd(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    if (a.N >= kJitMinTokens) {
        const cudaError_t e = jit_launch_fwd(plan, a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    switch (plan.vpt) {
        case 1: return dispatch_norm<1>(plan, a, stream);
        case 2: return dispatch_norm<2>(plan, a, stream);
        case 4: return dispatch_norm<4>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace attnres
