// attnres_bwd_opre.cu -- backward kernels with the output RMSNorm and the
// caller's FP32 o (the kernel template is in attnres_bwd_kernel.cuh).
#include "attnres_bwd_kernel.cuh"

namespace attnres {

cudaError_t launch_bwd_norm_saved(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    return launch_bwd_mode<2>(plan, a, stream);
}

unsigned take_bwd_error_saved() { return take_unit_error(); }

}  // namespace attnres
