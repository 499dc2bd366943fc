// attnres_bwd_norm.cu -- backward kernels with the output RMSNorm, o rebuilt
// from the source rows (the kernel template is in attnres_bwd_kernel.cuh).
#include "attnres_bwd_kernel.cuh"

namespace attnres {

cudaError_t launch_bwd_norm_rebuild(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    return launch_bwd_mode<1>(plan, a, stream);
}

unsigned take_bwd_error_rebuild() { return take_unit_error(); }

}  // namespace attnres
