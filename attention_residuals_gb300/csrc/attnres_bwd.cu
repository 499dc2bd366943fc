// attnres_bwd.cu -- backward launches of the Attention Residuals read
// operator: the kernels without the output norm (the run-time mode form;
// the norm modes are instantiated in attnres_bwd_norm.cu and
// attnres_bwd_opre.cu), the finalize launch, the mode dispatch and the error
// record.
#include "attnres_bwd_kernel.cuh"

namespace attnres {

cudaError_t launch_finalize(const float* part, int P, int R, int W, uint16_t* dq, float* dq_f32,
                            uint16_t* dw_o, float* dw_o_f32, cudaStream_t stream) {
    return launch_pdl(attnres_finalize_kernel, dim3((W + kFinCols - 1) / kFinCols), dim3(kFinCols * kFinSlices), 0,
                      stream, part, P, R, W, dq, dq_f32, dw_o, dw_o_f32);
}

unsigned take_bwd_error() {
    // every unit's record is read (and cleared); the first nonzero one is reported
    const unsigned e0 = take_unit_error();
    const unsigned e1 = take_bwd_error_rebuild();
    const unsigned e2 = take_bwd_error_saved();
    const unsigned e3 = take_bwd_error_cluster();
    return e0 ? e0 : (e1 ? e1 : (e2 ? e2 : e3));
}

cudaError_t launch_bwd(const Plan& plan, const BwdArgs& a, cudaStream_t stream) {
    if (plan.cl > 1) return launch_bwd_cluster(plan, a, stream);
    if (!a.out_norm) return launch_bwd_mode<-1>(plan, a, stream);
    return a.o_pre ? launch_bwd_norm_saved(plan, a, stream) : launch_bwd_norm_rebuild(plan, a, stream);
}

}  // namespace attnres
