/*
 * attnres_testing.h -- hooks the library's own tests use to exercise paths
 * that ordinary inputs never reach.  Not part of the operator's interface.
 */
#ifndef ATTNRES_TESTING_H_
#define ATTNRES_TESTING_H_

#include <stdint.h>

#include "attnres.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The forward (attnres_fwd, same arguments, output norm optional) with the
 * bounded-wait recovery path forced: the producer warp of CTA 0 never issues
 * its withhold_fill-th chunk fill (1-based; every earlier fill is issued and
 * consumed as usual, so no copy is in flight when the CTA finishes) and
 * stops, and every wait of the launch gives up after wait_us microseconds
 * instead of about two seconds.  CTA 0's consumers therefore time out
 * waiting for that fill, record the wait site and run to the end without
 * waiting again; the launch finishes, attnres_check_device_error() then
 * reports ATTNRES_ERR_DEVICE (and clears the record), the outputs of CTA 0's
 * tokens are garbage, and the next ordinary launch is unaffected.  This is
 * no device fault: nothing is read or written out of bounds and every wait
 * ends.  withhold_fill must be >= 1; wait_us 1 .. 1000000.
 */
attnres_status attnres_fwd_withhold_for_test(const attnres_params* p, const void* q, const void* w_o,
                                             void* y, float* alpha, float* rstd, float* logit,
                                             float* o_rstd, int64_t withhold_fill, uint32_t wait_us,
                                             void* stream);

/*
 * Which form a multi-query (E = 0) or selected-query (E = bank rows) forward
 * of these params runs: 1 the tensor-core form, 0 the other, -1 invalid
 * params or no device.  ATTNRES_MULTI_FWD=mma / simt in the environment
 * forces the choice where the shape allows it.
 */
int attnres_multi_fwd_tensor_cores(const attnres_multi_params* p, int32_t E);

/*
 * 1 when the library was compiled with -DATTNRES_DEBUG (python -m
 * attention_residuals_gb300.build --debug writes it beside the release
 * build as libattnres_gb300_debug.so), else 0.  In that build every kernel
 * checks each global store of an output (y, o_pre, the block partial sum,
 * every source gradient row, the single-query FP32 partial rows of dq and
 * dw_o) against the call's sizes before it is made; a store that would fall
 * outside them is skipped and recorded for attnres_check_device_error(),
 * never trapped.
 */
int attnres_debug_checks(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_TESTING_H_ */
