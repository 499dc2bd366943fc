"""GB300-native (sm_103a) Attention Residuals read operator.

The hot path lives in libattnres_gb300.so (C ABI: include/attnres.h); this
package is its thin Python binding plus seeded workload generators.
"""
from .ops import (  # noqa: F401
    EPS_DEFAULT,
    attnres,
    attnres_block_read,
    attnres_bwd,
    attnres_bwd_noalloc,
    attnres_bwd_workspace_bytes,
    attnres_check_device_error,
    attnres_fwd,
    attnres_jit_kernel_count,
    attnres_multi,
    attnres_multi_bwd,
    attnres_multi_fwd,
    attnres_multi_plan_info,
    attnres_partial_bwd,
    attnres_partial_fwd,
    attnres_plan_info,
    attnres_selected,
    attnres_selected_bwd,
    attnres_selected_fwd,
    attnres_step_host,
)
