"""GB300-native (sm_103a) Mixture-of-Experts grouped (ragged) GEMM.

The computation lives in ``lib/libgg.so`` (C ABI in ``include/gg.h``); this
package only loads it (``_lib``), marshals torch tensors into it (``api``)
and provides seeded synthetic inputs (``synth``).
"""
from . import api  # noqa: F401
from ._lib import GGError  # noqa: F401
from .api import (backward_dW, backward_dX, backward_dX_swiglu, dual_asym, forward,  # noqa: F401
                  forward_combine, forward_swiglu, permute, read_status, route_hist_offsets,
                  route_workspace_size, set_gemm_schedule, swiglu_bwd, unpermute_combine,
                  unpermute_combine_bwd, workspace_size)

__all__ = ["route_hist_offsets", "route_workspace_size", "permute", "unpermute_combine", "forward",
           "backward_dX", "backward_dW", "dual_asym", "unpermute_combine_bwd",
           "forward_swiglu", "swiglu_bwd", "forward_combine", "backward_dX_swiglu", "workspace_size",
           "read_status", "set_gemm_schedule"]
