"""deterministic_rl_gb300 -- a deterministic, batch-invariant MoE layer forward
with router replay for GB300 (sm_103a).

The computation lives in the CUDA library libmoedet.so (C ABI in
include/moe_det.h); ``binding`` marshals torch tensors into it, ``layer``
wraps it for convenience, ``synthetic`` draws seeded workloads.
"""
from . import binding  # noqa: F401
from .binding import (MoEError, moe_forward, moe_forward_replay, moe_get_status,  # noqa: F401
                      moe_route, moe_status_str, moe_workspace_layout, moe_workspace_size)
from .layer import MoELayer  # noqa: F401
