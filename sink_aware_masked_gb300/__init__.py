"""GB300-native exact sink-aware attention (forward and backward).

The computation runs in hand-written CUDA kernels for sm_103a, exported
through the C ABI in include/sinkattn.h (libsinkattn.so, built in-tree by
``sink_aware_masked_gb300.build``).  This package is the thin PyTorch
binding of that ABI.
"""
from .api import (  # noqa: F401
    WINDOW_INF,
    SinkAttention,
    bwd_workspace_bytes,
    decode_workspace_bytes,
    grpo_loss,
    grpo_workspace_bytes,
    kernel_launches,
    make_problem,
    sink_attention,
    sinkattn_bwd,
    sinkattn_decode_fwd,
    sinkattn_fwd,
    sinkattn_get_device_status,
    PROFILE_BWD_MAIN,
    PROFILE_DECODE,
    PROFILE_FWD,
    sinkattn_pack,
    sinkattn_set_profile_events,
    sinkattn_unpack,
    sinkattn_varlen_plan,
)
