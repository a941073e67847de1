"""B300-native routing attention (Routing Transformer, shared-QK).

The compute lives in ``librouting_attention.so`` (hand-written sm_103a CUDA,
C ABI in ``include/routing_attention.h``); this package is its thin binding.
"""

from ._binding import (  # noqa: F401
    LIB_PATH,
    RoutingAttentionError,
    Workspace,
    load_library,
    rt_centroid_ema,
    rt_centroid_ema_apply,
    rt_centroid_ema_sums,
    rt_centroid_ema_topw,
    rt_debug_inject_wait_timeout,
    rt_launch_count,
    rt_local_attention,
    rt_mixed_attention,
    rt_profile_kernel_name,
    rt_profile_set,
    rt_route_assign,
    rt_route_assign_noalloc,
    rt_routing_attention,
    rt_routing_attention_backward,
    rt_routing_attention_separate,
    rt_routing_attention_step,
    rt_workspace_bytes,
)
