"""GB300 (sm_103a) MoE layer with top-k routing and one shared expert.

The C ABI (include/moe.h) is exposed under the same names by the ctypes
binding; `MoELayer` runs a whole forward/backward through it.  The binding is
loaded on first use: if the CUDA library has not been built, that use raises
ImportError (there is no CPU fallback)."""

_BINDING_NAMES = {
    "moe_route_topk", "moe_permute", "moe_permute_static", "moe_grouped_swiglu", "moe_unpermute_combine",
    "moe_unpermute_combine_bwd", "moe_grouped_swiglu_bwd", "moe_route_topk_bwd", "moe_permute_bwd",
    "moe_router_balance_loss", "moe_grouped_swiglu_recompute", "moe_selftest_group_maps", "moe_selftest_wait_timeout",
    "moe_workspace_size", "moe_version", "moe_device_status", "MoEError", "status_string",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    if name == "MoELayer":
        from .layer import MoELayer
        return MoELayer
    raise AttributeError(name)
