"""GB300-native routed-expert MoE layer (sm_103a CUDA kernels behind a C ABI).

Importing this package does not load the CUDA library; the first call does
(building it in-tree if needed).  There is no CPU path.
"""
from . import _lib
from ._lib import (MoEError, moe_cache_fetch, moe_cache_plan, moe_combine, moe_expert_down, moe_expert_gateup,
                   moe_expert_swiglu_cached, moe_grouped_swiglu, moe_permute, moe_rmsnorm, moe_route,
                   moe_route_noalloc, moe_route_recall, route_block_dedup)
from .layer import CachedMoELayer, MoELayer, MoEStack, PrefillRing, pack_layer_experts

__all__ = ["_lib", "MoEError", "MoELayer", "CachedMoELayer", "MoEStack", "PrefillRing", "pack_layer_experts",
           "moe_cache_plan", "moe_cache_fetch", "moe_expert_swiglu_cached", "moe_route", "moe_permute", "moe_expert_gateup", "moe_expert_down",
           "moe_grouped_swiglu", "moe_combine", "route_block_dedup", "moe_rmsnorm", "moe_route_noalloc",
           "moe_route_recall"]
