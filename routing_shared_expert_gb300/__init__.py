"""GB300-native forward (and backward) pass of a routed + shared-expert MoE layer.

The compute path is the CUDA library ``libmoe_gb300.so`` (C ABI in
``include/moe_gb300.h``); this package is its thin Python binding.  Importing it
requires the built library: there is no CPU fallback.
"""
from ._native import (  # noqa: F401
    STATS, MoEError, alloc_workspace, copy_config, library, make_config, make_outputs, make_weights,
    moe_balance_stats, moe_bias_update, moe_combine,
    moe_grouped_swiglu, moe_layer_forward, moe_layer_forward_profiled, moe_merge_shared,
    moe_pack_weights, moe_packed_weights_size, pack_weights, moe_permute, moe_permute_noalloc,
    moe_read_status, moe_check_wait_bound, moe_backward_workspace_size, moe_layer_backward, make_grads,
    moe_route, moe_shared_mlp, moe_workspace_init, moe_workspace_size, version)
from .layer import STAGES, MoELayer, config_from_spec  # noqa: F401
