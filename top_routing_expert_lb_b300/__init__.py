"""B300-native forward pass of one top-k routed Mixture-of-Experts FFN layer.

The compute lives in ``libmoe_b300.so`` (CUDA C++ for sm_103a, C ABI in
``include/moe.h``); this package is its thin Python binding.  Importing the
package does not load the library; the first call does, and fails loudly if
the library has not been built.
"""
from ._binding import (  # noqa: F401
    MoeError, Shape, lib, moe_capacity, moe_check_status, moe_combine, moe_debug_timeout_probe,
    moe_error_string, moe_grouped_ffn, moe_layer_forward, moe_layer_forward_host,
    moe_layer_forward_host_batches, moe_max_rows,
    moe_pack_w13, moe_permute, moe_route, moe_set_wait_timeout_ns, moe_workspace_size,
    MoELayer, moe_profile_enable, moe_profile_collect, moe_launch_count, alloc_workspace,
    moe_route_noalloc, moe_route_ex, MOE_FLAG_SIGMOID, MOE_FLAG_NO_RENORM,
    moe_alf_bias_update, MOE_FLAG_PRIORITY_CAPACITY, MOE_FLAG_EXPERT_CHOICE, moe_ec_capacity,
    moe_ec_route, moe_ec_layer_forward, Tuning, MOE_TUNE_NO_HALF_TILES, MOE_TUNE_GEMM1_SPLIT,
    MOE_TUNE_FUSED_GATHER, MOE_TUNE_GATE_IN_EPILOGUE, MOE_TUNE_SWAP_ALL_TAILS, MOE_TUNE_TWO_CTAS_PER_SM,
    MOE_TUNE_NO_PDL,
)
