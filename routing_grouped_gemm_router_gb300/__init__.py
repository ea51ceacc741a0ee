"""GB300-native fused Mixture-of-Experts feed-forward layer.

The layer runs in ``libmoe_gb300.so`` (hand-written CUDA for sm_103a behind the C ABI of
``include/moe.h``). This package is the Python binding (``_lib``, same function names as
the C ABI) plus ``layer.MoELayer``, which owns the workspace and calls ``moe_forward``.
"""
from ._lib import (EXPORTED, MOE_BF16, MOE_F32, MOE_GEMM_DECODE_TC,  # noqa: F401
                   MOE_GEMM_INVALID, MOE_GEMM_PAIR_TC, MOE_GEMM_SIMT, MOE_GEMM_SMALL_BATCH,
                   MOE_ROUTE_SIGMOID_GROUPED,
                   MOE_ROUTE_SOFTMAX, MOE_WEIGHTS_FP8_E4M3_B128, MOE_WEIGHTS_NATIVE, MoeError,
                   make_config, moe_abi_version, moe_align, moe_align_noalloc,
                   moe_dequant_fp8_weights,
                   moe_align_workspace_size, moe_apply_expert_map, moe_block_m, moe_combine,
                   moe_combine_local, moe_config_t, moe_device_status, moe_expert_gemm1,
                   moe_expert_gemm1_gathered, moe_expert_gemm1_gathered_workspace_size,
                   moe_expert_gemm1_workspace_size, moe_expert_gemm2,
                   moe_expert_gemm2_workspace_size, moe_forward, moe_gather_rows, moe_gemm_kernel,
                   moe_grouped_swiglu, moe_grouped_swiglu_workspace_size, moe_masked_forward,
                   moe_masked_table, moe_masked_workspace_size, moe_max_padded_rows, moe_route,
                   moe_small_batch, moe_route_logits, moe_selftest_wait_timeout,
                   moe_workspace_layout, moe_workspace_size, status_string)
