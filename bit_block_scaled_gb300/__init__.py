"""Fused Mixture-of-Experts layer with 4-bit block-scaled expert weights for
one GB300 (sm_103a): a C-ABI CUDA library (libmoe4, include/moe4.h) and its
thin Python binding. See ``_lib`` for the entry points."""
from ._lib import (ACT, FMT, LAYOUT, ROUTE, STATUS, Act, MoeError, QWeight, act,  # noqa: F401
                   load, moe_align_permute, moe_clear_status, moe_forward, moe_forward_host, moe_forward_profile, moe_forward_static,
                   moe_grouped_gemm1_act, moe_grouped_gemm2_weighted, moe_last_launch_count,
                   moe_padded_rows, moe_read_status, moe_route_topk, moe_status_string,
                   moe_unpermute_reduce, moe_workspace_size, qweight, moe_import_gptq_int4,
                   moe_import_modelopt_global_scale, moe_wait_selftest)
