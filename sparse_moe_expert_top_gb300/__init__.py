"""GB300-native grouped MoE prefill: CUDA kernels for sm_103a behind a C-ABI.

The C-ABI is declared in include/moe.h and implemented in csrc/; ``moe``
is its Python binding (same function names, marshalling only).
"""

from .moe import (MOE_BF16, MOE_F32, MoEBuffers, MoEError, load, moe_check_device_error, moe_combine, moe_forward,
                  moe_grouped_down, moe_grouped_ffn, moe_grouped_gate_up, moe_prefix_offsets, moe_route_histogram,
                  moe_route_topk, moe_scatter_rows, moe_version, moe_workspace_size)

__all__ = ["MOE_BF16", "MOE_F32", "MoEBuffers", "MoEError", "load", "moe_check_device_error", "moe_combine",
           "moe_forward", "moe_grouped_down", "moe_grouped_ffn", "moe_grouped_gate_up", "moe_prefix_offsets",
           "moe_route_histogram", "moe_route_topk", "moe_scatter_rows", "moe_version", "moe_workspace_size"]
