"""The C-ABI library loads and exports every entry point that include/moe.h declares.

Runs without a GPU: the library is loaded and inspected, no compute call is
made.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declarations():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for m in re.finditer(r"(?:moe_status|int|const char\s*\*)\s+(moe_\w+)\s*\(([^;]*?)\)\s*;", text, flags=re.S):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        decls[m.group(1)] = params
    return decls


@pytest.fixture(scope="module")
def lib():
    from sparse_moe_expert_top_gb300 import build, moe
    build.build()
    return moe.load()


def test_header_declares_the_path_entry_points():
    names = set(_declarations())
    for required in ("moe_route_topk", "moe_route_histogram", "moe_prefix_offsets", "moe_scatter_rows",
                     "moe_grouped_ffn", "moe_grouped_gate_up", "moe_grouped_down", "moe_combine", "moe_forward",
                     "moe_quantize_weights_fp8", "moe_grouped_ffn_fp8", "moe_forward_fp8", "moe_scatter_rows_f16",
                     "moe_route_scatter_small", "moe_router_topk", "moe_scatter_index",
                     "moe_grouped_gate_up_gather", "moe_grouped_down_combine", "moe_forward_fused",
                     "moe_tile_counts_size", "moe_route_scatter_small_fused",
                     "moe_workspace_size", "moe_check_device_error", "moe_clear_device_error",
                     "moe_forward_fused_mode", "moe_plan_create", "moe_plan_destroy", "moe_plan_grouped_gate_up",
                     "moe_plan_grouped_down", "moe_plan_forward", "moe_ffn_paired"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from sparse_moe_expert_top_gb300 import moe
    decls = _declarations()
    for name, params in decls.items():
        assert hasattr(lib, name), name
        # the binding's argument list has the header's arity
        assert name in moe.SIGNATURES, name
        assert len(moe.SIGNATURES[name][0]) == len(params), (name, params)
    assert set(moe.SIGNATURES) == set(decls)


def test_host_only_calls(lib):
    """Calls that need no device: version, status strings, workspace sizing, argument rejection."""
    assert lib.moe_version() >= 100
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(99) == b"unknown status"
    assert lib.moe_status_string(5) == b"a value out of the fp16 operand range"
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(2048, 6, ctypes.byref(n)) == 0
    # header (32 words) + 64 chunks of 32 tokens x 256 counts + 12288 ranks + 64 chunks of 256 bases, int32
    assert n.value == 4 * (32 + 64 * 256 + 2048 * 6 + 64 * 256)
    # beyond 256 chunks of 32 tokens the chunks grow: 8193 tokens -> 129 chunks of 64 tokens
    assert lib.moe_workspace_size(8193, 6, ctypes.byref(n)) == 0
    assert n.value == 4 * (32 + 129 * 256 + 8193 * 6 + 129 * 256)
    assert lib.moe_workspace_size(10, 17, ctypes.byref(n)) == 1      # k > 16
    assert lib.moe_workspace_size(-1, 2, ctypes.byref(n)) == 1       # T < 0
    # argument checks reject before touching the device
    assert lib.moe_route_topk(None, 4, 300, 2, None, None, None) == 1   # E > 256
    assert lib.moe_route_topk(None, 4, 8, 9, None, None, None) == 1     # k > E
    assert lib.moe_combine(None, None, None, 4, 2, 6, None, None) == 1  # d not a multiple of 4
    assert lib.moe_grouped_ffn(None, None, 8, 4, 100, 128, None, None, None, 1, None, None, None) == 1  # bf16 d % 128
    assert lib.moe_grouped_ffn(None, None, 8, 4, 128, 128, None, None, None, 7, None, None, None) == 2  # dtype
    assert lib.moe_quantize_weights_fp8(None, 1, 4, 24, None, None, None) == 1      # K not a multiple of 16
    assert lib.moe_quantize_weights_fp8(None, 9, 4, 32, None, None, None) == 2      # dtype
    assert lib.moe_grouped_gate_up_fp8(None, None, 8, 4, 100, 128, None, None, None, None, None, None) == 1
    assert lib.moe_scatter_rows_f16(None, None, None, None, 4, 17, 128, 8, None, None, None, None, None) == 1  # k
    assert lib.moe_route_scatter_small(None, None, 1, 0, None, 129, 8, 2, 64, None, None, None, None, None, None,
                                       None, None) == 1                                    # T > 128
    assert lib.moe_router_topk(None, None, 4, 8, 96, 2, None, None, None, None) == 1     # d % 64
    # fused permutation: one counter per token and 128-feature slice
    fake = ctypes.c_void_p(4096)
    assert lib.moe_tile_counts_size(2048, 4096, ctypes.byref(n)) == 0 and n.value == 2048 * 32 * 4
    assert lib.moe_tile_counts_size(3, 130, ctypes.byref(n)) == 0 and n.value == 3 * 2 * 4
    assert lib.moe_scatter_index(None, None, None, 4, 2, 6, 8, None, None, None, None, None, None, None,
                                 None) == 1                                                       # d % 8
    assert lib.moe_scatter_index(fake, fake, fake, 4, 2, 8, 8, fake, None, fake, fake, fake, fake, fake,
                                 None) == 1                                                       # x without xs
    assert lib.moe_grouped_gate_up_gather(None, 4, 2, None, None, 8, 100, 128, None, None, None, None) == 1  # d
    assert lib.moe_grouped_gate_up_gather(None, 4, 17, None, None, 8, 128, 128, None, None, None, None) == 1  # k
    assert lib.moe_route_scatter_small_fused(None, None, None, 129, 8, 2, 128, None, None, None, None, None, None,
                                             None, None, None, None) == 1                        # T > 128
    # y of the fused down projection must be 128-byte aligned (its L2 lines are dropped after use)
    bad_y = ctypes.c_void_p(4096 + 16)
    assert lib.moe_grouped_down_combine(fake, fake, 4, 2, 8, 128, 128, fake, fake, fake, fake, bad_y, fake, fake,
                                        None) == 1
    assert lib.moe_forward_fused(None, None, None, 4, 8, 2, 100, 128, None, None, None, 0, None, None, None,
                                 None, None, None, None, None, None, None, None, None, None) == 1  # d % 128
    assert lib.moe_forward_fused(None, None, None, 4, 8, 2, 128, 128, None, None, None, 2, None, None, None,
                                 fake, None, None, None, None, None, None, None, None, None) == 1  # compact, no xs
    assert lib.moe_forward_fused(None, None, None, 4, 8, 2, 128, 128, None, None, None, 7, None, None, None,
                                 fake, fake, None, None, None, None, None, None, None, None) == 1  # mode


def test_plan_entry_points_reject_bad_arguments(lib):
    """Plan creation checks its arguments before touching a device and leaves *plan NULL on failure."""
    fake = ctypes.c_void_p(4096)
    plan = ctypes.c_void_p(1234)
    args = [fake] * 13
    assert lib.moe_plan_create(0, 8, 2, 128, 128, 1, *args, ctypes.byref(plan)) == 1      # T = 0
    assert plan.value is None
    plan = ctypes.c_void_p(1234)
    assert lib.moe_plan_create(4, 8, 2, 100, 128, 1, *args, ctypes.byref(plan)) == 1      # bf16 d % 128
    assert plan.value is None
    assert lib.moe_plan_create(4, 8, 2, 128, 128, 7, *args, ctypes.byref(plan)) == 2      # dtype
    bad = list(args)
    bad[7] = None                                                                           # xs missing
    assert lib.moe_plan_create(4, 8, 2, 128, 128, 1, *bad, ctypes.byref(plan)) == 1
    assert lib.moe_plan_create(4, 8, 2, 128, 128, 1, *args, None) == 1                   # no handle
    assert lib.moe_plan_destroy(None) == 0
    assert lib.moe_plan_forward(None, fake, fake, None, fake, None) == 1
    assert lib.moe_plan_grouped_gate_up(None, None) == 1
    assert lib.moe_plan_grouped_down(None, None) == 1
    mode = ctypes.c_int(-1)
    assert lib.moe_forward_fused_mode(4, 300, 2, 128, 1, ctypes.byref(mode)) == 1          # E > 256
    assert lib.moe_forward_fused_mode(4, 8, 2, 128, 1, None) == 1
    paired = ctypes.c_int(-1)
    assert lib.moe_ffn_paired(12288, ctypes.byref(paired)) == 0 and paired.value == 0      # 2,048 tokens, top-6
    assert lib.moe_ffn_paired(49152, ctypes.byref(paired)) == 0 and paired.value == 1      # 8,192 tokens, top-6
    assert lib.moe_ffn_paired(-1, ctypes.byref(paired)) == 1
    assert lib.moe_ffn_paired(4, None) == 1


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_expert_top_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in src.lower().replace("oracle-free", ""), fn
