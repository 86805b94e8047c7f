"""GPU parity of the fused permutation: token rows gathered inside the gate/up
kernel (or copied by the index scatter, compact mode), the weighted combine
inside the down kernel (through the C-ABI).

Two bars.  The fused path's h and out equal the unfused path's bit for bit
(the same bf16 operands in the same swizzled shared-memory layout, the same
MMAs, the same fixed-order fp32 combine); and out is within the bf16
tolerance of the oracle.  Sizes span several weight tiles, compact slices
of up to 256 rows (both epilogue groups), narrow items, masked slots and
tokens whose slots are all masked.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import (BF16_REL_FRO, assert_close, assert_close_bf16_rounded, error_stats, full_size_reference,
                           to_np)
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _weights(E, d, f, seed):
    g = torch.Generator().manual_seed(seed)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return wg, wu, wd


def _routing(T, E, k, seed, p_mask=0.0, skew=1.5):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + skew * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    return logits, mask


GATHER, COMPACT, NONE = M.MOE_FUSED_GATHER, M.MOE_FUSED_COMPACT, M.MOE_FUSED_NONE


def _both_paths(logits, x, mask, wg, wu, wd, k, mode=M.MOE_FUSED_AUTO):
    """Runs the unfused and the fused path on the same inputs; returns both buffer sets."""
    T, E = logits.shape
    d, f = x.shape[1], wg.shape[1]
    args = (logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), wg.cuda(), wu.cuda(), wd.cuda(), k)
    a = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    for t in (b.h, b.y, b.out):
        t.fill_(float("nan"))
    b.tile_counts.fill_(7)          # stale counters: the index scatter clears them
    M.moe_forward(*args, a)
    M.moe_forward_fused(*args, b, mode=mode)
    M.moe_check_device_error()
    return a, b


def _assert_fused_equals_unfused(a, b):
    for name in ("ids", "w", "counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    R = int(a.offsets[-1])
    assert torch.equal(b.h[:R].view(torch.int16), a.h[:R].view(torch.int16))
    assert torch.all(b.h[R:].float() == 0)
    assert torch.equal(b.out.view(torch.int32), a.out.view(torch.int32))


FUSED_CASES = [
    # E, d, f, T, k, p_mask
    (8, 256, 384, 300, 2, 0.0),
    (4, 128, 128, 77, 2, 0.2),
    (16, 512, 256, 600, 4, 0.1),
    (1, 128, 256, 200, 1, 0.0),
    (3, 384, 256, 150, 2, 0.0),    # d = 384: the last down feature slice holds a single tile
    (16, 512, 384, 20, 4, 0.1),    # T*k <= 64: narrow items
    (256, 256, 256, 4, 6, 0.0),    # a 4-token verification batch
    (32, 256, 256, 150, 8, 0.1),   # k = 8: two slot groups in the combine warps
    (32, 128, 128, 70, 16, 0.2),   # k = 16 (the largest k)
]


@pytest.mark.parametrize("mode", [GATHER, COMPACT, NONE])
@pytest.mark.parametrize("E,d,f,T,k,p", FUSED_CASES)
def test_fused_path_equals_unfused_and_oracle(E, d, f, T, k, p, mode):
    logits, mask = _routing(T, E, k, seed=E * 7 + T, p_mask=p)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(T * 5 + d)).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=d * 3 + f)
    a, b = _both_paths(logits, x, mask, wg, wu, wd, k, mode)
    _assert_fused_equals_unfused(a, b)
    w = (to_np(wg), to_np(wu), to_np(wd))
    ref = mo.moe_forward(logits.numpy(), to_np(x), w, k, None if mask is None else mask.numpy())
    R = int(ref["offsets"][-1])
    h_ref = mo.grouped_swiglu(ref["xs"], ref["offsets"], w)
    assert_close_bf16_rounded(b.h[:R], h_ref)
    # down and combine against the oracle applied to the GPU's own h, so that h's
    # bf16 rounding is not counted twice; the whole path within the Frobenius bar
    y_ref = mo.grouped_down(b.h[:R].cpu(), ref["offsets"], w)
    assert_close(b.out, mo.combine(y_ref, ref["row_of_route"], ref["w"], T, k), "bf16")
    assert error_stats(b.out, ref["out"])["rel_fro"] <= BF16_REL_FRO


@pytest.mark.parametrize("mode", [GATHER, COMPACT])
def test_tokens_with_every_slot_masked_get_plus_zero(mode):
    """Half of the tokens have all slots masked: no down item reaches them, the index scatter zeroes them."""
    E, d, f, T, k = 8, 256, 256, 90, 3
    logits, _ = _routing(T, E, k, seed=11)
    mask = torch.zeros(T, k, dtype=torch.uint8)
    mask[::2] = 1
    mask[1::4, 1] = 1
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=12)
    a, b = _both_paths(logits, x, mask, wg, wu, wd, k, mode)
    _assert_fused_equals_unfused(a, b)
    assert torch.all(b.out[::2].view(torch.int32) == 0)
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k, mask.numpy())
    assert_close(b.out, ref["out"], "bf16")


@pytest.mark.parametrize("mode", [GATHER, COMPACT])
def test_every_slot_masked(mode):
    E, d, f, T, k = 4, 128, 128, 20, 2
    logits, _ = _routing(T, E, k, seed=5)
    mask = torch.ones(T, k, dtype=torch.uint8)
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=2)
    a, b = _both_paths(logits, x, mask, wg, wu, wd, k, mode)
    assert int(b.offsets[-1]) == 0
    assert torch.all(b.out.view(torch.int32) == 0)


@pytest.mark.parametrize("mode", [GATHER, COMPACT])
@pytest.mark.parametrize("d,f", [(256, 256), (384, 256)])
def test_big_items_with_both_epilogue_groups(d, f, mode):
    """Most rows go to two experts: 256-row slices, both down epilogue groups, up to 256 tokens per list."""
    E, T, k = 8, 700, 2
    g = torch.Generator().manual_seed(d + 1)
    logits = torch.randn(T, E, generator=g)
    logits[:, 6] += 3.0
    logits[:, 7] += 2.5
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=f + 1)
    a, b = _both_paths(logits, x, None, wg, wu, wd, k, mode)
    counts = to_np(a.counts)
    assert np.maximum(counts - 128, 0).sum() * 2 >= counts.sum()      # the big-item carve-up applies
    _assert_fused_equals_unfused(a, b)
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k)
    assert_close(b.out, ref["out"], "bf16")


def test_wide_ffn_many_rows_per_expert():
    """f = 4096 (32 gate/up feature tiles, K = 4096 for the down projection) with ~1000 rows per expert."""
    E, d, f, T, k = 8, 128, 4096, 4100, 2
    logits, mask = _routing(T, E, k, seed=3, p_mask=0.05)
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=4)
    a, b = _both_paths(logits, x, mask, wg, wu, wd, k)
    _assert_fused_equals_unfused(a, b)
    ref = mo.moe_forward(logits.numpy(), to_np(x), (wg, wu, wd), k, mask.numpy())
    assert np.array_equal(to_np(b.ids), ref["ids"])
    assert_close(b.out, ref["out"], "bf16")


@pytest.mark.parametrize("mode", [GATHER, COMPACT])
def test_fused_calls_step_by_step_and_repeated(mode):
    """The fused entry points called one by one give moe_forward_fused's output, twice over."""
    E, d, f, T, k = 16, 256, 256, 333, 3
    logits, mask = _routing(T, E, k, seed=8, p_mask=0.15)
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, seed=9))
    m = mask.cuda()
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    whole = M.moe_forward_fused(logits.cuda(), x, m, wg, wu, wd, k, b, mode=mode).clone()
    s = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    for _ in range(2):
        s.out.fill_(float("nan"))
        M.moe_route_topk(logits.cuda(), k, s.ids, s.w)
        M.moe_route_histogram(s.ids, m, E, s.counts, s.ws)
        M.moe_prefix_offsets(s.counts, T, k, s.offsets, s.ws)
        if mode == GATHER:
            M.moe_scatter_index(s.ids, m, s.offsets, d, s.row_of_route, s.route_of_row, s.tile_counts, s.out, s.ws)
            M.moe_grouped_gate_up_gather(x, k, s.route_of_row, s.offsets, wg, wu, s.h)
        else:
            M.moe_scatter_index(s.ids, m, s.offsets, d, s.row_of_route, s.route_of_row, s.tile_counts, s.out, s.ws,
                                x=x, xs=s.xs)
            M.moe_grouped_gate_up(s.xs, s.offsets, wg, wu, s.h)
        M.moe_grouped_down_combine(s.h, s.offsets, wd, s.route_of_row, s.row_of_route, s.w, s.y, s.tile_counts,
                                   s.out)
        M.moe_check_device_error()
        assert torch.equal(s.out.view(torch.int32), whole.view(torch.int32))


def test_gather_flags_routes_outside_the_chunk():
    """route_of_row entries outside [0, T*k) for rows below R: flagged, token 0 read instead, nothing faults."""
    E, d, f, T, k = 4, 128, 128, 16, 2
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, _ = (w.cuda() for w in _weights(E, d, f, seed=1))
    offsets = torch.tensor([0, 8, 16, 24, 32], dtype=torch.int32, device="cuda")
    route_of_row = torch.arange(T * k, dtype=torch.int32, device="cuda")
    route_of_row[5] = -1
    route_of_row[20] = T * k + 3
    h = torch.empty(T * k, f, dtype=torch.bfloat16, device="cuda")
    M.moe_grouped_gate_up_gather(x, k, route_of_row, offsets, wg, wu, h)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    M.moe_check_device_error()


def test_down_combine_skips_work_on_inconsistent_offsets():
    E, d, f, T, k = 4, 128, 128, 8, 2
    h = torch.zeros(T * k, f, dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros(E, d, f, dtype=torch.bfloat16, device="cuda")
    offsets = torch.tensor([0, 4, 8, 12, 40], dtype=torch.int32, device="cuda")
    rr = torch.arange(T * k, dtype=torch.int32, device="cuda")
    w = torch.ones(T, k, device="cuda")
    y = torch.zeros(T * k, d, device="cuda")
    counts = torch.zeros(M.moe_tile_counts_size(T, d) // 4, dtype=torch.int32, device="cuda")
    out = torch.full((T, d), 5.0, device="cuda")
    M.moe_grouped_down_combine(h, offsets, wd, rr, rr, w, y, counts, out)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    assert torch.all(out == 5.0) and torch.all(counts == 0)


# ---------------------------------------------------------------------------
# full-size workloads: equal to the unfused path bit for bit; every output
# checked against the oracle (index outputs bit for bit, h on every compact
# row, out on every token)
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name,mode", [("verify_t4", M.MOE_FUSED_AUTO), ("prefill_t401", M.MOE_FUSED_AUTO),
                                       ("prefill_t2048", M.MOE_FUSED_AUTO), ("prefill_t2048", GATHER),
                                       ("prefill_t8192", M.MOE_FUSED_AUTO), ("prefill_t8192", COMPACT)])
def test_full_size_workload_fused(name, mode):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    args = (inp["logits"], inp["x"], inp["mask"], inp["w_gate"], inp["w_up"], inp["w_down"], cfg.k)
    a = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.bfloat16)
    b = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.bfloat16)
    M.moe_forward(*args, a)
    b.out.fill_(float("nan"))
    out = M.moe_forward_fused(*args, b, mode=mode)
    M.moe_check_device_error()
    _assert_fused_equals_unfused(a, b)
    ref = full_size_reference(inp)
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(b, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    assert_close_bf16_rounded(b.h[:R], ref["h"])
    assert_close(out, ref["out"], "bf16")


@pytest.mark.parametrize("mode", [GATHER, COMPACT])
def test_small_chunk_fused_routing_step_by_step(mode):
    """moe_route_scatter_small_fused + the gate/up and fused down calls equal moe_forward_fused on a small chunk."""
    E, d, f, T, k = 32, 256, 256, 40, 6
    logits, mask = _routing(T, E, k, seed=31, p_mask=0.2)
    mask[3] = 1                                   # one token with every slot masked
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, seed=32))
    m = mask.cuda()
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    whole = M.moe_forward_fused(logits.cuda(), x, m, wg, wu, wd, k, b, mode=mode).clone()
    s = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    s.out.fill_(float("nan"))
    s.tile_counts.fill_(3)
    M.moe_route_scatter_small_fused(logits.cuda(), x, m, k, s, gather=(mode == GATHER))
    if mode == GATHER:
        M.moe_grouped_gate_up_gather(x, k, s.route_of_row, s.offsets, wg, wu, s.h)
    else:
        M.moe_grouped_gate_up(s.xs, s.offsets, wg, wu, s.h)
    M.moe_grouped_down_combine(s.h, s.offsets, wd, s.route_of_row, s.row_of_route, s.w, s.y, s.tile_counts, s.out)
    M.moe_check_device_error()
    assert torch.equal(s.out.view(torch.int32), whole.view(torch.int32))
    assert torch.all(s.out[3].view(torch.int32) == 0)
    a = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    M.moe_forward(logits.cuda(), x, m, wg, wu, wd, k, a)
    assert torch.equal(a.out.view(torch.int32), whole.view(torch.int32))


@pytest.mark.parametrize("fused", [False, True])
def test_whole_path_is_capturable_in_a_cuda_graph(fused):
    """No allocation, synchronisation or host read inside the path: a CUDA graph of one call replays it."""
    E, d, f, T, k = 16, 256, 256, 300, 4
    logits, mask = _routing(T, E, k, seed=41, p_mask=0.1)
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, seed=42))
    args = (logits.cuda(), x, mask.cuda(), wg, wu, wd, k)
    fwd = M.moe_forward_fused if fused else M.moe_forward
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref = fwd(*args, b).clone()            # warm-up call off the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd(*args, b)
    b.out.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    M.moe_check_device_error()
    assert torch.equal(b.out.view(torch.int32), ref.view(torch.int32))
