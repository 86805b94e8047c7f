"""GPU tests of the plan object, the error-word clearing call and the fused-mode query (through the C-ABI).

A plan prepares the host side of moe_forward once (argument checks, device
lookup, the TMA tensor maps of the weights and compact buffers); its calls
must give moe_forward's results bit for bit, and those results must match
the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_bf16_rounded, to_np

pytestmark = pytest.mark.gpu


def _case(T, E, k, d, f, dtype, p_mask, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + torch.linspace(0, 1.5, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    x = torch.randn(T, d, generator=g).to(dtype)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(dtype)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(dtype)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(dtype)
    return logits, mask, x, wg, wu, wd


PLAN_CASES = [
    # T, E, k, d, f, dtype, p_mask
    (300, 8, 2, 256, 384, torch.bfloat16, 0.1),    # four routing launches
    (40, 16, 4, 256, 256, torch.bfloat16, 0.2),    # small chunk: routing in one launch
    (4, 64, 6, 256, 256, torch.bfloat16, 0.0),     # verification width: narrow items
    (700, 4, 2, 128, 256, torch.bfloat16, 0.0),    # heavy experts: big items
    (50, 5, 3, 96, 160, torch.float32, 0.3),       # fp32 SIMT path
]


@pytest.mark.parametrize("T,E,k,d,f,dtype,p", PLAN_CASES)
def test_plan_forward_equals_forward_and_matches_oracle(T, E, k, d, f, dtype, p):
    logits, mask, x, wg, wu, wd = _case(T, E, k, d, f, dtype, p, seed=T + E)
    dev = [t.cuda() if t is not None else None for t in (logits, mask, x, wg, wu, wd)]
    a = M.MoEBuffers(T, E, k, d, f, dtype)
    ref_gpu = M.moe_forward(dev[0], dev[2], dev[1], dev[3], dev[4], dev[5], k, a).clone()
    b = M.MoEBuffers(T, E, k, d, f, dtype)
    for t in (b.h, b.y, b.out):
        t.fill_(float("nan"))
    plan = M.moe_plan_create(dev[3], dev[4], dev[5], b)
    out = M.moe_plan_forward(plan, dev[0], dev[2], dev[1])
    M.moe_check_device_error()
    assert torch.equal(out.view(torch.int32), ref_gpu.view(torch.int32))
    for name in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    ref = mo.moe_forward(logits, x, (wg, wu, wd), k, mask)
    assert np.array_equal(to_np(b.ids), ref["ids"])
    R = int(ref["offsets"][-1])
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    if dtype == torch.bfloat16:
        assert_close_bf16_rounded(b.h[:R], ref["h"])
    assert_close(out, ref["out"], tol)
    # a second chunk through the same plan (new values, same buffers) is not served from the first
    logits2 = torch.randn(T, E, generator=torch.Generator().manual_seed(99))
    x2 = torch.randn(T, d, generator=torch.Generator().manual_seed(98)).to(dtype)
    out2 = M.moe_plan_forward(plan, logits2.cuda(), x2.cuda(), dev[1]).clone()
    ref2 = M.moe_forward(logits2.cuda(), x2.cuda(), dev[1], dev[3], dev[4], dev[5], k, a)
    M.moe_check_device_error()
    assert torch.equal(out2.view(torch.int32), ref2.view(torch.int32))
    plan.close()


def test_plan_ffn_steps_equal_the_plain_steps():
    T, E, k, d, f = 200, 8, 2, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, torch.bfloat16, 0.1, seed=7))
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    M.moe_forward(logits, x, mask, wg, wu, wd, k, b)
    h_ref, y_ref = b.h.clone(), b.y.clone()
    plan = M.moe_plan_create(wg, wu, wd, b)
    b.h.fill_(float("nan"))
    b.y.fill_(float("nan"))
    M.moe_plan_grouped_gate_up(plan)
    M.moe_plan_grouped_down(plan)
    M.moe_check_device_error()
    assert torch.equal(b.h.view(torch.int16), h_ref.view(torch.int16))
    assert torch.equal(b.y.view(torch.int32), y_ref.view(torch.int32))


def test_plan_replays_inside_a_cuda_graph():
    T, E, k, d, f = 4, 32, 6, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, torch.bfloat16, 0.0, seed=8))
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    plan = M.moe_plan_create(wg, wu, wd, b)
    ref = M.moe_plan_forward(plan, logits, x, mask).clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.moe_plan_forward(plan, logits, x, mask)
    b.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    M.moe_check_device_error()
    assert torch.equal(b.out.view(torch.int32), ref.view(torch.int32))


def test_clear_device_error_clears_without_a_check():
    """A bounded wait that runs out sets MOE_ERR_TIMEOUT; moe_clear_device_error clears it on the stream."""
    M.moe_selftest_bounded_wait(5)
    M.moe_clear_device_error()
    M.moe_check_device_error()           # nothing left to report
    M.moe_selftest_bounded_wait(5)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_TIMEOUT


@pytest.mark.parametrize("T,E,k,d", [(4, 256, 6, 4096), (401, 256, 6, 4096), (2048, 256, 6, 4096),
                                     (8192, 256, 6, 4096), (682, 256, 6, 4096), (683, 256, 6, 4096)])
def test_fused_mode_query_follows_the_documented_rule(T, E, k, d):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    cap = T * k
    expect = (M.MOE_FUSED_GATHER if cap <= 16 * E else
              M.MOE_FUSED_COMPACT if cap * d * 4 <= 2 * l2 else M.MOE_FUSED_NONE)
    assert M.moe_forward_fused_mode(T, E, k, d) == expect
    assert M.moe_forward_fused_mode(T, E, k, d, have_xs=False) == M.MOE_FUSED_GATHER
