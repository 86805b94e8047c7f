"""GPU parity of the paired-SM grouped FFN (clusters of two CTAs, M = 256 MMAs).

Chunks of many routes run the bf16 and E4M3 projections on pairs of SMs.
The cases below have enough routes to take that path (checked through
moe_ffn_paired) and small d and f, so that the oracle finishes in about a
second; they span heavy experts cut into several 256-row slices with ragged
tails, light experts (slices of 32 rows or fewer, the accumulator slots
alternating), empty experts, feature counts that leave the odd CTA's tile of
the last item outside the matrix (f or d = 128 mod 256 or mod 512), and
masked slots.  The full-size 8,192-token chunk takes the same path in
test_gpu_ffn, test_gpu_fused, test_gpu_plan and test_gpu_w8a8.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import BF16_REL_FRO, assert_close, assert_close_bf16_rounded, error_stats, to_np

pytestmark = pytest.mark.gpu


def _case(T, E, k, d, f, p_mask, seed, dead=0, heavy=()):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + 1.5 * torch.linspace(0, 1, E)[None, :]
    for e in range(dead):
        logits[:, e] = -50.0            # experts nobody routes to
    for e, b in heavy:
        logits[:, e] += b
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return logits, mask, x, wg, wu, wd


PAIR_CASES = [
    # T, E, k, d, f, p_mask, dead experts, heavy experts (id, logit bias)
    (4200, 16, 6, 256, 256, 0.1, 0, ()),                  # ~1,400 rows per expert: many 256-row slices
    (4100, 64, 6, 384, 384, 0.0, 2, ()),                  # f, d = 128 mod 256: the odd CTA's last tiles unused
    (3100, 256, 8, 128, 128, 0.2, 8, ()),                 # ~90 rows per expert: light items only
    (4096, 32, 6, 256, 512, 0.05, 4, ((30, 4.0), (31, 3.5))),   # two experts with ~4,000 rows each
]


@pytest.mark.parametrize("T,E,k,d,f,p,dead,heavy", PAIR_CASES)
def test_pair_ffn_matches_oracle(T, E, k, d, f, p, dead, heavy):
    assert M.moe_ffn_paired(T * k)
    logits, mask, x, wg, wu, wd = _case(T, E, k, d, f, p, seed=T + E, dead=dead, heavy=heavy)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    for b in (bufs.h, bufs.y):
        b.fill_(float("nan"))
    out = M.moe_forward(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), wg.cuda(), wu.cuda(),
                        wd.cuda(), k, bufs)
    M.moe_check_device_error()
    w = (to_np(wg), to_np(wu), to_np(wd))
    ref = mo.moe_forward(logits.numpy(), to_np(x), w, k, None if mask is None else mask.numpy())
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(bufs, key)), ref[key]), key
    counts = ref["counts"]
    if dead:
        assert np.all(counts[:dead] == 0)
    R = int(ref["offsets"][-1])
    assert_close_bf16_rounded(bufs.h[:R], ref["h"])
    # the down step and the combine against the oracle applied to the GPU's own h
    y_ref = mo.grouped_down(bufs.h[:R].cpu(), ref["offsets"], w)
    assert_close(bufs.y[:R], y_ref, "bf16")
    assert_close(out, mo.combine(y_ref, ref["row_of_route"], ref["w"], T, k), "bf16")
    # the whole path against the oracle: within the Frobenius bar here; with
    # k = 8 slots of f = 128 the bf16 rounding of h alone moves the largest
    # outputs (10 x rms) by up to ~2.2 % of rms, past the max-element bar
    st = error_stats(out, ref["out"])
    assert st["rel_fro"] <= BF16_REL_FRO, st
    if k <= 6:
        assert_close(out, ref["out"], "bf16")
    assert torch.all(bufs.h[R:].float() == 0) and torch.all(bufs.y[R:] == 0)


def test_pair_steps_repeat_bit_for_bit():
    """Two runs of the paired projections on the same inputs give the same bytes (fixed accumulation order)."""
    T, E, k, d, f = 4200, 16, 6, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, 0.1, seed=9))
    a = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    b = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    M.moe_forward(logits, x, mask, wg, wu, wd, k, a)
    M.moe_forward(logits, x, mask, wg, wu, wd, k, b)
    M.moe_check_device_error()
    assert torch.equal(a.h.view(torch.int16), b.h.view(torch.int16))
    assert torch.equal(a.out.view(torch.int32), b.out.view(torch.int32))


W8A8_PAIR_CASES = [
    (4200, 16, 6, 256, 256, 0.1, 0, ()),
    (3100, 256, 8, 128, 384, 0.0, 4, ()),
    (4096, 32, 6, 384, 256, 0.05, 2, ((31, 4.0),)),
]


@pytest.mark.parametrize("T,E,k,d,f,p,dead,heavy", W8A8_PAIR_CASES)
def test_pair_w8a8_matches_oracle(T, E, k, d, f, p, dead, heavy):
    assert M.moe_ffn_paired(T * k)
    logits, mask, x, wg, wu, wd = _case(T, E, k, d, f, p, seed=T * 3 + E, dead=dead, heavy=heavy)
    q = [M.moe_quantize_weights_fp8(t.cuda()) for t in (wg, wu, wd)]
    b = M.MoEBuffersW8A8(T, E, k, d, f)
    for t in (b.h, b.y, b.out):
        t.fill_(float("nan"))
    out = M.moe_forward_w8a8(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), *q, k, b)
    M.moe_check_device_error()
    qo = tuple(mo.quantize_bank_fp8(t) for t in (wg, wu, wd))
    R = int(b.offsets[-1])
    ref = mo.moe_forward_w8a8(logits, x, qo, k, mask, h_decided=b.h[:R].cpu())
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(b, key)), ref[key]), key
    assert_close_bf16_rounded(b.h[:R], ref["h"])
    hq = mo.quantize_bank_fp8(b.h[:R].cpu())
    assert np.array_equal(to_np(b.h_q[:R]), hq.codes)
    y_ref = mo.grouped_down(mo.dequantize_weights_fp8(hq.codes, hq.scales), ref["offsets"], qo)
    assert_close(b.y[:R], y_ref, "bf16")
    assert torch.all(b.y[R:] == 0)
    assert_close(out, ref["out"], "bf16")


def test_pair_kernels_reject_inconsistent_offsets():
    """offsets[E] beyond the capacity: both paired kernels skip their work and flag it; nothing hangs."""
    E, d, f, cap = 4, 128, 128, 24576
    assert M.moe_ffn_paired(cap)
    xs = torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros(E, f, d, dtype=torch.bfloat16, device="cuda")
    h = torch.zeros(cap, f, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(cap, d, dtype=torch.float32, device="cuda")
    offsets = torch.tensor([0, 4000, 8000, 12000, cap + 100], dtype=torch.int32, device="cuda")
    M.moe_grouped_ffn(xs, offsets, wg, wg, wg.transpose(1, 2).contiguous(), h, y)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    M.moe_check_device_error()  # the error word was cleared


@pytest.mark.slow
def test_pair_many_heavy_groups():
    """Every expert heavy and seven 256-feature tiles of gate/up each: 1,792 heavy groups, more than the
    shared block-start table of the dynamic hand-out holds, so the decode computes the block starts itself."""
    T, E, k, d, f = 16384, 256, 6, 128, 1792
    assert M.moe_ffn_paired(T * k)
    g = torch.Generator().manual_seed(77)
    logits = torch.randn(T, E, generator=g)          # uniform routing: ~384 rows per expert
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    out = M.moe_forward(logits.cuda(), x.cuda(), None, wg.cuda(), wu.cuda(), wd.cuda(), k, bufs)
    M.moe_check_device_error()
    w = (to_np(wg), to_np(wu), to_np(wd))
    ref = mo.moe_forward(logits.numpy(), to_np(x), w, k, None)
    counts = ref["counts"]
    assert counts.min() > 256            # every expert has more than one 256-row slice
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(bufs, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    assert_close_bf16_rounded(bufs.h[:R], ref["h"])
    y_ref = mo.grouped_down(bufs.h[:R].cpu(), ref["offsets"], w)
    assert_close(bufs.y[:R], y_ref, "bf16")
    assert_close(out, mo.combine(y_ref, ref["row_of_route"], ref["w"], T, k), "bf16")
