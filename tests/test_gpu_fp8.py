"""GPU parity of the FP8 E4M3 expert-weight path (quantizer, grouped FFN, whole path).

The quantizer's codes and scales must equal the oracle's bit for bit.  The
FFN with FP8 weights is compared with the oracle evaluated on the oracle's
own dequantized weights (scale * value(code), exact in float64), under the
tolerances of the bf16 path: the GPU widens the codes to fp16 exactly, takes
the bf16 token rows to fp16 exactly (in range), accumulates in fp32 and rounds
h to fp16; the oracle rounds nothing.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_f16_rounded, full_size_reference, to_np
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _oracle_quant(w):
    codes, scales = mo.quantize_weights_fp8(to_np(w).astype(np.float32))
    return codes, scales


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantizer_codes_and_scales_are_bit_exact(dtype):
    g = torch.Generator().manual_seed(5)
    E, rows, K = 3, 200, 1024
    w = torch.randn(E, rows, K, generator=g) * 0.02
    w[0, 0] = 0.0                                          # all-zero row: scale 1, codes 0
    w[0, 1] = -0.0
    w[0, 2, :] = 1e-5 * torch.randn(K, generator=g)        # small row: normal scale, full code range
    w[0, 2, 7] = 3e-3                                      # ... with one larger value
    w[1, 3, :] = torch.randn(K, generator=g) * 1e-6        # elements far below the row maximum ->
    w[1, 3, 0] = 1.0                                       # subnormal and zero codes
    # a row whose maximum is 448 has scale 1: its quotients are the weights
    # themselves, so RNE ties and the saturation edge are exercised exactly
    ties = torch.tensor([448.0, 1 + 1 / 16, 1.125 + 1 / 16, -(1 + 3 / 16), 2.0 ** -10, 3 * 2.0 ** -10,
                         240.0 + 8.0, -0.0, 2.0 ** -9, 0.75 * 2.0 ** -6])
    w[2, 4, :] = 0.0
    w[2, 4, :ties.numel()] = ties
    w = w.to(dtype)
    q = M.moe_quantize_weights_fp8(w.cuda())
    M.moe_check_device_error()
    codes, scales = _oracle_quant(w)
    assert np.array_equal(to_np(q.scales), scales)
    assert np.array_equal(to_np(q.codes), codes)


def test_quantizer_rejects_bad_shapes():
    w = torch.zeros(2, 4, 24, dtype=torch.bfloat16, device="cuda")   # K not a multiple of 16
    with pytest.raises(M.MoEError):
        M.moe_quantize_weights_fp8(w)


def _routing(T, E, k, seed, p_mask=0.0):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + 1.5 * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    return logits, mask


def _weights(E, d, f, seed):
    g = torch.Generator().manual_seed(seed)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return wg, wu, wd


FP8_CASES = [
    # E, d, f, T, k, p_mask
    (8, 256, 384, 300, 2, 0.0),
    (4, 128, 128, 77, 2, 0.2),
    (16, 512, 256, 600, 4, 0.1),
    (1, 128, 256, 200, 1, 0.0),
    (3, 384, 256, 150, 2, 0.0),    # d = 384: the down projection's last 256-feature item is half full
    (2, 128, 256, 700, 1, 0.0),    # one heavy expert: several 128-row slices
    (256, 256, 256, 4, 6, 0.0),    # a 4-token verification batch
]


@pytest.mark.parametrize("E,d,f,T,k,p", FP8_CASES)
def test_fp8_ffn_matches_oracle(E, d, f, T, k, p):
    logits, mask = _routing(T, E, k, seed=E * 17 + T, p_mask=p)
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, seed=d + 3 * f)
    qg, qu, qd = (M.moe_quantize_weights_fp8(w.cuda()) for w in (wg, wu, wd))
    bufs = M.MoEBuffers(T, E, k, d, f, torch.float16)
    for b in (bufs.xs, bufs.h, bufs.y):
        b.fill_(float("nan"))
    out = M.moe_forward_fp8(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), qg, qu, qd, k, bufs)
    M.moe_check_device_error()
    deq = [mo.dequantize_weights_fp8(*_oracle_quant(w)) for w in (wg, wu, wd)]
    ref = mo.moe_forward(logits.numpy(), to_np(x), tuple(deq), k, None if mask is None else mask.numpy())
    R = int(ref["offsets"][-1])
    assert np.array_equal(to_np(bufs.offsets), ref["offsets"])
    # the fp16 compact rows are the bf16 token rows rounded to fp16 (torch's
    # CPU cast is the reference rounding: exact except below 2^-17); unused rows are zero
    xs_ref = torch.from_numpy(ref["xs"]).to(torch.float16)
    assert torch.equal(bufs.xs[:R].cpu().view(torch.int16), xs_ref.view(torch.int16))
    assert torch.all(bufs.xs[R:] == 0)
    h_ref = mo.grouped_swiglu(ref["xs"], ref["offsets"], tuple(deq))
    assert_close_f16_rounded(bufs.h[:R], h_ref)
    # the down step against the oracle applied to the GPU's own h
    off = ref["offsets"]
    h_gpu = to_np(bufs.h[:R]).astype(np.float64)
    y_ref = np.zeros((R, d))
    for e in range(E):
        if off[e + 1] > off[e]:
            y_ref[off[e]:off[e + 1]] = mo.expert_down(h_gpu[off[e]:off[e + 1]], deq[2][e])
    assert_close(bufs.y[:R], y_ref, "bf16")
    assert_close(out, ref["out"], "bf16")
    assert torch.all(bufs.h[R:].float() == 0) and torch.all(bufs.y[R:] == 0)


def test_fp8_subnormal_codes_contribute():
    """Weights far below their row's maximum get subnormal E4M3 codes; the
    widening inside the SM must keep them (they alone drive this output)."""
    E, d, f, T, k = 1, 128, 128, 40, 1
    g = torch.Generator().manual_seed(11)
    # |w| / scale = 448 |w| stays mostly below 2^-6, the smallest normal E4M3
    wg = torch.randn(E, f, d, generator=g) * 1e-5
    wu = torch.randn(E, f, d, generator=g) * 1e-5
    wd = torch.randn(E, d, f, generator=g) * 1e-5
    for w in (wg, wu):
        w[:, :, 0] = 1.0            # row maximum on input feature 0 ...
    wd[:, :, 0] = 1.0
    wg, wu, wd = (w.to(torch.bfloat16) for w in (wg, wu, wd))
    x = torch.randn(T, d) * 1000.0  # large rows keep h well inside the fp16 range
    x[:, 0] = 0.0                   # ... which the inputs never use
    x = x.to(torch.bfloat16)
    codes, _ = _oracle_quant(wg)
    exp_field = (codes[0, :, 1:] >> 3) & 0xF
    assert (exp_field == 0).mean() > 0.5          # most codes used here are subnormal
    qg, qu, qd = (M.moe_quantize_weights_fp8(w.cuda()) for w in (wg, wu, wd))
    logits = torch.zeros(T, E)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.float16)
    M.moe_forward_fp8(logits.cuda(), x.cuda(), None, qg, qu, qd, k, bufs)
    M.moe_check_device_error()
    deq = [mo.dequantize_weights_fp8(*_oracle_quant(w)) for w in (wg, wu, wd)]
    h_ref = mo.grouped_swiglu(to_np(x).astype(np.float64), np.array([0, T]), tuple(deq))
    assert np.abs(h_ref).max() > 1e-3
    assert_close_f16_rounded(bufs.h[:T], h_ref)


def test_fp8_activation_beyond_fp16_range_is_reported():
    """A token row with |x| > 65504 cannot be an fp16 operand: MOE_ERR_RANGE, no fault."""
    E, d, f, T, k = 2, 128, 128, 8, 1
    wg, wu, wd = _weights(E, d, f, seed=2)
    qg, qu, qd = (M.moe_quantize_weights_fp8(w.cuda()) for w in (wg, wu, wd))
    x = torch.randn(T, d)
    x[3, 5] = 70000.0
    bufs = M.MoEBuffers(T, E, k, d, f, torch.float16)
    M.moe_forward_fp8(torch.randn(T, E).cuda(), x.to(torch.bfloat16).cuda(), None, qg, qu, qd, k, bufs)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_RANGE
    M.moe_check_device_error()   # the error word was cleared


def test_fp8_inconsistent_offsets_are_rejected_on_the_device():
    E, d, f, cap = 4, 128, 128, 32
    xs = torch.zeros(cap, d, dtype=torch.float16, device="cuda")
    w = torch.zeros(E, f, d, dtype=torch.bfloat16, device="cuda")
    q = M.moe_quantize_weights_fp8(w)
    offsets = torch.tensor([0, 10, 5, 20, 40], dtype=torch.int32, device="cuda")   # decreasing, > cap
    h = torch.empty(cap, f, dtype=torch.float16, device="cuda")
    M.moe_grouped_gate_up_fp8(xs, offsets, q, q, h)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    M.moe_check_device_error()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_t4", "prefill_t401", "prefill_t2048", "prefill_t8192"])
def test_fp8_full_size_workload(name):
    """Every FP8 code and scale of the bank bit for bit against the oracle's quantizer; h on every compact row
    within its fp16 rounding bound and out on every token within the bf16 tolerance, against the oracle on
    the values the codes stand for."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    qg, qu, qd = (M.moe_quantize_weights_fp8(inp[n]) for n in ("w_gate", "w_up", "w_down"))
    bufs = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.float16)
    bufs.h.fill_(float("nan"))
    out = M.moe_forward_fp8(inp["logits"], inp["x"], inp["mask"], qg, qu, qd, cfg.k, bufs)
    M.moe_check_device_error()
    checked = []

    def check_codes(e0, e1, banks):
        for q, ob in zip((qg, qu, qd), banks):
            assert np.array_equal(to_np(q.codes[e0:e1]), ob.codes)
            assert np.array_equal(to_np(q.scales[e0:e1]), ob.scales)
        checked.append((e0, e1))

    ref = full_size_reference(inp, fp8=True, check_codes=check_codes)
    assert checked, "the oracle visited no expert block"
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(bufs, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    assert_close_f16_rounded(bufs.h[:R], ref["h"])
    assert_close(out, ref["out"], "bf16")
