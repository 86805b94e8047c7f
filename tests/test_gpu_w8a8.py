"""GPU parity of the FP8-activation path: E4M3 weights and activations on kind::f8f6f4 tensor cores.

Every quantized operand is compared bit for bit with the oracle's quantizer:
the codes and scales of the token rows, of the compact rows (their scatter)
and of h (the quantizer applied to the GPU's own bf16 h).  h is compared with
the oracle's h within its bf16 rounding bound, y with the oracle's down
projection of the GPU's quantized h (the GPU accumulates the same E4M3
products in fp32), and out with the oracle's whole FP8-activation path within
the bf16 tolerance.  The E4M3 codes of h are decided from the kernel's bf16 h
on both sides (a quantization decision taken in the kernel's precision); the
kernel's h itself is checked against the oracle's h.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_bf16_rounded, to_np
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _case(T, E, k, d, f, p_mask, seed, skew=1.5):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + skew * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return logits, mask, x, wg, wu, wd


def _gpu_h(b):
    """The kernel's bf16 h of the R used compact rows (on the host)."""
    R = int(b.offsets[-1])
    return b.h[:R].cpu()


def _check_against_oracle(b, ref, q_gpu, k, d):
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(b, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    # the token rows' codes and scales are the oracle quantizer's
    assert np.array_equal(to_np(b.x_q), ref["x_q"].codes)
    assert np.array_equal(to_np(b.x_scales), ref["x_q"].scales)
    # compact rows: the scattered codes and scales
    tok = ref["route_of_row"][:R] // k
    assert np.array_equal(to_np(b.xs[:R]), ref["x_q"].codes[tok])
    assert np.array_equal(to_np(b.xs_scales[:R]), ref["x_q"].scales[tok])
    assert torch.all(b.xs[R:] == 0)
    # h against the oracle's h, within its bf16 rounding
    assert_close_bf16_rounded(b.h[:R], ref["h"])
    # h's codes and scales: the oracle quantizer applied to the GPU's own bf16 h
    hq = mo.quantize_bank_fp8(b.h[:R].cpu())
    assert np.array_equal(to_np(b.h_q[:R]), hq.codes)
    assert np.array_equal(to_np(b.h_scales[:R]), hq.scales)
    return R, hq


W8A8_CASES = [
    # T, E, k, d, f, p_mask
    (300, 8, 2, 256, 384, 0.0),
    (77, 4, 2, 128, 128, 0.2),
    (600, 16, 4, 512, 256, 0.1),
    (200, 1, 1, 128, 256, 0.0),
    (150, 3, 2, 384, 256, 0.0),     # d = 384: the last down feature pair is half a pair
    (20, 16, 4, 512, 512, 0.1),     # 80 routes: normal items
    (12, 16, 4, 512, 512, 0.0),     # 48 routes: narrow items (two 128-element k-blocks per stage)
    (4, 64, 6, 256, 256, 0.0),      # a verification-width batch
    (700, 8, 2, 256, 256, 0.0),     # heavy experts: big items
]


@pytest.mark.parametrize("T,E,k,d,f,p", W8A8_CASES)
def test_w8a8_path_matches_oracle(T, E, k, d, f, p):
    logits, mask, x, wg, wu, wd = _case(T, E, k, d, f, p, seed=T * 3 + E)
    if T == 700:
        logits[:, 6] += 3.0
        logits[:, 7] += 2.5
    q = [M.moe_quantize_weights_fp8(w.cuda()) for w in (wg, wu, wd)]
    b = M.MoEBuffersW8A8(T, E, k, d, f)
    for t in (b.h, b.y, b.out):
        t.fill_(float("nan"))
    out = M.moe_forward_w8a8(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), *q, k, b)
    M.moe_check_device_error()
    qo = tuple(mo.quantize_bank_fp8(w) for w in (wg, wu, wd))
    for qg, qr in zip(q, qo):
        assert np.array_equal(to_np(qg.codes), qr.codes) and np.array_equal(to_np(qg.scales), qr.scales)
    ref = mo.moe_forward_w8a8(logits, x, qo, k, mask, h_decided=_gpu_h(b))
    R, hq = _check_against_oracle(b, ref, q, k, d)
    if T == 700:
        counts = ref["counts"]
        assert np.maximum(counts - 128, 0).sum() * 2 >= counts.sum()      # the big-item carve-up applies
    # y: the oracle's down projection of the GPU's own quantized h (same E4M3 products, fp32 accumulation)
    y_ref = mo.grouped_down(mo.dequantize_weights_fp8(hq.codes, hq.scales), ref["offsets"], qo)
    assert_close(b.y[:R], y_ref, "bf16")
    assert torch.all(b.y[R:] == 0)
    assert_close(out, ref["out"], "bf16")


def test_w8a8_steps_equal_the_whole_path():
    T, E, k, d, f = 100, 8, 2, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, 0.1, seed=5))
    q = [M.moe_quantize_weights_fp8(w) for w in (wg, wu, wd)]
    a = M.MoEBuffersW8A8(T, E, k, d, f)
    whole = M.moe_forward_w8a8(logits, x, mask, *q, k, a).clone()
    b = M.MoEBuffersW8A8(T, E, k, d, f)
    M.moe_route_topk_offsets(logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws)
    xq = M.moe_quantize_weights_fp8(x)
    M.moe_scatter_rows_e4m3(xq.codes, xq.scales, b.ids, mask, b.offsets, b.xs, b.xs_scales, b.row_of_route,
                            b.route_of_row, b.ws)
    M.moe_grouped_gate_up_w8a8(b.xs, b.xs_scales, b.offsets, q[0], q[1], b.h)
    hq = M.moe_quantize_weights_fp8(b.h)
    M.moe_grouped_down_w8a8(hq.codes, hq.scales, b.offsets, q[2], b.y)
    M.moe_combine(b.y, b.row_of_route, b.w, b.out)
    M.moe_check_device_error()
    assert torch.equal(b.out.view(torch.int32), whole.view(torch.int32))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_t4", "prefill_t401", "prefill_t2048", "prefill_t8192"])
def test_w8a8_full_size_workload(name):
    """Every output at full size: the integer outputs and every code bit for bit, h on every compact row, out on
    every token against the oracle's FP8-activation path."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    q = [M.moe_quantize_weights_fp8(inp[n]) for n in ("w_gate", "w_up", "w_down")]
    b = M.MoEBuffersW8A8(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    out = M.moe_forward_w8a8(inp["logits"], inp["x"], inp["mask"], *q, cfg.k, b)
    M.moe_check_device_error()

    cache = {}

    def fetch(e0, e1):
        # the oracle quantizes each block of experts once (the gate/up and the down step both visit it)
        if (e0, e1) not in cache:
            banks = []
            for qq, name_w in zip(q, ("w_gate", "w_up", "w_down")):
                ob = mo.quantize_bank_fp8(inp[name_w][e0:e1].cpu())
                assert np.array_equal(to_np(qq.codes[e0:e1]), ob.codes)
                assert np.array_equal(to_np(qq.scales[e0:e1]), ob.scales)
                banks.append(ob)
            cache[(e0, e1)] = tuple(banks)
        return cache[(e0, e1)]

    ref = mo.moe_forward_w8a8(inp["logits"].cpu(), inp["x"].cpu(), fetch, cfg.k,
                              None if inp["mask"] is None else inp["mask"].cpu(), h_decided=_gpu_h(b))
    _check_against_oracle(b, ref, q, cfg.k, cfg.d)
    st = assert_close(out, ref["out"], "bf16")
    print(f"{name} W8A8: rel_fro={st['rel_fro']:.2e} max/rms={st['max_abs'] / st['rms_ref']:.2e}")


@pytest.mark.parametrize("T,E,k,d,f,p", [(300, 16, 4, 512, 384, 0.1), (40, 8, 6, 4096, 2048, 0.0),
                                         (33, 4, 2, 8192, 128, 0.2), (20, 4, 2, 256, 1920, 0.0)])
def test_fused_quantizers_equal_the_weight_quantizer(T, E, k, d, f, p):
    """The scatter that quantizes the token rows, and the row quantizer of h, give the codes and scales of
    moe_quantize_weights_fp8 (and of moe_scatter_rows_e4m3 on them) bit for bit."""
    logits, mask, x, *_ = _case(T, E, k, 128, 128, p, seed=d + T)
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    md = None if mask is None else mask.cuda()
    a = M.MoEBuffersW8A8(T, E, k, d, f)
    M.moe_route_topk_offsets(logits.cuda(), md, k, a.ids, a.w, a.counts, a.offsets, a.ws)
    ref_q = M.moe_quantize_weights_fp8(x)
    ref_xs = torch.empty_like(a.xs)
    ref_sc = torch.empty_like(a.xs_scales)
    ref_ror, ref_rro = torch.empty_like(a.row_of_route), torch.empty_like(a.route_of_row)
    M.moe_scatter_rows_e4m3(ref_q.codes, ref_q.scales, a.ids, md, a.offsets, ref_xs, ref_sc, ref_ror, ref_rro, a.ws)
    a.xs.fill_(7)
    a.xs_scales.fill_(float("nan"))
    M.moe_scatter_rows_quant_e4m3(x, a.ids, md, a.offsets, a.x_q, a.x_scales, a.xs, a.xs_scales, a.row_of_route,
                                  a.route_of_row, a.ws)
    M.moe_check_device_error()
    assert torch.equal(a.x_q, ref_q.codes) and torch.equal(a.x_scales, ref_q.scales)
    assert torch.equal(a.xs, ref_xs) and torch.equal(a.xs_scales.view(torch.int32), ref_sc.view(torch.int32))
    assert torch.equal(a.row_of_route, ref_ror) and torch.equal(a.route_of_row, ref_rro)
    # rows of h: the rows below R as the weight quantizer gives them, the rows beyond it zero codes, scale 1
    R = int(a.offsets[-1])
    h = torch.randn(T * k, f, device="cuda").to(torch.bfloat16)
    h[R:] = 0
    h[0, :5] = -0.0
    codes = torch.full((T * k, f), 9, dtype=torch.uint8, device="cuda")
    scales = torch.full((T * k,), float("nan"), device="cuda")
    M.moe_quantize_rows_e4m3(h, a.offsets, codes, scales)
    M.moe_check_device_error()
    ref_h = M.moe_quantize_weights_fp8(h)
    assert torch.equal(codes, ref_h.codes) and torch.equal(scales, ref_h.scales)


@pytest.mark.parametrize("T,E,k,d,p", [(4, 64, 6, 256, 0.0), (100, 8, 2, 256, 0.1), (64, 10, 8, 512, 0.3),
                                       (128, 256, 4, 128, 0.0), (1, 4, 2, 4096, 0.0)])
def test_small_chunk_routing_quantize_scatter_in_one_launch(T, E, k, d, p):
    """moe_route_scatter_quant_small_e4m3 gives the routing outputs of moe_route_topk_offsets and the rows of
    moe_scatter_rows_quant_e4m3, bit for bit."""
    logits, mask, *_ = _case(T, E, k, 128, 128, p, seed=T + d)
    x = (torch.randn(T, d) * 2).to(torch.bfloat16).cuda()
    lg, md = logits.cuda(), None if mask is None else mask.cuda()
    a = M.MoEBuffersW8A8(T, E, k, d, 128)
    M.moe_route_topk_offsets(lg, md, k, a.ids, a.w, a.counts, a.offsets, a.ws)
    M.moe_scatter_rows_quant_e4m3(x, a.ids, md, a.offsets, a.x_q, a.x_scales, a.xs, a.xs_scales, a.row_of_route,
                                  a.route_of_row, a.ws)
    b = M.MoEBuffersW8A8(T, E, k, d, 128)
    b.xs.fill_(5)
    b.xs_scales.fill_(float("nan"))
    b.route_of_row.fill_(77)
    M.moe_route_scatter_quant_small_e4m3(lg, x, md, k, b)
    M.moe_check_device_error()
    for name in ("ids", "counts", "offsets", "row_of_route", "route_of_row", "x_q", "xs"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    for name in ("w", "x_scales", "xs_scales"):
        assert torch.equal(getattr(a, name).view(torch.int32), getattr(b, name).view(torch.int32)), name
