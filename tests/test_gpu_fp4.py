"""GPU parity of the 4-bit block-scaled weight path (quantizer, grouped FFN, whole path).

The quantizer's codes, block scales and row scales must equal the oracle's
bit for bit (the GPU keeps the block scales in the tile-major layout the FFN
loads; the test reorders them).  The FFN is compared with the oracle on the
values the codes stand for, under the tolerances of the bf16 path: the GPU
widens code * block scale to fp16 exactly, takes the bf16 token rows to fp16
exactly, accumulates in fp32 and rounds h to fp16; the oracle rounds nothing.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_f16_rounded, to_np
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _oracle_layout(q: "M.FP4Weights"):
    """The GPU's tile-major block scales [E][K/64][M][4] in the oracle's row-major layout [E][M][K/16]."""
    bs = q.block_scales.permute(0, 2, 1, 3).contiguous()
    return bs.reshape(bs.shape[0], bs.shape[1], -1)


def _check_codes(q, ob, e0=0, e1=None):
    e1 = q.codes.shape[0] if e1 is None else e1
    assert np.array_equal(to_np(q.codes[e0:e1]), ob.codes)
    assert np.array_equal(to_np(_oracle_layout(q)[e0:e1]), ob.block_scales)
    assert np.array_equal(to_np(q.scales[e0:e1]), ob.scales)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fp4_quantizer_is_bit_exact(dtype):
    g = torch.Generator().manual_seed(6)
    E, rows, K = 3, 256, 512
    w = torch.randn(E, rows, K, generator=g) * 0.02
    w[0, 0] = 0.0                                       # all-zero row
    w[0, 1, :16] = 0.0                                  # an all-zero block
    w[0, 2, 16:32] = -0.0
    w[1, 3, :] *= 1e-4                                  # small row
    w[1, 4, 0] = 3.0                                    # one large value: the other blocks' scales are tiny
    w[2, 5, :16] = torch.tensor([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5,
                                 -5, -6]) * 0.01        # ties of the E2M1 rounding (up to the scale's rounding)
    w = w.to(dtype)
    q = M.moe_quantize_weights_fp4(w.cuda())
    M.moe_check_device_error()
    _check_codes(q, mo.quantize_bank_fp4(w))


def _routing(T, E, k, seed, p_mask=0.0):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + 1.5 * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    return logits, mask


FP4_CASES = [
    # E, d, f, T, k, p_mask
    (8, 256, 384, 300, 2, 0.0),
    (4, 128, 128, 77, 2, 0.2),
    (16, 512, 256, 600, 4, 0.1),
    (1, 128, 256, 200, 1, 0.0),
    (3, 384, 256, 150, 2, 0.0),
    (256, 256, 256, 4, 6, 0.0),
]


@pytest.mark.parametrize("E,d,f,T,k,p", FP4_CASES)
def test_fp4_ffn_matches_oracle(E, d, f, T, k, p):
    logits, mask = _routing(T, E, k, seed=E * 7 + T, p_mask=p)
    g = torch.Generator().manual_seed(d + f)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    banks = [(torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16),
             (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16),
             (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)]
    q = [M.moe_quantize_weights_fp4(b.cuda()) for b in banks]
    qo = tuple(mo.quantize_bank_fp4(b) for b in banks)
    for qq, ob in zip(q, qo):
        _check_codes(qq, ob)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.float16)
    bufs.h.fill_(float("nan"))
    out = M.moe_forward_fp4(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), *q, k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits, x, qo, k, mask)
    assert np.array_equal(to_np(bufs.ids), ref["ids"])
    assert np.array_equal(to_np(bufs.route_of_row), ref["route_of_row"])
    R = int(ref["offsets"][-1])
    assert_close_f16_rounded(bufs.h[:R], ref["h"])
    # the down step against the oracle applied to the GPU's own h
    y_ref = mo.grouped_down(bufs.h[:R].cpu(), ref["offsets"], qo)
    assert_close(bufs.y[:R], y_ref, "bf16")
    assert_close(out, ref["out"], "bf16")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_t4", "prefill_t401", "prefill_t2048", "prefill_t8192"])
def test_fp4_full_size_workload(name):
    """Every code, block scale and row scale of the bank bit for bit against the oracle's quantizer; h on every
    compact row and out on every token against the oracle on the values the codes stand for."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    q = [M.moe_quantize_weights_fp4(inp[n]) for n in ("w_gate", "w_up", "w_down")]
    bufs = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.float16)
    bufs.h.fill_(float("nan"))
    out = M.moe_forward_fp4(inp["logits"], inp["x"], inp["mask"], *q, cfg.k, bufs)
    M.moe_check_device_error()
    cache = {}

    def fetch(e0, e1):
        # the oracle quantizes each block of experts once and checks the GPU's codes of the block
        if (e0, e1) not in cache:
            banks = []
            for qq, name_w in zip(q, ("w_gate", "w_up", "w_down")):
                ob = mo.quantize_bank_fp4(inp[name_w][e0:e1].cpu())
                _check_codes(qq, ob, e0, e1)
                banks.append(ob)
            cache[(e0, e1)] = tuple(banks)
        return cache[(e0, e1)]

    ref = mo.moe_forward(inp["logits"].cpu(), inp["x"].cpu(), fetch, cfg.k,
                         None if inp["mask"] is None else inp["mask"].cpu())
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(bufs, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    assert_close_f16_rounded(bufs.h[:R], ref["h"])
    st = assert_close(out, ref["out"], "bf16")
    print(f"{name} FP4: rel_fro={st['rel_fro']:.2e} max/rms={st['max_abs'] / st['rms_ref']:.2e}")
