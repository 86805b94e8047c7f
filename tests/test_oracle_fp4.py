"""Pins of the oracle's 4-bit block-scaled weight format (E2M1 codes, an E4M3 scale per 16 values, an fp32
scale per row).

The E2M1 element type is checked against its code table, written out here
from the format's definition (sign, two exponent bits with bias 1, one
mantissa bit), and its rounding against a brute-force search over that table;
the quantizer against a hand-worked row and, on random rows, against a
brute-force nearest-value search per block; the FFN on 4-bit banks against a
dense SwiGLU FFN on weights decoded here from the table.
"""

import numpy as np
import torch

from oracle import moe_oracle as mo

# value of each 4-bit code, from the E2M1 definition: codes 0-7 positive, 8-15 their negatives
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
E4M3_448 = 0x7E     # 0 1111 110: 1.75 * 2^8


def _table_value(code):
    v = E2M1_TABLE[code & 7]
    return -v if code & 8 else v


def _brute_round(x):
    """Nearest table value; an exact tie goes to the code with mantissa bit 0; beyond 6 saturates."""
    best = None
    for code in range(8):
        v = E2M1_TABLE[code]
        dist = abs(abs(x) - v)
        if best is None or dist < best[0] or (dist == best[0] and (code & 1) == 0):
            best = (dist, code, v)
    return float(np.copysign(best[2], x))


def test_e2m1_code_table():
    codes = np.arange(16, dtype=np.uint8)
    vals = mo.e2m1_decode(codes)
    assert vals.tolist() == [_table_value(c) for c in range(16)]
    assert np.signbit(vals[8]) and not np.signbit(vals[0])       # code 8 is -0.0
    np.testing.assert_array_equal(mo.e2m1_encode(vals), codes)


def test_e2m1_rounding_against_brute_force():
    rng = np.random.default_rng(0)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]               # every tie between neighbours
    x = np.concatenate([rng.standard_normal(3000) * 3, rng.uniform(-8, 8, 3000), mids, [-m for m in mids],
                        [0.0, -0.0, 6.0, 6.5, 100.0, -100.0, 1e-9, -1e-9]])
    got = mo.e2m1_round(x)
    ref = np.array([_brute_round(v) for v in x])
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    # the ties by hand: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert mo.e2m1_round(np.array(mids)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_fp4_quantizer_hand_worked_row():
    """Row max 2.625 makes the row scale exactly 2.625 / 2688 = 2^-10.
    Block 0 (max 2.625): 2.625 / 6 / 2^-10 = 448 -> block scale 448 (code 0x7E), divisor 448 * 2^-10 = 0.4375,
    so the values 0.4375 * v take the codes of v; 0.109375 and 0.328125 are the ties 0.25 and 0.75.
    Block 1 (max 0.4375): 0.4375 / 6 / 2^-10 = 74.67 -> E4M3 72 (9 * 8; code 0 1101 001 = 0x69), divisor
    72 * 2^-10 = 0.0703125, so 0.4375 -> 6.22 saturates to 6 and 0.0703125 -> 1."""
    b0 = np.array([2.625, 1.3125, -0.65625, 0.21875, 0.109375, 0.328125, 0.0, -0.0,
                   0.4375, -0.4375, 0.875, 1.75, -2.625, 0.0546875, 0.1640625, 0.0], dtype=np.float32)
    b1 = np.zeros(16, dtype=np.float32)
    b1[:4] = [0.4375, 0.0703125, -0.140625, 0.03515625]
    w = np.concatenate([b0, b1])[None]
    codes, bs, sc = mo.quantize_weights_fp4(w)
    assert sc.tolist() == [2.0 ** -10]
    assert bs.tolist() == [[E4M3_448, 0x69]]
    q = [(codes[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
    # block 0: 6, 3, -1.5, 0.5, tie 0.25 -> 0, tie 0.75 -> 1, 0, -0, 1, -1, 2, 4, -6, tie 0.125 -> 0, 0.375 -> 0.5, 0
    assert [_table_value(c) for c in q[:16]] == [6, 3, -1.5, 0.5, 0, 1, 0, -0.0, 1, -1, 2, 4, -6, 0, 0.5, 0]
    # block 1: 0.4375 / 0.0703125 = 6.22 -> 6, 1, -2, 0.5, then zeros
    assert [_table_value(c) for c in q[16:20]] == [6, 1, -2, 0.5]
    deq = mo.dequantize_weights_fp4(codes, bs, sc)
    assert deq[0, 0] == 2.625 and deq[0, 16] == 6 * 72 * 2.0 ** -10


def test_fp4_quantizer_picks_the_nearest_value_of_each_block():
    """On random rows: every dequantized weight is the nearest (ties to the even code) among the 15 values
    row scale * block scale * E2M1 that its block offers; the row's largest block has the scale of its max."""
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((6, 64)) * 0.02).astype(np.float32)
    w[2, 16:32] = 0.0                               # an all-zero block: scale code 0, codes 0
    w[3, :] *= 1e-3
    codes, bs, sc = mo.quantize_weights_fp4(w)
    deq = mo.dequantize_weights_fp4(codes, bs, sc)
    bsv = mo.e4m3_decode(bs)
    for r in range(w.shape[0]):
        for j in range(4):
            unit = float(sc[r]) * bsv[r, j]
            for i in range(16 * j, 16 * j + 16):
                q = w[r, i] / np.float32(np.float32(bsv[r, j]) * sc[r]) if unit > 0 else 0.0
                assert deq[r, i] == (_brute_round(float(np.float32(q))) * unit if unit > 0 else 0.0)
    assert np.all(bs[2, 1] == 0) and np.all(deq[2, 16:32] == 0)
    # relative error of the format on N(0, s^2) rows: about 10 % (E2M1 has one mantissa bit)
    err = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert 0.02 < err < 0.2


def test_fp4_bank_ffn_is_the_dequantized_ffn():
    """The FFN on a 4-bit bank is the dense SwiGLU FFN on the weights its codes stand for, decoded here from
    the code table and PyTorch's float8_e4m3fn (independently of the oracle's decoder)."""
    rng = np.random.default_rng(2)
    n, d, f = 5, 64, 48
    x = rng.standard_normal((n, d))
    banks = [(rng.standard_normal((1, f, d)) / d ** 0.5).astype(np.float32),
             (rng.standard_normal((1, f, d)) / d ** 0.5).astype(np.float32),
             (rng.standard_normal((1, d, f)) / f ** 0.5).astype(np.float32)]
    q = [mo.quantize_bank_fp4(b) for b in banks]
    table = np.array([_table_value(c) for c in range(16)])

    def decode(bank):
        c = bank.codes[0]
        codes = np.stack([c & 0xF, c >> 4], axis=-1).reshape(c.shape[0], -1)
        bsv = torch.from_numpy(bank.block_scales[0]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return torch.from_numpy(bank.scales[0].astype(np.float64)[:, None] * np.repeat(bsv, 16, axis=1)
                                * table[codes])

    wg, wu, wd = (decode(b) for b in q)
    xt = torch.from_numpy(x)
    ref = torch.nn.functional.linear(torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T), wd).numpy()
    got = mo.grouped_ffn(x, np.array([0, n], dtype=np.int32), tuple(q))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def _restated_fp4_values(rows32):
    """The 4-bit format restated here, in fp32 like the quantizer: s = amax / 2688, block scale = E4M3 (PyTorch's
    float8_e4m3fn cast) of (block max / 6) / s, codes by brute force over the E2M1 table; returns the values
    the codes stand for, float64."""
    r = rows32.to(torch.float32)
    amax = r.abs().amax(dim=-1)
    s = torch.where(amax > 0, amax / 2688.0, torch.ones_like(amax))
    blocks = r.reshape(*r.shape[:-1], -1, 16)
    bmax = blocks.abs().amax(dim=-1)
    bv = ((bmax / 6.0) / s[..., None]).to(torch.float8_e4m3fn).to(torch.float32)
    denom = bv * s[..., None]
    q = torch.where(denom[..., None] > 0, blocks / denom[..., None], torch.zeros_like(blocks))
    vals = np.vectorize(_brute_round)(q.numpy().astype(np.float64))
    # the value a code stands for: s * value(block scale) * value(code), exactly (float64)
    unit = bv.numpy().astype(np.float64) * s.numpy().astype(np.float64)[..., None]
    out = vals * unit[..., None]
    return torch.from_numpy(out.reshape(r.shape))


def test_w4a4_path_is_the_dense_ffn_on_quantized_operands():
    """E=1, k=1: the 4-bit-activation path is a dense SwiGLU FFN on 4-bit-quantized x, weights and h, each
    quantization restated here (PyTorch's E4M3 cast for the block scales, a brute-force E2M1 search), and
    the bf16 rounding of h by PyTorch's cast."""
    g = torch.Generator().manual_seed(4)
    T, d, f = 9, 64, 48
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(1, f, d, generator=g) / d ** 0.5).float()
    wu = (torch.randn(1, f, d, generator=g) / d ** 0.5).float()
    wd = (torch.randn(1, d, f, generator=g) / f ** 0.5).float()
    logits = torch.randn(T, 1, generator=g)
    xq = _restated_fp4_values(x.float())
    gq, uq, dq = (_restated_fp4_values(w[0]) for w in (wg, wu, wd))
    h = torch.nn.functional.silu(xq @ gq.T) * (xq @ uq.T)
    h_b = h.to(torch.float32).to(torch.bfloat16).float()
    ref = (_restated_fp4_values(h_b) @ dq.T).numpy()
    res = mo.moe_forward_w4a4(logits, x, tuple(mo.quantize_bank_fp4(w) for w in (wg, wu, wd)), 1)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-14)
