"""Pins of the oracle's FP8 E4M3 weight quantization.

The rounding is checked against PyTorch's float8_e4m3fn cast (an independent
implementation of the same OCP format), the codes against the format's bit
layout, and the per-channel scaling against its defining properties.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 100,                    # normals
        rng.standard_normal(5000) * 2.0 ** -8,               # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11]),
    ]).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref_t = torch.from_numpy(x).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(mo.e4m3_round(x), ref_t.to(torch.float64).numpy())
    # byte codes too, so that the sign of zero results is compared as well
    np.testing.assert_array_equal(mo.e4m3_encode(mo.e4m3_round(x)), ref_t.view(torch.uint8).numpy())


def test_negative_values_that_round_to_zero_keep_their_sign():
    x = np.array([-0.0, -1e-9, -2.0 ** -11, 0.0, 1e-9], dtype=np.float32)
    codes = mo.e4m3_encode(mo.e4m3_round(x))
    assert codes.tolist() == [0x80, 0x80, 0x80, 0x00, 0x00]


def test_e4m3_ties_go_to_even_and_saturate():
    # 1 + 1/16 lies halfway between 1 and 1.125: even mantissa (1.0) wins
    assert mo.e4m3_round(1.0 + 1 / 16) == 1.0
    # 1.125 + 1/16 lies between 1.125 (odd) and 1.25 (even): 1.25 wins
    assert mo.e4m3_round(1.125 + 1 / 16) == 1.25
    assert mo.e4m3_round(460.0) == 448.0 and mo.e4m3_round(1e6) == 448.0 and mo.e4m3_round(-1e6) == -448.0
    assert mo.e4m3_round(2.0 ** -10) == 0.0            # half of the smallest subnormal -> even (0)
    assert mo.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8  # 1.5 quanta -> 2 quanta (even)


def test_code_layout_and_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # all but NaN
    vals = mo.e4m3_decode(codes)
    assert vals.max() == 448.0 and vals.min() == -448.0
    assert mo.e4m3_decode(np.array([0x38]))[0] == 1.0         # 0 0111 000
    assert mo.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9   # smallest subnormal
    np.testing.assert_array_equal(mo.e4m3_encode(vals), codes)
    torch_vals = torch.from_numpy(codes.view(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals, torch_vals)


def test_per_channel_scaling_properties():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((3, 16, 64)) * 0.02).astype(np.float32)
    w[1, 5] = 0.0                                       # an all-zero channel
    codes, scales = mo.quantize_weights_fp8(w)
    assert codes.dtype == np.uint8 and scales.dtype == np.float32 and scales.shape == (3, 16)
    q = mo.e4m3_decode(codes)
    assert scales[1, 5] == 1.0 and np.all(q[1, 5] == 0)
    amax_q = np.abs(q).max(axis=-1)
    nz = np.abs(w).max(axis=-1) > 0
    assert np.all(amax_q[nz] == 448.0)                  # the largest element lands on the largest code
    deq = mo.dequantize_weights_fp8(codes, scales)
    # RNE error bound: half a quantum of the element's binade, at most 2^-4 of |w| for normals
    err = np.abs(deq - w.astype(np.float64))
    assert np.all(err <= np.abs(w) * 2.0 ** -4 + scales[..., None].astype(np.float64) * 2.0 ** -10 + 1e-30)


def test_quantize_reads_float32_quotients():
    """The quotient is rounded to float32 before the E4M3 rounding (both sides compute it in float32)."""
    w = np.array([[0.1, 0.3, -0.7]], dtype=np.float32)
    codes, scales = mo.quantize_weights_fp8(w)
    expect_q = mo.e4m3_round((w / scales[:, None]).astype(np.float32))
    np.testing.assert_array_equal(mo.e4m3_decode(codes), expect_q)


def test_quantized_bank_ffn_is_the_dequantized_ffn():
    """The FFN on a bank of E4M3 codes + row scales is the dense SwiGLU FFN on the weights those codes stand
    for, decoded here by PyTorch's float8_e4m3fn (an implementation independent of the oracle's decoder)."""
    rng = np.random.default_rng(2)
    n, d, f = 5, 32, 48
    x = rng.standard_normal((n, d))
    banks = [(rng.standard_normal((1, f, d)) / d ** 0.5).astype(np.float32),
             (rng.standard_normal((1, f, d)) / d ** 0.5).astype(np.float32),
             (rng.standard_normal((1, d, f)) / f ** 0.5).astype(np.float32)]
    q = [mo.quantize_bank_fp8(b) for b in banks]

    def torch_dequant(qb):
        vals = torch.from_numpy(qb.codes).view(torch.float8_e4m3fn).to(torch.float64)
        return vals * torch.from_numpy(qb.scales).to(torch.float64)[..., None]

    wg, wu, wd = (torch_dequant(b)[0] for b in q)
    xt = torch.from_numpy(x)
    ref = torch.nn.functional.linear(torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T), wd).numpy()
    got = mo.grouped_ffn(x, np.array([0, n], dtype=np.int32), tuple(q))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_bf16_rounding_matches_torch_cast():
    """bf16 rounding of float32 values (exact in float64) against PyTorch's float32 -> bfloat16 cast."""
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 3,
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),          # fp32 subnormals
        np.array([0.0, -0.0, 3.3895e38, -3.3895e38, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = mo.round_bf16(x)
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    # hand-worked ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (even: 1); 1 + 3*2^-8 -> 1 + 2^-6
    assert mo.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert mo.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert np.isinf(mo.round_bf16(3.4e38))


def test_w8a8_path_is_the_dense_ffn_on_quantized_operands():
    """E=1, k=1: the FP8-activation path is a dense SwiGLU FFN on E4M3-quantized x, weights and h.  Here every
    quantization and the bf16 rounding of h run through PyTorch's own casts (float8_e4m3fn, bfloat16)."""
    g = torch.Generator().manual_seed(3)
    T, d, f = 13, 32, 48
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(1, f, d, generator=g) / d ** 0.5).float()
    wu = (torch.randn(1, f, d, generator=g) / d ** 0.5).float()
    wd = (torch.randn(1, d, f, generator=g) / f ** 0.5).float()
    logits = torch.randn(T, 1, generator=g)

    def torch_quant(rows32):
        # per-row scale amax / 448 in fp32, codes = E4M3 of the fp32 quotient; returns the values in float64
        amax = rows32.abs().amax(dim=-1)
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        q = (rows32 / scale[..., None]).to(torch.float8_e4m3fn)
        return q.to(torch.float64) * scale.to(torch.float64)[..., None]

    xq = torch_quant(x.float())
    gq, uq, dq = (torch_quant(w[0]) for w in (wg, wu, wd))
    h = torch.nn.functional.silu(xq @ gq.T) * (xq @ uq.T)
    h_b = h.to(torch.float32).to(torch.bfloat16).float()
    ref = (torch_quant(h_b) @ dq.T).numpy()
    res = mo.moe_forward_w8a8(logits, x, tuple(mo.quantize_bank_fp8(w) for w in (wg, wu, wd)), 1)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-14)
