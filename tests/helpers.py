"""Shared helpers of the test suite: tolerances and oracle adapters."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances of the floating-point outputs (the workloads' statement of the
# bar): bf16 operands with fp32 accumulation -> max|gpu - ref| <= 2e-2 *
# rms(ref) and relative Frobenius error <= 5e-3; fp32 operands -> relative
# error <= 1e-5 (Frobenius, and max|gpu - ref| <= 1e-5 * max|ref|).
BF16_MAX_OVER_RMS = 2e-2
BF16_REL_FRO = 5e-3
F32_REL = 1e-5
# gate weights are computed in fp32 with expf against a float64 oracle
WEIGHT_REL = 1e-6


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.numpy()
    return np.asarray(t)


def error_stats(got, ref):
    got = to_np(got).astype(np.float64)
    ref = to_np(ref).astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    fro = float(np.linalg.norm(ref))
    return {
        "max_abs": float(np.max(np.abs(diff))) if diff.size else 0.0,
        "rms_ref": rms,
        "max_ref": float(np.max(np.abs(ref))) if ref.size else 0.0,
        "rel_fro": float(np.linalg.norm(diff) / fro) if fro > 0 else float(np.linalg.norm(diff)),
        "finite": bool(np.all(np.isfinite(got))),
    }


def assert_close(got, ref, dtype: str):
    st = error_stats(got, ref)
    assert st["finite"], st
    if dtype == "bf16":
        assert st["max_abs"] <= BF16_MAX_OVER_RMS * st["rms_ref"], st
        assert st["rel_fro"] <= BF16_REL_FRO, st
    else:
        assert st["rel_fro"] <= F32_REL, st
        assert st["max_abs"] <= F32_REL * max(st["max_ref"], 1e-30), st
    return st


def assert_close_bf16_rounded(got, ref):
    """An intermediate stored in bf16 (h): each element within its bf16 rounding bound.

    Round-to-nearest-even to bf16 (8 significant bits) moves a value by at
    most 2^-8 of its magnitude; 1e-3 * rms(ref) covers the fp32-versus-fp64
    accumulation difference of elements that cancel to near zero.
    """
    g = to_np(got).astype(np.float64)
    r = to_np(ref).astype(np.float64)
    assert g.shape == r.shape
    st = error_stats(g, r)
    assert st["finite"], st
    bound = 2.0 ** -8 * np.abs(r) + 1e-3 * st["rms_ref"]
    worst = float(np.max(np.abs(g - r) - bound)) if g.size else -1.0
    assert worst <= 0.0, (worst, st)
    assert st["rel_fro"] <= BF16_REL_FRO, st
    return st


def assert_close_f16_rounded(got, ref):
    """An intermediate stored in fp16 (h of the FP8-weight path): each element
    within its fp16 rounding bound, 2^-11 of its magnitude, plus 1e-3 * rms(ref)
    for the fp32-versus-fp64 accumulation difference of elements near zero."""
    g = to_np(got).astype(np.float64)
    r = to_np(ref).astype(np.float64)
    assert g.shape == r.shape
    st = error_stats(g, r)
    assert st["finite"], st
    bound = 2.0 ** -11 * np.abs(r) + 1e-3 * st["rms_ref"]
    worst = float(np.max(np.abs(g - r) - bound)) if g.size else -1.0
    assert worst <= 0.0, (worst, st)
    assert st["rel_fro"] <= BF16_REL_FRO, st
    return st


def oracle_weights(w_gate, w_up, w_down, fp8=False, check_codes=None):
    """The oracle's view of expert banks that may live on the GPU: fetch(e0, e1) copies experts e0 .. e1-1
    to host memory (bf16 read exactly by the oracle).  With fp8 the oracle quantizes each block itself
    (FP8 E4M3 codes + per-channel scales) and works on the values the codes stand for; check_codes, if
    given, is called as check_codes(e0, e1, banks) with the oracle's quantized banks of the block."""
    from oracle import moe_oracle as mo
    quantized = {}

    def fetch(e0, e1):
        banks = tuple(None if w is None else w[e0:e1].detach().cpu() for w in (w_gate, w_up, w_down))
        if fp8:
            # each block is quantized once (the gate/up and the down step both visit it)
            if (e0, e1) not in quantized:
                quantized[(e0, e1)] = tuple(None if b is None else mo.quantize_bank_fp8(b) for b in banks)
                if check_codes is not None:
                    check_codes(e0, e1, quantized[(e0, e1)])
            banks = quantized[(e0, e1)]
        return banks

    return fetch


# full-size oracle results, computed once per workload and test session
_FULL_SIZE = {}


def full_size_reference(inp, fp8=False, check_codes=None):
    """The oracle's moe_forward of a full-size workload (ids, w, counts, offsets, the permutation, h, out).

    The weight bank is fetched 16 experts at a time from wherever it lives.  Results are cached per
    (workload, weight format) for the session; xs and y are dropped to bound host memory.
    """
    from oracle import moe_oracle as mo
    cfg = inp["cfg"]
    key = (cfg.name, cfg.seed, fp8)
    if key not in _FULL_SIZE:
        mask = None if inp["mask"] is None else inp["mask"].cpu()
        res = mo.moe_forward(inp["logits"].cpu(), inp["x"].cpu(),
                             oracle_weights(inp["w_gate"], inp["w_up"], inp["w_down"], fp8, check_codes),
                             cfg.k, mask)
        del res["xs"], res["y"]
        _FULL_SIZE[key] = res
    return _FULL_SIZE[key]
