"""Python marshalling of the C++ CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this module.  The product path (the
CUDA library and its Python binding) never calls it, and this module imports
nothing from the product package.

Every computation of the method happens in ``moe_oracle.cpp`` (plain C++,
double precision; its header states what it computes, the pages' passages it
follows, the readings of points the pages leave open and what pins it).  This
module only converts arguments to contiguous arrays, passes pointers and
sizes, and composes the steps of the path in the pages' order.

Operands may be numpy arrays or CPU torch tensors; bfloat16 tensors are
passed as their raw bits and read exactly by the oracle.  A weight argument is
either a tuple ``(w_gate, w_up, w_down)`` of whole banks ([E][f][d],
[E][f][d], [E][d][f]) or a callable ``fetch(e0, e1)`` returning the banks of
experts e0 .. e1-1 only, so that a bank that does not fit in host memory can
be visited a block of experts at a time.  A bank may also be a
``QuantizedBank`` of FP8 E4M3 codes with one fp32 scale per row.
"""

from __future__ import annotations

import contextlib
import ctypes
import dataclasses
import os
import threading

import numpy as np

from . import build as _build

ORC_F64, ORC_F32, ORC_BF16, ORC_E4M3, ORC_FP4 = 0, 1, 2, 3, 4

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_longlong
_SIGNATURES = {
    "oracle_version": (),
    "oracle_threads": (),
    "oracle_route_topk": (_P, _L, _I, _I, _P, _P),
    "oracle_route_histogram": (_P, _P, _L, _I, _I, _P),
    "oracle_prefix_offsets": (_P, _I, _P),
    "oracle_scatter_permutation": (_P, _P, _L, _I, _P, _P),
    "oracle_gather_rows": (_P, _I, _L, _I, _P, _L, _I, _P),
    "oracle_grouped_swiglu": (_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P),
    "oracle_grouped_down": (_P, _P, _I, _I, _I, _I, _P, _I, _P, _P),
    "oracle_combine": (_P, _L, _P, _P, _L, _I, _I, _P),
    "oracle_silu": (_P, _L, _P),
    "oracle_e4m3_round": (_P, _L, _P),
    "oracle_e4m3_encode": (_P, _L, _P),
    "oracle_round_bf16": (_P, _L, _P),
    "oracle_e4m3_decode": (_P, _L, _P),
    "oracle_quantize_fp8": (_P, _I, _L, _I, _P, _P),
    "oracle_dequantize_fp8": (_P, _P, _L, _I, _P),
    "oracle_router_logits": (_P, _I, _P, _I, _L, _I, _I, _P),
    "oracle_e2m1_round": (_P, _L, _P),
    "oracle_e2m1_encode": (_P, _L, _P),
    "oracle_e2m1_decode": (_P, _L, _P),
    "oracle_quantize_fp4": (_P, _I, _L, _I, _P, _P, _P),
    "oracle_dequantize_fp4": (_P, _P, _P, _L, _I, _P),
}

_state = threading.local()
_default = {"lib": None}


def _open(path: str):
    lib = ctypes.CDLL(path)
    for name, args in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = list(args)
        fn.restype = ctypes.c_int
    return lib


def _lib():
    lib = getattr(_state, "lib", None)
    if lib is not None:
        return lib
    if _default["lib"] is None:
        _default["lib"] = _open(_build.build())
    return _default["lib"]


@contextlib.contextmanager
def use_library(path: str):
    """Run the oracle from another build of its source (the mutation tests' planted mistakes)."""
    prev = getattr(_state, "lib", None)
    _state.lib = _open(path)
    try:
        yield
    finally:
        _state.lib = prev


def threads() -> int:
    """Threads of the oracle's parallel loops."""
    return int(_lib().oracle_threads())


def _call(name, *args):
    if getattr(_lib(), name)(*args) != 0:
        raise ValueError(f"{name}: invalid argument")


# ---------------------------------------------------------------------------
# marshalling helpers (no arithmetic of the method)
# ---------------------------------------------------------------------------

def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _np(a, dtype):
    """Contiguous numpy copy/view of `a` with the given dtype (values converted exactly)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu()
            if a.dtype == torch.bfloat16:
                a = a.float()
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    return np.ascontiguousarray(a, dtype=dtype).reshape(a.shape)


def _operand(a):
    """(contiguous array, storage code) of a floating-point operand, read exactly by the oracle."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16), ORC_BF16
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), ORC_F32
    return np.ascontiguousarray(a, dtype=np.float64), ORC_F64


def _mask(mask, shape):
    if mask is None:
        return None
    return np.ascontiguousarray(_np(mask, np.uint8).reshape(shape))


def _opt_ptr(a):
    return None if a is None else _ptr(a)


@dataclasses.dataclass
class QuantizedBank:
    """FP8 E4M3 weights: codes uint8 [..., M, K] and one fp32 scale per row, [..., M]."""

    codes: np.ndarray
    scales: np.ndarray

    @property
    def shape(self):
        return self.codes.shape

    def __getitem__(self, sl):
        return QuantizedBank(self.codes[sl], self.scales[sl])


@dataclasses.dataclass
class Fp4Bank:
    """4-bit weights: E2M1 codes uint8 [..., M, K/2] (element 2i in the low nibble of byte i), E4M3 block
    scales uint8 [..., M, K/16] (one per 16 consecutive values) and one fp32 scale per row, [..., M]."""

    codes: np.ndarray
    block_scales: np.ndarray
    scales: np.ndarray

    @property
    def shape(self):
        return self.codes.shape[:-1] + (2 * self.codes.shape[-1],)

    def __getitem__(self, sl):
        return Fp4Bank(self.codes[sl], self.block_scales[sl], self.scales[sl])


class _Fp4BankC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("block_scales", ctypes.c_void_p)]


class _BankArg:
    """A weight bank marshalled for the oracle: .ptr, .shape (logical [..., M, K]), .code, .scales."""

    def __init__(self, w):
        self.scales = None
        if isinstance(w, Fp4Bank):
            self._codes = np.ascontiguousarray(w.codes, dtype=np.uint8)
            self._bs = np.ascontiguousarray(w.block_scales, dtype=np.uint8)
            self.scales = np.ascontiguousarray(w.scales, dtype=np.float32)
            self._struct = _Fp4BankC(self._codes.ctypes.data, self._bs.ctypes.data)
            self.ptr = ctypes.cast(ctypes.pointer(self._struct), ctypes.c_void_p)
            self.shape, self.code = w.shape, ORC_FP4
        elif isinstance(w, QuantizedBank):
            self._data = np.ascontiguousarray(w.codes, dtype=np.uint8)
            self.scales = np.ascontiguousarray(w.scales, dtype=np.float32)
            self.ptr, self.shape, self.code = _ptr(self._data), self._data.shape, ORC_E4M3
        else:
            self._data, self.code = _operand(w)
            self.ptr, self.shape = _ptr(self._data), self._data.shape

    @property
    def scales_ptr(self):
        return _opt_ptr(self.scales)


def _fetcher(weights):
    """fetch(e0, e1) -> (gate, up, down) banks of experts e0 .. e1-1."""
    if callable(weights):
        return weights
    return lambda e0, e1: tuple(None if w is None else w[e0:e1] for w in weights)


# experts per block when a weight bank is fetched a block at a time
EXPERT_BLOCK = 16


def _blocks(offsets, E):
    """Expert blocks [e0, e1) holding at least one row."""
    for e0 in range(0, E, EXPERT_BLOCK):
        e1 = min(E, e0 + EXPERT_BLOCK)
        if offsets[e1] > offsets[e0]:
            yield e0, e1


# ---------------------------------------------------------------------------
# A1 .. A4
# ---------------------------------------------------------------------------

def route_topk(logits, k: int):
    """ids int32 [T][k] (logit descending, ties to the lower id), w float64 [T][k] (softmax over the k)."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _call("oracle_route_topk", _ptr(lg), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def route_histogram(ids, mask, E: int):
    """counts[e] = unmasked routes to expert e."""
    ids = _np(ids, np.int32)
    T, k = ids.shape if ids.ndim == 2 else (ids.size, 1)
    m = _mask(mask, ids.shape)
    counts = np.empty(E, dtype=np.int32)
    _call("oracle_route_histogram", _ptr(ids), _opt_ptr(m), T, k, E, _ptr(counts))
    return counts


def prefix_offsets(counts):
    """offsets [E+1]: offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]."""
    counts = _np(counts, np.int32)
    offsets = np.empty(counts.size + 1, dtype=np.int32)
    _call("oracle_prefix_offsets", _ptr(counts), counts.size, _ptr(offsets))
    return offsets


def scatter_permutation(ids, mask):
    """row_of_route [T*k] (-1 masked) and route_of_row [T*k] (-1 beyond R)."""
    ids = _np(ids, np.int32)
    T, k = ids.shape if ids.ndim == 2 else (ids.size, 1)
    m = _mask(mask, ids.shape)
    ror = np.empty(T * k, dtype=np.int32)
    rro = np.empty(T * k, dtype=np.int32)
    _call("oracle_scatter_permutation", _ptr(ids), _opt_ptr(m), T, k, _ptr(ror), _ptr(rro))
    return ror, rro


def scatter_rows(x, route_of_row, k: int):
    """xs [R][d] float64: xs[i] = x[token of route_of_row[i]] for the R used rows."""
    xa, code = _operand(x)
    rro = _np(route_of_row, np.int32)
    R = int(np.count_nonzero(rro >= 0))
    T, d = xa.shape
    xs = np.empty((R, d), dtype=np.float64)
    _call("oracle_gather_rows", _ptr(xa), code, T, d, _ptr(rro), R, k, _ptr(xs))
    return xs


# ---------------------------------------------------------------------------
# A5 / A6
# ---------------------------------------------------------------------------

def silu(a):
    """silu(a) = a / (1 + exp(-a)) in float64 (overflow of exp gives -0.0, never NaN)."""
    arr = _np(a, np.float64)
    out = np.empty_like(arr)
    _call("oracle_silu", _ptr(arr), arr.size, _ptr(out))
    return out


def grouped_swiglu(xs, offsets, weights):
    """h [R][f] float64: rows offsets[e] .. offsets[e+1]-1 through expert e's gate/up step."""
    xs = _np(xs, np.float64)
    off = _np(offsets, np.int32)
    E = off.size - 1
    R = int(off[E])
    fetch = _fetcher(weights)
    h = None
    for e0, e1 in _blocks(off, E):
        wg, wu, _ = fetch(e0, e1)
        g, u = _BankArg(wg), _BankArg(wu)
        assert g.code == u.code
        f, d = g.shape[-2], g.shape[-1]
        if h is None:
            h = np.zeros((R, f), dtype=np.float64)
        _call("oracle_grouped_swiglu", _ptr(xs), _ptr(off), e0, e1, d, f, g.ptr, u.ptr, g.code, g.scales_ptr,
              u.scales_ptr, _ptr(h))
    if h is None:
        _, wu, _ = fetch(0, 1)
        h = np.zeros((R, _BankArg(wu).shape[-2]), dtype=np.float64)
    return h


def grouped_down(h, offsets, weights):
    """y [R][d] float64: rows offsets[e] .. offsets[e+1]-1 of h through expert e's down step."""
    h = _np(h, np.float64)
    off = _np(offsets, np.int32)
    E = off.size - 1
    R = int(off[E])
    fetch = _fetcher(weights)
    y = None
    for e0, e1 in _blocks(off, E):
        _, _, wd = fetch(e0, e1)
        dn = _BankArg(wd)
        d, f = dn.shape[-2], dn.shape[-1]
        if y is None:
            y = np.zeros((R, d), dtype=np.float64)
        _call("oracle_grouped_down", _ptr(h), _ptr(off), e0, e1, d, f, dn.ptr, dn.code, dn.scales_ptr, _ptr(y))
    if y is None:
        _, _, wd = fetch(0, 1)
        y = np.zeros((R, _BankArg(wd).shape[-2]), dtype=np.float64)
    return y


def grouped_ffn(xs, offsets, weights):
    """Expert outputs y [R][d]: the gate/up step, then the down step, per expert segment."""
    return grouped_down(grouped_swiglu(xs, offsets, weights), offsets, weights)


def _one_expert(rows, *mats):
    rows = _np(rows, np.float64)
    off = np.array([0, rows.shape[0]], dtype=np.int32)
    return rows, off, tuple(m[None] if not isinstance(m, (QuantizedBank, Fp4Bank)) else
                            type(m)(*(getattr(m, f.name)[None] for f in dataclasses.fields(m))) for m in mats)


def expert_swiglu(rows, w_gate_e, w_up_e):
    """h = silu(x.Wg) * (x.Wu) for each row x (w_gate_e, w_up_e [f][d])."""
    rows, off, (g, u) = _one_expert(rows, w_gate_e, w_up_e)
    return grouped_swiglu(rows, off, (g, u, None))


def expert_down(h, w_down_e):
    """y = h . Wd for each row h (w_down_e [d][f])."""
    h, off, (dn,) = _one_expert(h, w_down_e)
    return grouped_down(h, off, (None, None, dn))


def expert_ffn(rows, w_gate_e, w_up_e, w_down_e):
    """y = (silu(x.Wg) * (x.Wu)) . Wd for each row x."""
    return expert_down(expert_swiglu(rows, w_gate_e, w_up_e), w_down_e)


# ---------------------------------------------------------------------------
# A7 and the whole path
# ---------------------------------------------------------------------------

def combine(y, row_of_route, w, T: int, k: int):
    """out [T][d] float64: +0.0, then w[t,s] * y[row(t,s)] for ascending unmasked slots."""
    y = _np(y, np.float64)
    if y.ndim != 2:
        y = y.reshape(0, 0)
    ror = _np(row_of_route, np.int32).reshape(-1)
    w = _np(w, np.float64).reshape(-1)
    d = y.shape[1]
    out = np.empty((T, d), dtype=np.float64)
    _call("oracle_combine", _ptr(y), y.shape[0], _ptr(ror), _ptr(w), T, k, d, _ptr(out))
    return out


def moe_forward(logits, x, weights, k: int, mask=None):
    """Every intermediate of the path for one chunk (A1 .. A7, in order), as a dict."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids, w = route_topk(lg, k)
    counts = route_histogram(ids, mask, E)
    offsets = prefix_offsets(counts)
    row_of_route, route_of_row = scatter_permutation(ids, mask)
    xs = scatter_rows(x, route_of_row, k)
    h = grouped_swiglu(xs, offsets, weights)
    y = grouped_down(h, offsets, weights)
    out = combine(y, row_of_route, w, T, k)
    return {"ids": ids, "w": w, "counts": counts, "offsets": offsets, "row_of_route": row_of_route,
            "route_of_row": route_of_row, "xs": xs, "h": h, "y": y, "out": out}


# ---------------------------------------------------------------------------
# FP8 E4M3 expert weights (one fp32 scale per output channel)
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(x):
    """Nearest E4M3 value (ties to even), saturating at +-448, as float64."""
    a = _np(x, np.float64)
    out = np.empty_like(a)
    _call("oracle_e4m3_round", _ptr(a), a.size, _ptr(out))
    return out


def round_bf16(x):
    """Nearest bf16 value of each element (ties to even), as float64."""
    a = _np(x, np.float64)
    out = np.empty_like(a)
    _call("oracle_round_bf16", _ptr(a), a.size, _ptr(out))
    return out


def e4m3_encode(v):
    """Byte codes of E4M3 values."""
    a = _np(v, np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    _call("oracle_e4m3_encode", _ptr(a), a.size, _ptr(out))
    return out


def e4m3_decode(code):
    """Values of E4M3 byte codes."""
    c = _np(code, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _call("oracle_e4m3_decode", _ptr(c), c.size, _ptr(out))
    return out


def quantize_weights_fp8(w):
    """Per-row FP8 E4M3 quantization of a bank [..., M, K] (fp32, or bf16 tensors read exactly).

    Returns (codes uint8 [..., M, K], scales float32 [..., M]).
    """
    data, code = _operand(w)
    K = data.shape[-1]
    rows = data.size // K if K else 0
    codes = np.empty(data.shape, dtype=np.uint8)
    scales = np.empty(data.shape[:-1], dtype=np.float32)
    _call("oracle_quantize_fp8", _ptr(data), code, rows, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_bank_fp8(w) -> QuantizedBank:
    return QuantizedBank(*quantize_weights_fp8(w))


def dequantize_weights_fp8(codes, scales):
    """scale * value(code), float64 [..., M, K]."""
    c = _np(codes, np.uint8)
    s = _np(scales, np.float32)
    K = c.shape[-1]
    out = np.empty(c.shape, dtype=np.float64)
    _call("oracle_dequantize_fp8", _ptr(c), _ptr(s), c.size // K if K else 0, K, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# 4-bit weights: E2M1 codes, an E4M3 scale per 16 values, an fp32 scale per row
# ---------------------------------------------------------------------------

def e2m1_round(x):
    """Nearest E2M1 value (ties to even), saturating at +-6, as float64."""
    a = _np(x, np.float64)
    out = np.empty_like(a)
    _call("oracle_e2m1_round", _ptr(a), a.size, _ptr(out))
    return out


def e2m1_encode(v):
    """4-bit codes (in uint8) of E2M1 values."""
    a = _np(v, np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    _call("oracle_e2m1_encode", _ptr(a), a.size, _ptr(out))
    return out


def e2m1_decode(code):
    """Values of 4-bit E2M1 codes (the low nibble of each uint8)."""
    c = _np(code, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _call("oracle_e2m1_decode", _ptr(c), c.size, _ptr(out))
    return out


def quantize_weights_fp4(w):
    """4-bit block-scaled quantization of rows [..., M, K] (K a multiple of 16).

    Returns (codes uint8 [..., M, K/2], block scales uint8 [..., M, K/16], scales float32 [..., M]).
    """
    data, code = _operand(w)
    K = data.shape[-1]
    rows = data.size // K if K else 0
    codes = np.empty(data.shape[:-1] + (K // 2,), dtype=np.uint8)
    bs = np.empty(data.shape[:-1] + (K // 16,), dtype=np.uint8)
    scales = np.empty(data.shape[:-1], dtype=np.float32)
    _call("oracle_quantize_fp4", _ptr(data), code, rows, K, _ptr(codes), _ptr(bs), _ptr(scales))
    return codes, bs, scales


def quantize_bank_fp4(w) -> Fp4Bank:
    return Fp4Bank(*quantize_weights_fp4(w))


def dequantize_weights_fp4(codes, block_scales, scales):
    """scale * block scale * value(code), float64 [..., M, K]."""
    c = _np(codes, np.uint8)
    b = _np(block_scales, np.uint8)
    sc = _np(scales, np.float32)
    K = 2 * c.shape[-1]
    out = np.empty(c.shape[:-1] + (K,), dtype=np.float64)
    _call("oracle_dequantize_fp4", _ptr(c), _ptr(b), _ptr(sc), sc.size, K, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# FP8 E4M3 weights and activations
# ---------------------------------------------------------------------------
#
# Both operands of every expert GEMM are E4M3 codes with one fp32 scale per
# row, made by the quantizer above: the weights per output channel, the
# token rows x per token, the rows of h per compact row.  h is rounded to
# bf16 (the intermediate the GPU stores) before its rows are quantized.  The
# FFN then runs on the values the codes stand for, in float64.

def moe_forward_w8a8(logits, x, weights_q, k: int, mask=None, h_decided=None):
    """Every intermediate of the FP8-activation path for one chunk (A1 .. A7 in order), as a dict.

    weights_q: (gate, up, down) QuantizedBanks, or fetch(e0, e1) returning them.
    h_decided: the bf16 h [R][f] of the implementation under test, or None.  The E4M3 codes of h are an
    integer decision taken from a floating-point h; where an implementation's h is given, the codes are
    decided from it (in that implementation's precision), so that a one-ulp difference of h at an E4M3
    rounding midpoint is not mistaken for an error of what follows.  Its agreement with this oracle's own
    h is for the caller to check (res["h"]).
    """
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids, w = route_topk(lg, k)
    counts = route_histogram(ids, mask, E)
    offsets = prefix_offsets(counts)
    row_of_route, route_of_row = scatter_permutation(ids, mask)
    x_q = quantize_bank_fp8(x)
    xs = scatter_rows(dequantize_weights_fp8(x_q.codes, x_q.scales), route_of_row, k)
    h = grouped_swiglu(xs, offsets, weights_q)
    h_bf16 = round_bf16(h) if h_decided is None else h_decided
    h_q = quantize_bank_fp8(h_bf16)
    y = grouped_down(dequantize_weights_fp8(h_q.codes, h_q.scales), offsets, weights_q)
    out = combine(y, row_of_route, w, T, k)
    return {"ids": ids, "w": w, "counts": counts, "offsets": offsets, "row_of_route": row_of_route,
            "route_of_row": route_of_row, "x_q": x_q, "h": h, "h_bf16": h_bf16, "h_q": h_q, "y": y, "out": out}


def moe_forward_w4a4(logits, x, weights_q, k: int, mask=None, h_decided=None):
    """Every intermediate of the 4-bit-activation path for one chunk (A1 .. A7 in order), as a dict.

    The FP8-activation path with the 4-bit block-scaled format in place of E4M3: the token rows and the
    bf16 rows of h are quantized by the weights' 4-bit quantizer and the FFN runs on the values the codes
    stand for.  weights_q: (gate, up, down) Fp4Banks, or fetch(e0, e1) returning them.  h_decided: as for
    moe_forward_w8a8 (the codes of h decided from the implementation's own bf16 h).
    """
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids, w = route_topk(lg, k)
    counts = route_histogram(ids, mask, E)
    offsets = prefix_offsets(counts)
    row_of_route, route_of_row = scatter_permutation(ids, mask)
    x_q = quantize_bank_fp4(x)
    xs = scatter_rows(dequantize_weights_fp4(x_q.codes, x_q.block_scales, x_q.scales), route_of_row, k)
    h = grouped_swiglu(xs, offsets, weights_q)
    h_bf16 = round_bf16(h) if h_decided is None else h_decided
    h_q = quantize_bank_fp4(h_bf16)
    y = grouped_down(dequantize_weights_fp4(h_q.codes, h_q.block_scales, h_q.scales), offsets, weights_q)
    out = combine(y, row_of_route, w, T, k)
    return {"ids": ids, "w": w, "counts": counts, "offsets": offsets, "row_of_route": row_of_route,
            "route_of_row": route_of_row, "x_q": x_q, "h": h, "h_bf16": h_bf16, "h_q": h_q, "y": y, "out": out}


# ---------------------------------------------------------------------------
# The router projection in front of A1
# ---------------------------------------------------------------------------

def router_logits(x, wr):
    """logits [T][E] float64 = x [T][d] . wr [E][d]^T."""
    xa, xc = _operand(x)
    wa, wc = _operand(wr)
    T, d = xa.shape
    E = wa.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _call("oracle_router_logits", _ptr(xa), xc, _ptr(wa), wc, T, E, d, _ptr(out))
    return out


def route_from_router(x, wr, k: int):
    """Logits, ids and gate weights of the router step followed by A1."""
    logits = router_logits(x, wr)
    ids, w = route_topk(logits, k)
    return logits, ids, w
