"""Python binding of the C-ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but check tensor dtypes/shapes/devices, pass raw device pointers and
the current CUDA stream, and turn a non-zero status into ``MoEError``.  All
arithmetic of the path runs in the library's CUDA kernels; PyTorch only owns
the device memory and the stream.  If the shared library is missing the
import of this module fails: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_RANGE = range(6)
MOE_F32, MOE_BF16 = 0, 1
MOE_FUSED_AUTO, MOE_FUSED_GATHER, MOE_FUSED_COMPACT, MOE_FUSED_NONE = 0, 1, 2, 3

# (name, argtypes) of every exported entry point; the ABI test checks this
# list against include/moe.h.
_P, _I, _L, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "moe_version": ([], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_last_cuda_error": ([], _I),
    "moe_check_device_error": ([_P], _I),
    "moe_selftest_bounded_wait": ([_I, _P], _I),
    "moe_workspace_size": ([_I, _I, _SZ], _I),
    "moe_route_topk": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_router_topk": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_route_histogram": ([_P, _P, _I, _I, _I, _P, _P, _P], _I),
    "moe_route_histogram_noalloc": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "moe_prefix_offsets": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_scatter_rows": ([_P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_scatter_rows_f16": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_route_scatter_small": ([_P, _P, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gate_up": ([_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P], _I),
    "moe_grouped_down": ([_P, _P, _I, _I, _I, _I, _P, _I, _P, _P], _I),
    "moe_grouped_ffn": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P], _I),
    "moe_combine": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_forward": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _I,
                     _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_quantize_weights_fp8": ([_P, _I, _L, _I, _P, _P, _P], _I),
    "moe_grouped_gate_up_fp8": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_down_fp8": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_ffn_fp8": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_forward_fp8": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                         _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_tile_counts_size": ([_I, _I, _SZ], _I),
    "moe_scatter_index": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_route_scatter_small_fused": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gate_up_gather": ([_P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_down_combine": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_forward_fused": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _I,
                           _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_clear_device_error": ([_P], _I),
    "moe_quantize_weights_fp4": ([_P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_gate_up_fp4": ([_P, _P, _I, _I, _I, _I] + [_P] * 8, _I),
    "moe_grouped_down_fp4": ([_P, _P, _I, _I, _I, _I] + [_P] * 5, _I),
    "moe_forward_fp4": ([_P, _P, _P, _I, _I, _I, _I, _I] + [_P] * 9 + [_P] * 12, _I),
    "moe_scatter_rows_e4m3": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_scatter_rows_quant_e4m3": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_quantize_rows_e4m3": ([_P, _P, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gate_up_w8a8": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_down_w8a8": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_forward_w8a8": ([_P, _P, _P, _I, _I, _I, _I, _I] + [_P] * 6 + [_P] * 17, _I),
    "moe_quantize_rows_fp4": ([_P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_scatter_rows_fp4": ([_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P], _I),
    "moe_scatter_rows_quant_fp4": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P],
                                   _I),
    "moe_route_scatter_quant_small_e4m3": ([_P, _P, _P, _I, _I, _I, _I] + [_P] * 11, _I),
    "moe_route_scatter_quant_small_fp4": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P,
                                           _P, _P, _P], _I),
    "moe_grouped_gate_up_w4a4": ([_P, _P, _I, _P, _P, _I, _I, _I, _I] + [_P] * 8, _I),
    "moe_grouped_down_w4a4": ([_P, _P, _I, _P, _P, _I, _I, _I, _I] + [_P] * 5, _I),
    "moe_forward_w4a4": ([_P, _P, _P, _I, _I, _I, _I, _I] + [_P] * 9 + [_P] * 20, _I),
    "moe_route_topk_offsets": ([_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_forward_fused_mode": ([_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)], _I),
    "moe_ffn_paired": ([_I, ctypes.POINTER(ctypes.c_int)], _I),
    "moe_plan_create": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                         ctypes.POINTER(ctypes.c_void_p)], _I),
    "moe_plan_destroy": ([_P], _I),
    "moe_plan_grouped_gate_up": ([_P, _P], _I),
    "moe_plan_grouped_down": ([_P, _P], _I),
    "moe_plan_forward": ([_P, _P, _P, _P, _P, _P], _I),
}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load()
        msg = lib.moe_status_string(status).decode()
        if status == MOE_ERR_CUDA:
            msg += f" (cudaError {lib.moe_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load the shared library (raises OSError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with `python -m sparse_moe_expert_top_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


class _Recorder:
    """Stands in for the library while `bind` marshals a call: records the C calls instead of making them."""

    def __init__(self, lib):
        self._real = lib
        self.calls = []

    def __getattr__(self, name):
        real = getattr(self._real, name)

        def record(*args):
            self.calls.append((name, real, args))
            return MOE_OK

        return record


def bind(fn, *args, **kwargs):
    """Marshal one call of a binding function now and return a zero-argument
    callable that makes the same C call(s) again (same pointers, sizes and
    stream) without repeating the Python-side checks.  Meant for timed loops
    of tiny batches, where the checks would cost more than the kernels.  The
    callable keeps references to the arguments, so the tensors behind the
    recorded pointers stay allocated as long as it lives."""
    global _lib
    lib = load()
    rec = _Recorder(lib)
    _lib = rec
    try:
        fn(*args, **kwargs)
    finally:
        _lib = lib
    calls = rec.calls
    keep = (args, kwargs)   # the recorded pointers stay valid while the callable lives

    def run():
        assert keep is not None
        for name, f, a in calls:
            status = f(*a)
            if status != MOE_OK:
                raise MoEError(name, status)

    return run


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise ValueError(f"unsupported operand dtype {t.dtype}")


def _expect(t, dtype, shape, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def moe_version() -> int:
    return load().moe_version()


def moe_check_device_error(stream=None) -> None:
    _check("moe_check_device_error", load().moe_check_device_error(_stream(stream)))


def moe_clear_device_error(stream=None) -> None:
    """Enqueue the clearing of the device error word on the stream (no synchronisation)."""
    _check("moe_clear_device_error", load().moe_clear_device_error(_stream(stream)))


def moe_selftest_bounded_wait(limit_ms: int, stream=None) -> None:
    """Run one bounded wait that is bound to run out (see include/moe.h)."""
    _check("moe_selftest_bounded_wait", load().moe_selftest_bounded_wait(limit_ms, _stream(stream)))


def moe_workspace_size(T: int, k: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", load().moe_workspace_size(T, k, ctypes.byref(n)))
    return n.value


def moe_route_topk(logits, k, ids, w, stream=None):
    T, E = logits.shape
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(w, torch.float32, (T, k), "w")
    _check("moe_route_topk", load().moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream(stream)))


def moe_router_topk(x, wr, k, ids, w, logits=None, stream=None):
    """Router logits x . wr^T (bf16, fp32 accumulation) and their top-k routing; logits optional."""
    T, d = x.shape
    E = wr.shape[0]
    _expect(x, torch.bfloat16, (T, d), "x")
    _expect(wr, torch.bfloat16, (E, d), "wr")
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(w, torch.float32, (T, k), "w")
    if logits is not None:
        _expect(logits, torch.float32, (T, E), "logits")
    _check("moe_router_topk", load().moe_router_topk(_ptr(x), _ptr(wr), T, E, d, k, _ptr(logits), _ptr(ids), _ptr(w),
                                                     _stream(stream)))


def moe_route_histogram(ids, mask, E, counts, ws, stream=None):
    T, k = ids.shape
    _expect(ids, torch.int32, (T, k), "ids")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect(counts, torch.int32, (E,), "counts")
    _check("moe_route_histogram", load().moe_route_histogram(_ptr(ids), _ptr(mask), T, k, E, _ptr(counts), _ptr(ws),
                                                             _stream(stream)))


def moe_route_topk_offsets(logits, mask, k, ids, w, counts, offsets, ws, stream=None):
    """A1-A3 in one launch (moe_route_topk + moe_route_histogram + moe_prefix_offsets)."""
    T, E = logits.shape
    _expect(logits, torch.float32, (T, E), "logits")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(w, torch.float32, (T, k), "w")
    _expect(counts, torch.int32, (E,), "counts")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_route_topk_offsets", load().moe_route_topk_offsets(
        _ptr(logits), _ptr(mask), T, E, k, _ptr(ids), _ptr(w), _ptr(counts), _ptr(offsets), _ptr(ws),
        _stream(stream)))


def moe_route_histogram_noalloc(ids, mask, E, counts, stream=None):
    """moe_route_histogram without a workspace: for callers that cannot allocate device memory.

    The scratch is a static device array in the library (T*k <= 65536);
    calls that overlap on the GPU race, so serialise them.
    """
    T, k = ids.shape
    _expect(ids, torch.int32, (T, k), "ids")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect(counts, torch.int32, (E,), "counts")
    _check("moe_route_histogram_noalloc", load().moe_route_histogram_noalloc(_ptr(ids), _ptr(mask), T, k, E,
                                                                             _ptr(counts), _stream(stream)))


def moe_prefix_offsets(counts, T, k, offsets, ws, stream=None):
    E = counts.shape[0]
    _expect(counts, torch.int32, (E,), "counts")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_prefix_offsets", load().moe_prefix_offsets(_ptr(counts), T, k, E, _ptr(offsets), _ptr(ws),
                                                           _stream(stream)))


def moe_scatter_rows(x, ids, mask, offsets, xs, row_of_route, route_of_row, ws, stream=None):
    T, d = x.shape
    k = ids.shape[1]
    E = offsets.shape[0] - 1
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(xs, x.dtype, (T * k, d), "xs")
    _expect(row_of_route, torch.int32, (T * k,), "row_of_route")
    _expect(route_of_row, torch.int32, (T * k,), "route_of_row")
    _check("moe_scatter_rows", load().moe_scatter_rows(_ptr(x), _dtype_code(x), _ptr(ids), _ptr(mask), _ptr(offsets),
                                                       T, k, d, E, _ptr(xs), _ptr(row_of_route), _ptr(route_of_row),
                                                       _ptr(ws), _stream(stream)))


def moe_scatter_rows_f16(x, ids, mask, offsets, xs, row_of_route, route_of_row, ws, stream=None):
    """moe_scatter_rows for the FP8-weight path: bf16 x in, fp16 compact rows out."""
    T, d = x.shape
    k = ids.shape[1]
    E = offsets.shape[0] - 1
    _expect(x, torch.bfloat16, (T, d), "x")
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(xs, torch.float16, (T * k, d), "xs")
    _expect(row_of_route, torch.int32, (T * k,), "row_of_route")
    _expect(route_of_row, torch.int32, (T * k,), "route_of_row")
    _check("moe_scatter_rows_f16", load().moe_scatter_rows_f16(
        _ptr(x), _ptr(ids), _ptr(mask), _ptr(offsets), T, k, d, E, _ptr(xs), _ptr(row_of_route),
        _ptr(route_of_row), _ptr(ws), _stream(stream)))


def moe_route_scatter_small(logits, x, mask, k, bufs, stream=None):
    """A1-A4 in one launch for a small chunk (T <= 128, T*k <= 512) into ``bufs``.

    ``bufs.xs`` is fp16 (FP8-weight path, x bf16) or of x's type."""
    T, E = logits.shape
    d = x.shape[1]
    b = bufs
    _expect(logits, torch.float32, (T, E), "logits")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    xs_f16 = b.xs.dtype == torch.float16 and x.dtype == torch.bfloat16
    if not xs_f16:
        _expect(b.xs, x.dtype, (T * k, d), "xs")
    _check("moe_route_scatter_small", load().moe_route_scatter_small(
        _ptr(logits), _ptr(x), _dtype_code(x), 1 if xs_f16 else 0, _ptr(mask), T, E, k, d, _ptr(b.ids), _ptr(b.w),
        _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route), _ptr(b.route_of_row),
        _stream(stream)))


def moe_grouped_gate_up(xs, offsets, w_gate, w_up, h, stream=None):
    cap, d = xs.shape
    E, f, _ = w_gate.shape
    _expect(w_gate, xs.dtype, (E, f, d), "w_gate")
    _expect(w_up, xs.dtype, (E, f, d), "w_up")
    _expect(h, xs.dtype, (cap, f), "h")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_grouped_gate_up", load().moe_grouped_gate_up(_ptr(xs), _ptr(offsets), cap, E, d, f, _ptr(w_gate),
                                                             _ptr(w_up), _dtype_code(xs), _ptr(h), _stream(stream)))


def moe_grouped_down(h, offsets, w_down, y, stream=None):
    cap, f = h.shape
    E, d, _ = w_down.shape
    _expect(w_down, h.dtype, (E, d, f), "w_down")
    _expect(y, torch.float32, (cap, d), "y")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_grouped_down", load().moe_grouped_down(_ptr(h), _ptr(offsets), cap, E, d, f, _ptr(w_down),
                                                       _dtype_code(h), _ptr(y), _stream(stream)))


def moe_grouped_ffn(xs, offsets, w_gate, w_up, w_down, h, y, stream=None):
    cap, d = xs.shape
    E, f, _ = w_gate.shape
    _expect(w_gate, xs.dtype, (E, f, d), "w_gate")
    _expect(w_up, xs.dtype, (E, f, d), "w_up")
    _expect(w_down, xs.dtype, (E, d, f), "w_down")
    _expect(h, xs.dtype, (cap, f), "h")
    _expect(y, torch.float32, (cap, d), "y")
    _check("moe_grouped_ffn", load().moe_grouped_ffn(_ptr(xs), _ptr(offsets), cap, E, d, f, _ptr(w_gate), _ptr(w_up),
                                                     _ptr(w_down), _dtype_code(xs), _ptr(h), _ptr(y), _stream(stream)))


def moe_combine(y, row_of_route, w, out, stream=None):
    T, k = w.shape
    d = out.shape[1]
    _expect(y, torch.float32, (y.shape[0], d), "y")
    _expect(row_of_route, torch.int32, (T * k,), "row_of_route")
    _expect(out, torch.float32, (T, d), "out")
    _check("moe_combine", load().moe_combine(_ptr(y), _ptr(row_of_route), _ptr(w), T, k, d, _ptr(out),
                                             _stream(stream)))


class MoEBuffers:
    """Caller-owned device buffers for one chunk shape (T, E, k, d, f, dtype).

    The library never allocates; this helper allocates every intermediate
    of the path once with PyTorch so that repeated calls reuse them.
    """

    def __init__(self, T: int, E: int, k: int, d: int, f: int, dtype: torch.dtype, device="cuda"):
        self.T, self.E, self.k, self.d, self.f, self.dtype = T, E, k, d, f, dtype
        cap = T * k
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.empty(T, k, **i32)
        self.w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.xs = torch.empty(cap, d, dtype=dtype, device=device)
        self.row_of_route = torch.empty(cap, **i32)
        self.route_of_row = torch.empty(cap, **i32)
        self.h = torch.empty(cap, f, dtype=dtype, device=device)
        self.y = torch.empty(cap, d, dtype=torch.float32, device=device)
        self.out = torch.empty(T, d, dtype=torch.float32, device=device)
        # the workspace must start zero-filled (it keeps a completion counter)
        self.ws = torch.zeros(max(moe_workspace_size(T, k), 16) // 4 + 4, dtype=torch.int32, device=device)
        # slot counters of the fused combine (moe_forward_fused)
        self.tile_counts = torch.zeros(max(moe_tile_counts_size(T, d), 4) // 4, dtype=torch.int32, device=device)


def moe_forward(logits, x, mask, w_gate, w_up, w_down, k: int, bufs: MoEBuffers, stream=None) -> torch.Tensor:
    """The whole path on the current stream; returns ``bufs.out`` ([T][d] fp32)."""
    T, E = logits.shape
    d = x.shape[1]
    f = w_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f, bufs.dtype) != (T, E, k, d, f, x.dtype):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect(w_gate, x.dtype, (E, f, d), "w_gate")
    _expect(w_up, x.dtype, (E, f, d), "w_up")
    _expect(w_down, x.dtype, (E, d, f), "w_down")
    b = bufs
    _check("moe_forward", load().moe_forward(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f, _ptr(w_gate), _ptr(w_up), _ptr(w_down), _dtype_code(x),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route),
        _ptr(b.route_of_row), _ptr(b.h), _ptr(b.y), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out


# ---------------------------------------------------------------------------
# Fused permutation (bf16): row gather in the gate/up kernel, combine in the
# down kernel
# ---------------------------------------------------------------------------

def moe_tile_counts_size(T: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_tile_counts_size", load().moe_tile_counts_size(T, d, ctypes.byref(n)))
    return n.value


def moe_scatter_index(ids, mask, offsets, d, row_of_route, route_of_row, tile_counts, out, ws, x=None, xs=None,
                      stream=None):
    """A4 with the fused combine's preparation: clears ``tile_counts``, zeroes ``out`` rows of all-masked
    tokens; copies the compact rows ``xs`` only when ``x`` and ``xs`` are given."""
    T, k = ids.shape
    E = offsets.shape[0] - 1
    if (x is None) != (xs is None):
        raise ValueError("give both x and xs, or neither")
    if x is not None:
        _expect(x, torch.bfloat16, (T, d), "x")
        _expect(xs, torch.bfloat16, (T * k, d), "xs")
    _expect(ids, torch.int32, (T, k), "ids")
    _expect(row_of_route, torch.int32, (T * k,), "row_of_route")
    _expect(route_of_row, torch.int32, (T * k,), "route_of_row")
    _expect(out, torch.float32, (T, d), "out")
    if tile_counts.dtype != torch.int32 or tile_counts.numel() * 4 < moe_tile_counts_size(T, d):
        raise ValueError("tile_counts: expected int32 of moe_tile_counts_size(T, d) bytes")
    _check("moe_scatter_index", load().moe_scatter_index(
        _ptr(ids), _ptr(mask), _ptr(offsets), T, k, d, E, _ptr(x), _ptr(xs), _ptr(row_of_route),
        _ptr(route_of_row), _ptr(tile_counts), _ptr(out), _ptr(ws), _stream(stream)))


def moe_route_scatter_small_fused(logits, x, mask, k, bufs, gather: bool = True, stream=None):
    """A1-A4 in one launch for a small chunk, with the fused combine's preparation (bf16 x); copies the
    compact rows into ``bufs.xs`` only when ``gather`` is False."""
    T, E = logits.shape
    d = x.shape[1]
    b = bufs
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _check("moe_route_scatter_small_fused", load().moe_route_scatter_small_fused(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets),
        None if gather else _ptr(b.xs), _ptr(b.row_of_route), _ptr(b.route_of_row), _ptr(b.tile_counts),
        _ptr(b.out), _stream(stream)))


def moe_grouped_gate_up_gather(x, k, route_of_row, offsets, w_gate, w_up, h, stream=None):
    """A5 reading token rows of x through route_of_row (no compact copy)."""
    T, d = x.shape
    E, f, _ = w_gate.shape
    _expect(x, torch.bfloat16, (T, d), "x")
    _expect(route_of_row, torch.int32, (T * k,), "route_of_row")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _expect(w_gate, torch.bfloat16, (E, f, d), "w_gate")
    _expect(w_up, torch.bfloat16, (E, f, d), "w_up")
    _expect(h, torch.bfloat16, (T * k, f), "h")
    _check("moe_grouped_gate_up_gather", load().moe_grouped_gate_up_gather(
        _ptr(x), T, k, _ptr(route_of_row), _ptr(offsets), E, d, f, _ptr(w_gate), _ptr(w_up), _ptr(h),
        _stream(stream)))


def moe_grouped_down_combine(h, offsets, w_down, route_of_row, row_of_route, w, y, tile_counts, out, stream=None):
    """A6 + A7 in one kernel; ``y`` is scratch, ``tile_counts`` must be zero (moe_scatter_index)."""
    T, k = w.shape
    cap, f = h.shape
    E, d, _ = w_down.shape
    _expect(h, torch.bfloat16, (T * k, f), "h")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _expect(w_down, torch.bfloat16, (E, d, f), "w_down")
    _expect(route_of_row, torch.int32, (T * k,), "route_of_row")
    _expect(row_of_route, torch.int32, (T * k,), "row_of_route")
    _expect(w, torch.float32, (T, k), "w")
    _expect(y, torch.float32, (T * k, d), "y")
    _expect(out, torch.float32, (T, d), "out")
    if tile_counts.dtype != torch.int32 or tile_counts.numel() * 4 < moe_tile_counts_size(T, d):
        raise ValueError("tile_counts: expected int32 of moe_tile_counts_size(T, d) bytes")
    _check("moe_grouped_down_combine", load().moe_grouped_down_combine(
        _ptr(h), _ptr(offsets), T, k, E, d, f, _ptr(w_down), _ptr(route_of_row), _ptr(row_of_route), _ptr(w),
        _ptr(y), _ptr(tile_counts), _ptr(out), _stream(stream)))


def moe_forward_fused(logits, x, mask, w_gate, w_up, w_down, k: int, bufs: MoEBuffers, mode: int = MOE_FUSED_AUTO,
                      stream=None) -> torch.Tensor:
    """The whole path with the fused combine (bf16); returns ``bufs.out``.  ``mode``: MOE_FUSED_AUTO,
    MOE_FUSED_GATHER (rows gathered by the gate/up kernel, ``bufs.xs`` unused), MOE_FUSED_COMPACT or
    MOE_FUSED_NONE (the unfused path).  ``bufs.y`` is scratch."""
    T, E = logits.shape
    d = x.shape[1]
    f = w_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f, bufs.dtype) != (T, E, k, d, f, torch.bfloat16):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect(w_gate, torch.bfloat16, (E, f, d), "w_gate")
    _expect(w_up, torch.bfloat16, (E, f, d), "w_up")
    _expect(w_down, torch.bfloat16, (E, d, f), "w_down")
    b = bufs
    _check("moe_forward_fused", load().moe_forward_fused(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f, _ptr(w_gate), _ptr(w_up), _ptr(w_down), int(mode),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route),
        _ptr(b.route_of_row), _ptr(b.h), _ptr(b.y), _ptr(b.tile_counts), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out


# ---------------------------------------------------------------------------
# FP8 E4M3 expert weights (one fp32 scale per output channel)
# ---------------------------------------------------------------------------

class FP8Weights:
    """Rows in FP8 E4M3: ``codes`` uint8 [..., rows, K] and one fp32 scale per row, ``scales`` [..., rows]
    (an expert bank [E][rows][K], or activation rows [rows][K])."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor):
        if codes.dtype != torch.uint8 or scales.dtype != torch.float32 or codes.dim() < 2:
            raise ValueError("expected uint8 codes [..., rows, K] and fp32 scales [..., rows]")
        if tuple(scales.shape) != tuple(codes.shape[:-1]):
            raise ValueError(f"scales {tuple(scales.shape)} do not match codes {tuple(codes.shape)}")
        self.codes, self.scales = codes, scales

    @property
    def shape(self):
        return self.codes.shape


def moe_quantize_weights_fp8(w, codes=None, scales=None, stream=None) -> FP8Weights:
    """Quantize rows (a bank [E][rows][K], or activation rows [rows][K]; bf16 or fp32) to FP8 E4M3 codes and
    one scale per row."""
    if w.dim() < 2:
        raise ValueError("expected rows [..., rows, K]")
    K = w.shape[-1]
    n_rows = w.numel() // K if K else 0
    if codes is None:
        codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _expect(codes, torch.uint8, tuple(w.shape), "codes")
    _expect(scales, torch.float32, tuple(w.shape[:-1]), "scales")
    _check("moe_quantize_weights_fp8", load().moe_quantize_weights_fp8(
        _ptr(w), _dtype_code(w), n_rows, K, _ptr(codes), _ptr(scales), _stream(stream)))
    return FP8Weights(codes, scales)


def _expect_fp8(q, shape, name):
    if not isinstance(q, FP8Weights):
        raise ValueError(f"{name}: expected FP8Weights")
    _expect(q.codes, torch.uint8, shape, name + ".codes")
    _expect(q.scales, torch.float32, shape[:2], name + ".scales")


def moe_grouped_gate_up_fp8(xs, offsets, q_gate: FP8Weights, q_up: FP8Weights, h, stream=None):
    cap, d = xs.shape
    E, f, _ = q_gate.shape
    _expect(xs, torch.float16, (cap, d), "xs")
    _expect_fp8(q_gate, (E, f, d), "q_gate")
    _expect_fp8(q_up, (E, f, d), "q_up")
    _expect(h, torch.float16, (cap, f), "h")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_grouped_gate_up_fp8", load().moe_grouped_gate_up_fp8(
        _ptr(xs), _ptr(offsets), cap, E, d, f, _ptr(q_gate.codes), _ptr(q_gate.scales), _ptr(q_up.codes),
        _ptr(q_up.scales), _ptr(h), _stream(stream)))


def moe_grouped_down_fp8(h, offsets, q_down: FP8Weights, y, stream=None):
    cap, f = h.shape
    E, d, _ = q_down.shape
    _expect(h, torch.float16, (cap, f), "h")
    _expect_fp8(q_down, (E, d, f), "q_down")
    _expect(y, torch.float32, (cap, d), "y")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _check("moe_grouped_down_fp8", load().moe_grouped_down_fp8(
        _ptr(h), _ptr(offsets), cap, E, d, f, _ptr(q_down.codes), _ptr(q_down.scales), _ptr(y), _stream(stream)))


def moe_grouped_ffn_fp8(xs, offsets, q_gate: FP8Weights, q_up: FP8Weights, q_down: FP8Weights, h, y, stream=None):
    cap, d = xs.shape
    E, f, _ = q_gate.shape
    _expect(xs, torch.float16, (cap, d), "xs")
    _expect_fp8(q_gate, (E, f, d), "q_gate")
    _expect_fp8(q_up, (E, f, d), "q_up")
    _expect_fp8(q_down, (E, d, f), "q_down")
    _expect(h, torch.float16, (cap, f), "h")
    _expect(y, torch.float32, (cap, d), "y")
    _check("moe_grouped_ffn_fp8", load().moe_grouped_ffn_fp8(
        _ptr(xs), _ptr(offsets), cap, E, d, f, _ptr(q_gate.codes), _ptr(q_gate.scales), _ptr(q_up.codes),
        _ptr(q_up.scales), _ptr(q_down.codes), _ptr(q_down.scales), _ptr(h), _ptr(y), _stream(stream)))


def moe_forward_fp8(logits, x, mask, q_gate: FP8Weights, q_up: FP8Weights, q_down: FP8Weights, k: int,
                    bufs: MoEBuffers, stream=None) -> torch.Tensor:
    """The whole path with FP8 expert weights; returns ``bufs.out`` ([T][d] fp32).

    x is bf16; ``bufs`` holds fp16 compact activations (``MoEBuffers(..., torch.float16)``).
    """
    T, E = logits.shape
    d = x.shape[1]
    f = q_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f, bufs.dtype) != (T, E, k, d, f, torch.float16):
        raise ValueError("buffers were allocated for another shape (the FP8 path keeps xs and h in fp16)")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect_fp8(q_gate, (E, f, d), "q_gate")
    _expect_fp8(q_up, (E, f, d), "q_up")
    _expect_fp8(q_down, (E, d, f), "q_down")
    b = bufs
    _check("moe_forward_fp8", load().moe_forward_fp8(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f, _ptr(q_gate.codes), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.scales), _ptr(q_down.codes), _ptr(q_down.scales),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route),
        _ptr(b.route_of_row), _ptr(b.h), _ptr(b.y), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out


def moe_ffn_paired(cap: int) -> bool:
    """Whether the bf16 and E4M3 grouped projections run on pairs of SMs for `cap` compact rows."""
    paired = ctypes.c_int(-1)
    _check("moe_ffn_paired", load().moe_ffn_paired(cap, ctypes.byref(paired)))
    return paired.value == 1


def moe_forward_fused_mode(T: int, E: int, k: int, d: int, have_xs: bool = True) -> int:
    """The mode moe_forward_fused picks for MOE_FUSED_AUTO on the current device."""
    mode = ctypes.c_int(-1)
    _check("moe_forward_fused_mode", load().moe_forward_fused_mode(T, E, k, d, 1 if have_xs else 0,
                                                                   ctypes.byref(mode)))
    return mode.value


# ---------------------------------------------------------------------------
# Plans: shapes, weights and buffers fixed, host work done once
# ---------------------------------------------------------------------------

class MoEPlan:
    """A moe_plan handle with the tensors behind its pointers (kept alive while the plan lives)."""

    def __init__(self, handle, keep):
        self._handle = handle
        self._keep = keep

    @property
    def handle(self):
        return self._handle

    def close(self):
        if self._handle is not None and _lib is not None:
            load().moe_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def moe_plan_create(w_gate, w_up, w_down, bufs: MoEBuffers) -> MoEPlan:
    """A plan for chunks of bufs.T tokens with these weights and buffers (see include/moe.h)."""
    b = bufs
    T, E, k, d, f = b.T, b.E, b.k, b.d, b.f
    _expect(w_gate, b.dtype, (E, f, d), "w_gate")
    _expect(w_up, b.dtype, (E, f, d), "w_up")
    _expect(w_down, b.dtype, (E, d, f), "w_down")
    handle = ctypes.c_void_p()
    _check("moe_plan_create", load().moe_plan_create(
        T, E, k, d, f, _dtype_code(w_gate), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(b.ids), _ptr(b.w),
        _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route), _ptr(b.route_of_row), _ptr(b.h),
        _ptr(b.y), _ptr(b.ws), ctypes.byref(handle)))
    return MoEPlan(handle, (w_gate, w_up, w_down, b))


def moe_plan_grouped_gate_up(plan: MoEPlan, stream=None):
    _check("moe_plan_grouped_gate_up", load().moe_plan_grouped_gate_up(plan.handle, _stream(stream)))


def moe_plan_grouped_down(plan: MoEPlan, stream=None):
    _check("moe_plan_grouped_down", load().moe_plan_grouped_down(plan.handle, _stream(stream)))


def moe_plan_forward(plan: MoEPlan, logits, x, mask, out=None, stream=None) -> torch.Tensor:
    """moe_forward through the plan; returns out (default: the plan's bufs.out)."""
    b = plan._keep[3]
    out = b.out if out is None else out
    _expect(logits, torch.float32, (b.T, b.E), "logits")
    _expect(x, b.dtype, (b.T, b.d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (b.T, b.k), "mask")
    _expect(out, torch.float32, (b.T, b.d), "out")
    _check("moe_plan_forward", load().moe_plan_forward(plan.handle, _ptr(logits), _ptr(x), _ptr(mask), _ptr(out),
                                                       _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# FP8 E4M3 weights and activations (kind::f8f6f4 tensor-core MMAs)
# ---------------------------------------------------------------------------

class MoEBuffersW8A8:
    """Caller-owned device buffers of the FP8-activation path for one chunk shape (bf16 x)."""

    def __init__(self, T: int, E: int, k: int, d: int, f: int, device="cuda"):
        self.T, self.E, self.k, self.d, self.f = T, E, k, d, f
        cap = T * k
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.empty(T, k, **i32)
        self.w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.x_q = torch.empty(T, d, dtype=torch.uint8, device=device)
        self.x_scales = torch.empty(T, dtype=torch.float32, device=device)
        self.xs = torch.empty(cap, d, dtype=torch.uint8, device=device)
        self.xs_scales = torch.empty(cap, dtype=torch.float32, device=device)
        self.row_of_route = torch.empty(cap, **i32)
        self.route_of_row = torch.empty(cap, **i32)
        self.h = torch.empty(cap, f, dtype=torch.bfloat16, device=device)
        self.h_q = torch.empty(cap, f, dtype=torch.uint8, device=device)
        self.h_scales = torch.empty(cap, dtype=torch.float32, device=device)
        self.y = torch.empty(cap, d, dtype=torch.float32, device=device)
        self.out = torch.empty(T, d, dtype=torch.float32, device=device)
        self.ws = torch.zeros(max(moe_workspace_size(T, k), 16) // 4 + 4, dtype=torch.int32, device=device)


def moe_scatter_rows_e4m3(x_q, x_scales, ids, mask, offsets, xs, xs_scales, row_of_route, route_of_row, ws,
                          stream=None):
    T, d = x_q.shape
    k = ids.shape[1]
    E = offsets.shape[0] - 1
    _expect(x_q, torch.uint8, (T, d), "x_q")
    _expect(x_scales, torch.float32, (T,), "x_scales")
    _expect(xs, torch.uint8, (T * k, d), "xs")
    _expect(xs_scales, torch.float32, (T * k,), "xs_scales")
    _check("moe_scatter_rows_e4m3", load().moe_scatter_rows_e4m3(
        _ptr(x_q), _ptr(x_scales), _ptr(ids), _ptr(mask), _ptr(offsets), T, k, d, E, _ptr(xs), _ptr(xs_scales),
        _ptr(row_of_route), _ptr(route_of_row), _ptr(ws), _stream(stream)))


def moe_route_scatter_quant_small_e4m3(logits, x, mask, k: int, bufs: "MoEBuffersW8A8", stream=None):
    """A1-A4 with E4M3 rows in one launch for small chunks (T <= 128, T*k <= 512), into ``bufs``."""
    T, E = logits.shape
    d = x.shape[1]
    b = bufs
    if (b.T, b.E, b.k, b.d) != (T, E, k, d):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _check("moe_route_scatter_quant_small_e4m3", load().moe_route_scatter_quant_small_e4m3(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets),
        _ptr(b.x_q), _ptr(b.x_scales), _ptr(b.xs), _ptr(b.xs_scales), _ptr(b.row_of_route), _ptr(b.route_of_row),
        _stream(stream)))


def moe_scatter_rows_quant_e4m3(x, ids, mask, offsets, x_q, x_scales, xs, xs_scales, row_of_route, route_of_row,
                                ws, stream=None):
    T, d = x.shape
    k = ids.shape[1]
    E = offsets.shape[0] - 1
    _expect(x, torch.bfloat16, (T, d), "x")
    _expect(x_q, torch.uint8, (T, d), "x_q")
    _expect(x_scales, torch.float32, (T,), "x_scales")
    _expect(xs, torch.uint8, (T * k, d), "xs")
    _expect(xs_scales, torch.float32, (T * k,), "xs_scales")
    _check("moe_scatter_rows_quant_e4m3", load().moe_scatter_rows_quant_e4m3(
        _ptr(x), _ptr(ids), _ptr(mask), _ptr(offsets), T, k, d, E, _ptr(x_q), _ptr(x_scales), _ptr(xs),
        _ptr(xs_scales), _ptr(row_of_route), _ptr(route_of_row), _ptr(ws), _stream(stream)))


def moe_quantize_rows_e4m3(a, offsets, codes, scales, stream=None):
    cap, K = a.shape
    E = offsets.shape[0] - 1
    _expect(a, torch.bfloat16, (cap, K), "a")
    _expect(codes, torch.uint8, (cap, K), "codes")
    _expect(scales, torch.float32, (cap,), "scales")
    _check("moe_quantize_rows_e4m3", load().moe_quantize_rows_e4m3(
        _ptr(a), _ptr(offsets), E, cap, K, _ptr(codes), _ptr(scales), _stream(stream)))


def moe_grouped_gate_up_w8a8(xs, xs_scales, offsets, q_gate: FP8Weights, q_up: FP8Weights, h, stream=None):
    cap, d = xs.shape
    E, f, _ = q_gate.shape
    _expect(xs, torch.uint8, (cap, d), "xs")
    _expect(xs_scales, torch.float32, (cap,), "xs_scales")
    _expect_fp8(q_gate, (E, f, d), "q_gate")
    _expect_fp8(q_up, (E, f, d), "q_up")
    _expect(h, torch.bfloat16, (cap, f), "h")
    _check("moe_grouped_gate_up_w8a8", load().moe_grouped_gate_up_w8a8(
        _ptr(xs), _ptr(xs_scales), _ptr(offsets), cap, E, d, f, _ptr(q_gate.codes), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.scales), _ptr(h), _stream(stream)))


def moe_grouped_down_w8a8(h_q, h_scales, offsets, q_down: FP8Weights, y, stream=None):
    cap, f = h_q.shape
    E, d, _ = q_down.shape
    _expect(h_q, torch.uint8, (cap, f), "h_q")
    _expect(h_scales, torch.float32, (cap,), "h_scales")
    _expect_fp8(q_down, (E, d, f), "q_down")
    _expect(y, torch.float32, (cap, d), "y")
    _check("moe_grouped_down_w8a8", load().moe_grouped_down_w8a8(
        _ptr(h_q), _ptr(h_scales), _ptr(offsets), cap, E, d, f, _ptr(q_down.codes), _ptr(q_down.scales), _ptr(y),
        _stream(stream)))


def moe_forward_w8a8(logits, x, mask, q_gate: FP8Weights, q_up: FP8Weights, q_down: FP8Weights, k: int,
                     bufs: MoEBuffersW8A8, stream=None) -> torch.Tensor:
    """The whole path on E4M3 weights and activations; returns ``bufs.out`` ([T][d] fp32)."""
    T, E = logits.shape
    d = x.shape[1]
    f = q_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f) != (T, E, k, d, f):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect_fp8(q_gate, (E, f, d), "q_gate")
    _expect_fp8(q_up, (E, f, d), "q_up")
    _expect_fp8(q_down, (E, d, f), "q_down")
    b = bufs
    _check("moe_forward_w8a8", load().moe_forward_w8a8(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f, _ptr(q_gate.codes), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.scales), _ptr(q_down.codes), _ptr(q_down.scales),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets), _ptr(b.x_q), _ptr(b.x_scales), _ptr(b.xs),
        _ptr(b.xs_scales), _ptr(b.row_of_route), _ptr(b.route_of_row), _ptr(b.h), _ptr(b.h_q), _ptr(b.h_scales),
        _ptr(b.y), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out


# ---------------------------------------------------------------------------
# 4-bit block-scaled expert weights
# ---------------------------------------------------------------------------

class FP4Weights:
    """One expert bank in the 4-bit format: ``codes`` uint8 [E][M][K/2], ``block_scales`` uint8 [E][K/64][M][4]
    (E4M3), ``scales`` fp32 [E][M]."""

    def __init__(self, codes, block_scales, scales):
        E, M, K2 = codes.shape
        if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or scales.dtype != torch.float32:
            raise ValueError("expected uint8 codes and block scales, fp32 scales")
        if tuple(block_scales.shape) != (E, 2 * K2 // 64, M, 4) or tuple(scales.shape) != (E, M):
            raise ValueError("block scales [E][K/64][M][4] and scales [E][M] do not match the codes")
        self.codes, self.block_scales, self.scales = codes, block_scales, scales

    @property
    def shape(self):
        E, M, K2 = self.codes.shape
        return (E, M, 2 * K2)


def moe_quantize_weights_fp4(w, stream=None) -> FP4Weights:
    """Quantize a bank [E][M][K] (bf16 or fp32, K a multiple of 64) to the 4-bit block-scaled format."""
    E, M, K = w.shape
    codes = torch.empty(E, M, K // 2, dtype=torch.uint8, device=w.device)
    bs = torch.empty(E, K // 64, M, 4, dtype=torch.uint8, device=w.device)
    scales = torch.empty(E, M, dtype=torch.float32, device=w.device)
    _check("moe_quantize_weights_fp4", load().moe_quantize_weights_fp4(
        _ptr(w), _dtype_code(w), E, M, K, _ptr(codes), _ptr(bs), _ptr(scales), _stream(stream)))
    return FP4Weights(codes, bs, scales)


def _expect_fp4(q, shape, name):
    if not isinstance(q, FP4Weights) or tuple(q.shape) != tuple(shape):
        raise ValueError(f"{name}: expected FP4Weights of shape {tuple(shape)}")


def moe_grouped_gate_up_fp4(xs, offsets, q_gate: FP4Weights, q_up: FP4Weights, h, stream=None):
    cap, d = xs.shape
    E, f, _ = q_gate.shape
    _expect(xs, torch.float16, (cap, d), "xs")
    _expect_fp4(q_gate, (E, f, d), "q_gate")
    _expect_fp4(q_up, (E, f, d), "q_up")
    _expect(h, torch.float16, (cap, f), "h")
    _check("moe_grouped_gate_up_fp4", load().moe_grouped_gate_up_fp4(
        _ptr(xs), _ptr(offsets), cap, E, d, f, _ptr(q_gate.codes), _ptr(q_gate.block_scales), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.block_scales), _ptr(q_up.scales), _ptr(h), _stream(stream)))


def moe_grouped_down_fp4(h, offsets, q_down: FP4Weights, y, stream=None):
    cap, f = h.shape
    E, d, _ = q_down.shape
    _expect(h, torch.float16, (cap, f), "h")
    _expect_fp4(q_down, (E, d, f), "q_down")
    _expect(y, torch.float32, (cap, d), "y")
    _check("moe_grouped_down_fp4", load().moe_grouped_down_fp4(
        _ptr(h), _ptr(offsets), cap, E, d, f, _ptr(q_down.codes), _ptr(q_down.block_scales), _ptr(q_down.scales),
        _ptr(y), _stream(stream)))


def moe_forward_fp4(logits, x, mask, q_gate: FP4Weights, q_up: FP4Weights, q_down: FP4Weights, k: int,
                    bufs: MoEBuffers, stream=None) -> torch.Tensor:
    """The whole path with 4-bit weights; ``bufs`` holds fp16 compact activations; returns ``bufs.out``."""
    T, E = logits.shape
    d = x.shape[1]
    f = q_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f, bufs.dtype) != (T, E, k, d, f, torch.float16):
        raise ValueError("buffers were allocated for another shape (the 4-bit path keeps xs and h in fp16)")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect_fp4(q_gate, (E, f, d), "q_gate")
    _expect_fp4(q_up, (E, f, d), "q_up")
    _expect_fp4(q_down, (E, d, f), "q_down")
    b = bufs
    _check("moe_forward_fp4", load().moe_forward_fp4(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f,
        _ptr(q_gate.codes), _ptr(q_gate.block_scales), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.block_scales), _ptr(q_up.scales),
        _ptr(q_down.codes), _ptr(q_down.block_scales), _ptr(q_down.scales),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets), _ptr(b.xs), _ptr(b.row_of_route),
        _ptr(b.route_of_row), _ptr(b.h), _ptr(b.y), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out


# ---------------------------------------------------------------------------
# 4-bit operands on both sides (block-scaled tensor-core MMAs)
# ---------------------------------------------------------------------------

def fp4_ld(rows: int) -> int:
    """Leading dimension of the block scales of `rows` activation rows (a multiple of 4)."""
    return (rows + 3) // 4 * 4


class FP4Rows:
    """Rows of activations in the 4-bit format: ``codes`` uint8 [rows][K/2], ``block_scales`` uint8
    [K/64][ld][4] (E4M3, ld = fp4_ld(rows)), ``scales`` fp32 [rows]."""

    def __init__(self, codes, block_scales, scales):
        rows, K2 = codes.shape
        if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or scales.dtype != torch.float32:
            raise ValueError("expected uint8 codes and block scales, fp32 scales")
        if tuple(block_scales.shape) != (2 * K2 // 64, fp4_ld(rows), 4) or tuple(scales.shape) != (rows,):
            raise ValueError("block scales [K/64][ld][4] and scales [rows] do not match the codes")
        self.codes, self.block_scales, self.scales = codes, block_scales, scales

    @classmethod
    def empty(cls, rows: int, K: int, device="cuda"):
        return cls(torch.empty(rows, K // 2, dtype=torch.uint8, device=device),
                   torch.zeros(K // 64, fp4_ld(rows), 4, dtype=torch.uint8, device=device),
                   torch.empty(rows, dtype=torch.float32, device=device))

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return 2 * self.codes.shape[1]

    @property
    def ld(self) -> int:
        return self.block_scales.shape[1]


def moe_quantize_rows_fp4(a, out: "FP4Rows | None" = None, stream=None) -> FP4Rows:
    """The 4-bit quantizer applied to the rows of ``a`` [rows][K] (bf16 or fp32, K a multiple of 64)."""
    rows, K = a.shape
    out = FP4Rows.empty(rows, K, a.device) if out is None else out
    if (out.rows, out.K) != (rows, K):
        raise ValueError("output rows were allocated for another shape")
    _check("moe_quantize_rows_fp4", load().moe_quantize_rows_fp4(
        _ptr(a), _dtype_code(a), rows, out.ld, K, _ptr(out.codes), _ptr(out.block_scales), _ptr(out.scales),
        _stream(stream)))
    return out


def moe_scatter_rows_fp4(x_q: FP4Rows, ids, mask, offsets, xs_q: FP4Rows, row_of_route, route_of_row, ws,
                         stream=None):
    T, k = ids.shape
    E = offsets.shape[0] - 1
    d = x_q.K
    if x_q.rows != T or xs_q.rows != T * k or xs_q.K != d:
        raise ValueError("4-bit rows do not match the routing")
    _check("moe_scatter_rows_fp4", load().moe_scatter_rows_fp4(
        _ptr(x_q.codes), _ptr(x_q.block_scales), x_q.ld, _ptr(x_q.scales), _ptr(ids), _ptr(mask), _ptr(offsets),
        T, k, d, E, _ptr(xs_q.codes), _ptr(xs_q.block_scales), xs_q.ld, _ptr(xs_q.scales), _ptr(row_of_route),
        _ptr(route_of_row), _ptr(ws), _stream(stream)))


def moe_scatter_rows_quant_fp4(x, ids, mask, offsets, x_q: FP4Rows, xs_q: FP4Rows, row_of_route, route_of_row, ws,
                               stream=None):
    """Quantizes the bf16 token rows x [T][d] into x_q and scatters them into xs_q, in one kernel."""
    T, d = x.shape
    k = ids.shape[1]
    E = offsets.shape[0] - 1
    _expect(x, torch.bfloat16, (T, d), "x")
    if x_q.rows != T or x_q.K != d or xs_q.rows != T * k or xs_q.K != d:
        raise ValueError("4-bit rows do not match the routing")
    _check("moe_scatter_rows_quant_fp4", load().moe_scatter_rows_quant_fp4(
        _ptr(x), _ptr(ids), _ptr(mask), _ptr(offsets), T, k, d, E, _ptr(x_q.codes), _ptr(x_q.block_scales), x_q.ld,
        _ptr(x_q.scales), _ptr(xs_q.codes), _ptr(xs_q.block_scales), xs_q.ld, _ptr(xs_q.scales), _ptr(row_of_route),
        _ptr(route_of_row), _ptr(ws), _stream(stream)))


def moe_route_scatter_quant_small_fp4(logits, x, mask, k: int, bufs: "MoEBuffersW4A4", stream=None):
    """A1-A4 with 4-bit rows in one launch for small chunks (T <= 128, T*k <= 512), into ``bufs``."""
    T, E = logits.shape
    d = x.shape[1]
    b = bufs
    if (b.T, b.E, b.k, b.d) != (T, E, k, d):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _check("moe_route_scatter_quant_small_fp4", load().moe_route_scatter_quant_small_fp4(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets),
        _ptr(b.x_q.codes), _ptr(b.x_q.block_scales), b.x_q.ld, _ptr(b.x_q.scales), _ptr(b.xs_q.codes),
        _ptr(b.xs_q.block_scales), b.xs_q.ld, _ptr(b.xs_q.scales), _ptr(b.row_of_route), _ptr(b.route_of_row),
        _stream(stream)))


def moe_grouped_gate_up_w4a4(xs_q: FP4Rows, offsets, q_gate: FP4Weights, q_up: FP4Weights, h, stream=None):
    E, f, d = q_gate.shape
    cap = xs_q.rows
    _expect_fp4(q_up, (E, f, d), "q_up")
    _expect(h, torch.bfloat16, (cap, f), "h")
    if xs_q.K != d:
        raise ValueError("compact rows do not match the weights")
    _check("moe_grouped_gate_up_w4a4", load().moe_grouped_gate_up_w4a4(
        _ptr(xs_q.codes), _ptr(xs_q.block_scales), xs_q.ld, _ptr(xs_q.scales), _ptr(offsets), cap, E, d, f,
        _ptr(q_gate.codes), _ptr(q_gate.block_scales), _ptr(q_gate.scales), _ptr(q_up.codes),
        _ptr(q_up.block_scales), _ptr(q_up.scales), _ptr(h), _stream(stream)))


def moe_grouped_down_w4a4(h_q: FP4Rows, offsets, q_down: FP4Weights, y, stream=None):
    E, d, f = q_down.shape
    cap = h_q.rows
    _expect(y, torch.float32, (cap, d), "y")
    if h_q.K != f:
        raise ValueError("rows of h do not match the weights")
    _check("moe_grouped_down_w4a4", load().moe_grouped_down_w4a4(
        _ptr(h_q.codes), _ptr(h_q.block_scales), h_q.ld, _ptr(h_q.scales), _ptr(offsets), cap, E, d, f,
        _ptr(q_down.codes), _ptr(q_down.block_scales), _ptr(q_down.scales), _ptr(y), _stream(stream)))


class MoEBuffersW4A4:
    """Caller-owned device buffers of the 4-bit-activation path for one chunk shape (bf16 x)."""

    def __init__(self, T: int, E: int, k: int, d: int, f: int, device="cuda"):
        self.T, self.E, self.k, self.d, self.f = T, E, k, d, f
        cap = T * k
        i32 = dict(dtype=torch.int32, device=device)
        self.ids = torch.empty(T, k, **i32)
        self.w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.x_q = FP4Rows.empty(T, d, device)
        self.xs_q = FP4Rows.empty(cap, d, device)
        self.row_of_route = torch.empty(cap, **i32)
        self.route_of_row = torch.empty(cap, **i32)
        self.h = torch.empty(cap, f, dtype=torch.bfloat16, device=device)
        self.h_q = FP4Rows.empty(cap, f, device)
        self.y = torch.empty(cap, d, dtype=torch.float32, device=device)
        self.out = torch.empty(T, d, dtype=torch.float32, device=device)
        self.ws = torch.zeros(max(moe_workspace_size(T, k), 16) // 4 + 4, dtype=torch.int32, device=device)


def moe_forward_w4a4(logits, x, mask, q_gate: FP4Weights, q_up: FP4Weights, q_down: FP4Weights, k: int,
                     bufs: MoEBuffersW4A4, stream=None) -> torch.Tensor:
    """The whole path on 4-bit weights and activations; returns ``bufs.out`` ([T][d] fp32)."""
    T, E = logits.shape
    d = x.shape[1]
    f = q_gate.shape[1]
    if (bufs.T, bufs.E, bufs.k, bufs.d, bufs.f) != (T, E, k, d, f):
        raise ValueError("buffers were allocated for another shape")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(x, torch.bfloat16, (T, d), "x")
    if mask is not None:
        _expect(mask, torch.uint8, (T, k), "mask")
    _expect_fp4(q_gate, (E, f, d), "q_gate")
    _expect_fp4(q_up, (E, f, d), "q_up")
    _expect_fp4(q_down, (E, d, f), "q_down")
    b = bufs
    _check("moe_forward_w4a4", load().moe_forward_w4a4(
        _ptr(logits), _ptr(x), _ptr(mask), T, E, k, d, f,
        _ptr(q_gate.codes), _ptr(q_gate.block_scales), _ptr(q_gate.scales),
        _ptr(q_up.codes), _ptr(q_up.block_scales), _ptr(q_up.scales),
        _ptr(q_down.codes), _ptr(q_down.block_scales), _ptr(q_down.scales),
        _ptr(b.ids), _ptr(b.w), _ptr(b.counts), _ptr(b.offsets),
        _ptr(b.x_q.codes), _ptr(b.x_q.block_scales), _ptr(b.x_q.scales),
        _ptr(b.xs_q.codes), _ptr(b.xs_q.block_scales), _ptr(b.xs_q.scales),
        _ptr(b.row_of_route), _ptr(b.route_of_row), _ptr(b.h),
        _ptr(b.h_q.codes), _ptr(b.h_q.block_scales), _ptr(b.h_q.scales),
        _ptr(b.y), _ptr(b.out), _ptr(b.ws), _stream(stream)))
    return b.out
