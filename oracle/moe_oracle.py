"""CPU oracle of grouped MoE prefill -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import or run this module.  The product
path (the CUDA library and its Python binding) never calls it, and this
module imports nothing from the product package.

What it computes follows the page "perf(ds4): batch heterogeneous MoE prefill
by expert" (Luce-Org/lucebox PR #640), Summary: tokens are routed to their
top-k of up to 256 routed experts; a route histogram, an exclusive prefix over
the expert counts and a scatter put token rows in expert-major order; grouped
gate/up projections with SwiGLU and a grouped down projection run per expert;
a weighted combine brings the expert outputs back to token order, and masked
(non-owned) routes contribute exactly zero ("Summary" and "Correctness and
validation").  The combine is the fused expert-major route combine of the page
"perf(ds4): accelerate ROCm decode and long-context selection" (PR #667),
lucebox8 A/B section, whose qualification on the page "perf(ds4): extend
sparse prefill scheduling to 10K" (PR #684, "Historical qualification")
includes a byte-exact signed-zero case.

Everything floating-point is evaluated in float64 with no intermediate
rounding.  The integer results (ids, counts, offsets, the permutation) are the
plain definitions: a stable sort, a bincount, a cumulative sum.

Readings of points the pages leave open (each one is also listed in the
design notes of the repository):

* top-k order: experts sorted by logit descending, ties to the lower expert
  id; -0.0 and +0.0 compare equal.
* gate weights: softmax over the k selected logits (identical to a softmax
  over all experts renormalised over the selected k).
* the mask applies after selection: a masked route keeps its slot and its
  weight, is left out of the histogram, the scatter and the combine, and the
  remaining weights are NOT renormalised.
* row order inside an expert segment: ascending route index r = t*k + s.
* SwiGLU: silu(x.Wg) * (x.Wu) with silu(a) = a / (1 + exp(-a)), no clamp.
* combine: out[t] starts at +0.0 and adds w[t,s] * y(t,s) for ascending s,
  skipping masked slots (never multiplying them).

Storage: ``w_gate``/``w_up`` are [E][f][d] and ``w_down`` is [E][d][f]
(K-contiguous rows).  A weight argument may also be a callable
``e -> (w_gate_e, w_up_e, w_down_e)`` so that a caller can fetch one expert at
a time from a bank that does not fit in host memory.

Pins (tests marked "not gpu" check each function against something other
than itself): hand-derived golden fixtures, brute-force top-k over all
orderings on tiny inputs, a closed-form two-expert softmax, counting and
permutation invariants, the E=1/k=1 reduction to a dense SwiGLU FFN, the k=E
reduction to a full softmax mixture, and the all-masked exact +0.0 case.
The FP8 E4M3 weight quantization at the end of the module is pinned against
PyTorch's float8_e4m3fn cast (an independent implementation of the format),
the format's bit layout and hand-worked ties.  The router projection is
pinned by a hand-worked case, one-hot router rows and linearity/permutation
properties.  No function here is unpinned.
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# A1: top-k routing
# ---------------------------------------------------------------------------

def route_topk(logits, k: int):
    """Top-k expert ids and their gate weights for every token.

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (routed experts, up to 256 of them); the page "perf(ds4): extend sparse
    prefill scheduling to 10K", Summary (native top-6 routing is preserved).

    Returns ``ids`` int32 [T][k] (descending logit, ties to the lower id) and
    ``w`` float64 [T][k], the softmax of the k selected logits.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    expert = np.arange(E)
    for t in range(T):
        # Stable order by (-logit, expert id).  np.lexsort sorts by the LAST key
        # first, so the logit key comes last.  -0.0 and +0.0 compare equal.
        order = np.lexsort((expert, -logits[t].astype(np.float64)))
        chosen = order[:k]
        ids[t] = chosen
        sel = logits[t, chosen].astype(np.float64)
        z = np.exp(sel - sel[0])           # sel[0] is the largest selected logit
        w[t] = z / z.sum()
    return ids, w


# ---------------------------------------------------------------------------
# A2 / A3: route histogram and exclusive prefix
# ---------------------------------------------------------------------------

def _unmasked(ids, mask):
    ids = np.asarray(ids)
    if mask is None:
        return np.ones(ids.shape, dtype=bool)
    return np.asarray(mask).reshape(ids.shape) == 0


def route_histogram(ids, mask, E: int):
    """counts[e] = number of unmasked routes whose expert is e.

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (GPU-native route histogram for up to 256 experts; masked owner routes are
    not computed here).
    """
    ids = np.asarray(ids)
    keep = _unmasked(ids, mask)
    return np.bincount(ids[keep].ravel(), minlength=E).astype(np.int32)


def prefix_offsets(counts):
    """offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]  (length E+1).

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (exclusive prefix over the expert counts).
    """
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.zeros(counts.size + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return offsets.astype(np.int32)


# ---------------------------------------------------------------------------
# A4: scatter to expert-major order
# ---------------------------------------------------------------------------

def scatter_permutation(ids, mask):
    """Expert-major permutation of the unmasked routes.

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (GPU-native scatter); row order within an expert keeps the route order,
    as the page "perf(ds4): extend sparse prefill scheduling to 10K" asks of
    selected rows (Summary: selected-row order is preserved).

    Returns ``row_of_route`` int32 [T*k] (-1 for a masked route) and
    ``route_of_row`` int32 [T*k] (-1 for the unused rows R .. T*k-1), where
    R is the number of unmasked routes.
    """
    ids = np.asarray(ids)
    flat = ids.reshape(-1)
    keep = _unmasked(ids, mask).reshape(-1)
    routes = np.nonzero(keep)[0]                       # ascending route index
    order = np.argsort(flat[routes], kind="stable")    # group by expert, keep route order
    route_of_row = np.full(flat.size, -1, dtype=np.int32)
    route_of_row[: routes.size] = routes[order]
    row_of_route = np.full(flat.size, -1, dtype=np.int32)
    row_of_route[routes[order]] = np.arange(routes.size, dtype=np.int32)
    return row_of_route, route_of_row


def scatter_rows(x, route_of_row, k: int):
    """xs[i] = x[token of route route_of_row[i]] for the R used rows."""
    x = np.asarray(x)
    used = np.asarray(route_of_row)
    used = used[used >= 0]
    return x[used // k]


# ---------------------------------------------------------------------------
# A5 / A6: per-expert SwiGLU FFN
# ---------------------------------------------------------------------------

def silu(a):
    """silu(a) = a / (1 + exp(-a)); exp overflow gives -0.0, never NaN."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def _expert(weights, e):
    if callable(weights):
        wg, wu, wd = weights(e)
    else:
        wg, wu, wd = weights[0][e], weights[1][e], weights[2][e]
    return (np.asarray(wg, dtype=np.float64), np.asarray(wu, dtype=np.float64),
            np.asarray(wd, dtype=np.float64))


def expert_swiglu(rows, w_gate_e, w_up_e):
    """h = silu(x.Wg) * (x.Wu) for each row x, in float64 (gate/up step).

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (grouped gate/up projections); the SwiGLU is the "DS4 SwiGLU split op" of
    the page "perf(ggml): reuse ROCmFP4 weights across q=4 columns".
    Storage: w_gate_e, w_up_e [f][d].
    """
    x = np.asarray(rows, dtype=np.float64)
    g = x @ np.asarray(w_gate_e, dtype=np.float64).T    # [n][f]
    u = x @ np.asarray(w_up_e, dtype=np.float64).T      # [n][f]
    return silu(g) * u                                   # [n][f]


def expert_down(h, w_down_e):
    """y = h . Wd for each row h, in float64 (down step).  Storage: w_down_e [d][f]."""
    return np.asarray(h, dtype=np.float64) @ np.asarray(w_down_e, dtype=np.float64).T  # [n][d]


def expert_ffn(rows, w_gate_e, w_up_e, w_down_e):
    """y = (silu(x.Wg) * (x.Wu)) . Wd for each row x: the gate/up step then the down step."""
    return expert_down(expert_swiglu(rows, w_gate_e, w_up_e), w_down_e)


def grouped_swiglu(xs, offsets, weights):
    """h [R][f]: rows offsets[e] .. offsets[e+1]-1 go through expert e's gate/up step."""
    xs = np.asarray(xs, dtype=np.float64)
    offsets = np.asarray(offsets)
    E = offsets.size - 1
    h = None
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            wg, wu, _ = _expert(weights, e)
            he = expert_swiglu(xs[lo:hi], wg, wu)
            if h is None:
                h = np.zeros((int(offsets[E]), he.shape[1]), dtype=np.float64)
            h[lo:hi] = he
    return h


def grouped_ffn(xs, offsets, weights):
    """Expert outputs y [R][d]: rows offsets[e] .. offsets[e+1]-1 go through expert e.

    Page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
    (one grouped gate/up/down graph instead of a serial graph per active
    expert).  Experts with no rows are skipped.
    """
    xs = np.asarray(xs, dtype=np.float64)
    offsets = np.asarray(offsets)
    E = offsets.size - 1
    y = np.zeros((int(offsets[E]), xs.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = expert_ffn(xs[lo:hi], *_expert(weights, e))
    return y


# ---------------------------------------------------------------------------
# A7: weighted combine back to token order
# ---------------------------------------------------------------------------

def combine(y, row_of_route, w, T: int, k: int):
    """out[t] = +0.0 + sum over ascending unmasked slots s of w[t,s] * y[row(t,s)].

    Page "perf(ds4): accelerate ROCm decode and long-context selection",
    lucebox8 A/B (fused expert-major combine replacing the reduce/multiply
    launches); page "perf(ds4): batch heterogeneous MoE prefill by expert",
    Summary (masked owner routes are exact zero contributions).
    """
    y = np.asarray(y, dtype=np.float64)
    rows = np.asarray(row_of_route).reshape(T, k)
    w = np.asarray(w, dtype=np.float64).reshape(T, k)
    d = y.shape[1] if y.ndim == 2 else 0
    out = np.zeros((T, d), dtype=np.float64)          # +0.0 everywhere
    for s in range(k):
        used = rows[:, s] >= 0
        out[used] += w[used, s, None] * y[rows[used, s]]
    return out


# ---------------------------------------------------------------------------
# The whole path, and a per-token form for spot checks at full size
# ---------------------------------------------------------------------------

def moe_forward(logits, x, weights, k: int, mask=None):
    """Every intermediate of the path for one chunk, as a dict."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids, w = route_topk(logits, k)
    counts = route_histogram(ids, mask, E)
    offsets = prefix_offsets(counts)
    row_of_route, route_of_row = scatter_permutation(ids, mask)
    xs = scatter_rows(x, route_of_row, k)
    y = grouped_ffn(xs, offsets, weights)
    out = combine(y, row_of_route, w, T, k)
    return {"ids": ids, "w": w, "counts": counts, "offsets": offsets,
            "row_of_route": row_of_route, "route_of_row": route_of_row,
            "xs": xs, "y": y, "out": out}


def token_outputs(tokens, ids, w, mask, x, weights):
    """out[t] for the listed tokens, evaluated route by route from the definition.

    Same result as ``moe_forward(...)["out"][tokens]`` (up to float64
    rounding order) without running the other tokens: used to spot-check
    full-size runs on a sample of tokens.
    """
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    keep = _unmasked(ids, mask)
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros((len(tokens), x.shape[1]), dtype=np.float64)
    for i, t in enumerate(tokens):
        for s in range(ids.shape[1]):
            if keep[t, s]:
                y = expert_ffn(x[t][None, :], *_expert(weights, int(ids[t, s])))[0]
                out[i] += w[t, s] * y
    return out


# ---------------------------------------------------------------------------
# Low-bit expert weights: FP8 E4M3 codes with one scale per output channel
# ---------------------------------------------------------------------------
#
# The pages run their experts on quantized weights (page "perf(ds4): batch
# heterogeneous MoE prefill by expert", "Fresh main-snapshot requalification":
# a ROCmFP2 model; page "perf(ggml): reuse ROCmFP4 weights across q=4
# columns": ROCmFP4/FPX formats).  The GB300 counterpart here is the OCP FP8
# E4M3 format (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
# infinities; the all-ones code is NaN, so the largest finite value is 448;
# subnormals down to 2^-9) with one float32 scale per output channel:
#   s[e][m] = max_k |w[e][m][k]| / 448  (1 when the row is all zero),
#   q[e][m][k] = E4M3 round-to-nearest-even of the float32 quotient
#                w[e][m][k] / s[e][m], saturating at +-448,
# and the dequantized weight is s * q.  Both divisions are float32 (IEEE),
# so the codes are a function of the float32 inputs alone.

E4M3_MAX = 448.0


def e4m3_round(x):
    """Nearest E4M3 value (ties to even), saturating at +-448, as float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # exponent of a: a = frac * 2^E with frac in [0.5, 1)  ->  binade 2^(E-1)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    binade = np.maximum(E - 1, -6)                  # subnormals share the 2^-6 binade's spacing
    quantum = np.ldexp(1.0, binade - 3)             # 3 mantissa bits
    r = np.round(a / quantum) * quantum             # np.round: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)                        # the format has a signed zero: -tiny -> -0


def e4m3_encode(v):
    """Byte code of E4M3 values (as produced by e4m3_round)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    e_field = np.where(a >= 2.0 ** -6, E - 1 + 7, 0)
    mant = np.where(e_field > 0, a / np.ldexp(1.0, E - 1) * 8 - 8, a / 2.0 ** -9)
    code = (sign.astype(np.int64) << 7) | (e_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    return np.where(a == 0, sign.astype(np.int64) << 7, code).astype(np.uint8)


def e4m3_decode(code):
    """Values of E4M3 byte codes (NaN code excluded)."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e > 0, np.ldexp(1.0 + m / 8.0, e - 7), np.ldexp(m / 8.0, -6))
    return sign * val


def quantize_weights_fp8(w):
    """Per-output-channel FP8 E4M3 quantization of a weight bank [..., M, K].

    Returns (codes uint8 [..., M, K], scales float32 [..., M]).  The
    dequantized weights are scales[..., None] * e4m3_decode(codes).
    """
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    quotient = (w32 / scale[..., None]).astype(np.float32)
    return e4m3_encode(e4m3_round(quotient)), scale


def dequantize_weights_fp8(codes, scales):
    return np.asarray(scales, dtype=np.float64)[..., None] * e4m3_decode(codes)


# ---------------------------------------------------------------------------
# The router projection in front of A1
# ---------------------------------------------------------------------------
#
# The pages route every token to its top-6 of 256 routed experts from router
# logits (page "perf(ds4): extend sparse prefill scheduling to 10K", Summary:
# native top-6 routing); the logits are the token row times the router
# matrix.  Here the router matrix is stored like the expert weights,
# K-contiguous: wr [E][d], logits[t][e] = sum_j x[t][j] * wr[e][j].

def router_logits(x, wr):
    """Router logits [T][E] = x [T][d] . wr[E][d]^T, in float64."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(wr, dtype=np.float64).T


def route_from_router(x, wr, k: int):
    """Logits, ids and gate weights of the router step followed by A1."""
    logits = router_logits(x, wr)
    ids, w = route_topk(logits, k)
    return logits, ids, w
