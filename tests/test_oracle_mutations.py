"""Planted mistakes in the oracle must be caught by its pins.

Each mutant replaces one oracle function with a plausible wrong version
(a swapped operand, a wrong tie-break, a renormalised mask, ...) and runs the
pins; at least one pin has to fail.  Mistakes are planted on the CPU, in the
oracle, never in the CUDA path.
"""

import json
import os

import numpy as np
import pytest

from oracle import moe_oracle as mo
import tests.test_oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)["cases"]


def _all_pins():
    """Run every pin once; return the number that fail."""
    failures = 0
    checks = []
    for c in _cases("topk_cases.json"):
        checks.append(lambda c=c: pins.test_golden_topk(c))
    for c in _cases("softmax_cases.json"):
        checks.append(lambda c=c: pins.test_golden_softmax(c))
    for c in _cases("ffn_cases.json"):
        checks.append(lambda c=c: pins.test_golden_ffn(c))
    for c in _cases("combine_cases.json"):
        checks.append(lambda c=c: pins.test_golden_combine(c))
    checks += [
        pins.test_topk_brute_force_with_ties,
        pins.test_softmax_matches_full_softmax_renormalised,
        lambda: pins.test_histogram_offsets_permutation(33, 16, 6, 0.25),
        lambda: pins.test_histogram_offsets_permutation(64, 12, 12, 0.5),
        pins.test_scatter_then_gather_is_identity,
        pins.test_single_expert_is_dense_swiglu,
        pins.test_k_equals_E_is_full_softmax_mixture,
        pins.test_all_masked_gives_plus_zero,
        pins.test_masked_expert_never_touched,
    ]
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    return failures


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins() == 0


def _topk_high_id_ties(logits, k):
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k))
    for t in range(T):
        order = np.lexsort((-np.arange(E), -logits[t].astype(np.float64)))[:k]
        ids[t] = order
        z = np.exp(logits[t, order] - logits[t, order[0]])
        w[t] = z / z.sum()
    return ids, w


def _topk_full_softmax(logits, k):
    ids, _ = ORIG["route_topk"](logits, k)
    lg = np.asarray(logits, dtype=np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return ids, np.take_along_axis(p, ids.astype(np.int64), axis=1)   # not renormalised


def _ffn_swapped_gate_up(rows, wg, wu, wd):
    return ORIG["expert_ffn"](rows, wu, wg, wd)


def _ffn_transposed_down(rows, wg, wu, wd):
    x = np.asarray(rows, dtype=np.float64)
    h = mo.silu(x @ np.asarray(wg).T) * (x @ np.asarray(wu).T)
    return h @ np.asarray(wd, dtype=np.float64)        # missing transpose (only shape-valid when d == f)


def _silu_is_sigmoid(a):
    a = np.asarray(a, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-a))


def _combine_renormalised(y, row_of_route, w, T, k):
    rows = np.asarray(row_of_route).reshape(T, k)
    w = np.asarray(w, dtype=np.float64).reshape(T, k).copy()
    keep = rows >= 0
    s = (w * keep).sum(axis=1, keepdims=True)
    w = np.where(s > 0, w / np.where(s > 0, s, 1), w)
    return ORIG["combine"](y, row_of_route, w, T, k)


def _combine_minus_zero_start(y, row_of_route, w, T, k):
    out = ORIG["combine"](y, row_of_route, w, T, k)
    return np.where(out == 0, -0.0, out)


def _combine_multiplies_masked(y, row_of_route, w, T, k):
    y = np.asarray(y, dtype=np.float64)
    rows = np.asarray(row_of_route).reshape(T, k)
    w = np.asarray(w, dtype=np.float64).reshape(T, k)
    out = np.zeros((T, y.shape[1]))
    for s in range(k):
        src = np.where(rows[:, s] >= 0, rows[:, s], 0)
        out += w[:, s, None] * (y[src] if y.shape[0] else 0.0) * (rows[:, s, None] >= 0)
    return out


def _perm_reversed_within_expert(ids, mask):
    row_of_route, route_of_row = ORIG["scatter_permutation"](ids, mask)
    flat = np.asarray(ids).reshape(-1)
    R = int(np.count_nonzero(route_of_row >= 0))
    used = route_of_row[:R]
    out = used.copy()
    for e in np.unique(flat[used]):
        sel = np.nonzero(flat[used] == e)[0]
        out[sel] = used[sel][::-1]
    route_of_row = route_of_row.copy()
    route_of_row[:R] = out
    row_of_route = np.full_like(row_of_route, -1)
    row_of_route[out] = np.arange(R)
    return row_of_route, route_of_row


def _prefix_inclusive(counts):
    c = np.cumsum(np.asarray(counts, dtype=np.int64))
    return np.concatenate([c, c[-1:]]).astype(np.int32)


def _histogram_counts_masked(ids, mask, E):
    return np.bincount(np.asarray(ids).ravel(), minlength=E).astype(np.int32)


ORIG = {name: getattr(mo, name) for name in
        ("route_topk", "expert_ffn", "combine", "scatter_permutation", "prefix_offsets", "route_histogram",
         "silu")}

MUTANTS = [
    ("route_topk", _topk_high_id_ties),
    ("route_topk", _topk_full_softmax),
    ("expert_ffn", _ffn_swapped_gate_up),
    ("expert_ffn", _ffn_transposed_down),
    ("silu", _silu_is_sigmoid),
    ("combine", _combine_renormalised),
    ("combine", _combine_minus_zero_start),
    ("combine", _combine_multiplies_masked),
    ("scatter_permutation", _perm_reversed_within_expert),
    ("prefix_offsets", _prefix_inclusive),
    ("route_histogram", _histogram_counts_masked),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(mo, name, mutant)
    with np.errstate(all="ignore"):
        assert _all_pins() > 0
