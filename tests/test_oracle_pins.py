"""Pins of the CPU oracle against facts it does not compute itself.

Each test checks the oracle against a hand-derived fixture, a brute-force
search, a library routine for a special case that reduces to it, or an
invariant of the mathematics.  None of them re-types the oracle's formula.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as mo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# ---------------------------------------------------------------------------
# golden fixtures (hand-derived closed forms)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("topk_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_topk(case):
    logits = np.array([case["logits"]], dtype=np.float32)
    ids, w = mo.route_topk(logits, case["k"])
    assert ids[0].tolist() == case["ids"]


@pytest.mark.parametrize("case", _golden("softmax_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_softmax(case):
    logits = np.array([case["logits"]], dtype=np.float32)
    _, w = mo.route_topk(logits, case["k"])
    np.testing.assert_allclose(w[0], case["w"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("case", _golden("ffn_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_ffn(case):
    y = mo.expert_ffn(np.array([case["x"]]), np.array(case["w_gate"]), np.array(case["w_up"]),
                      np.array(case["w_down"]))
    np.testing.assert_allclose(y[0], case["y"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("case", _golden("combine_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_combine(case):
    out = mo.combine(np.array(case["y"], dtype=np.float64), np.array(case["row_of_route"]), np.array(case["w"]),
                     case["T"], case["k"])
    expect = np.array(case["out"], dtype=np.float64)
    assert np.array_equal(out, expect)
    # byte-exact: the sign bits must match too (+0.0 expected wherever 0 is expected)
    assert np.array_equal(np.signbit(out), np.signbit(expect))


# ---------------------------------------------------------------------------
# top-k against brute force
# ---------------------------------------------------------------------------

def _brute_force_order(row):
    """The unique ordering in which each expert beats the next (higher logit, or equal and lower id)."""
    E = len(row)
    for perm in itertools.permutations(range(E)):
        if all(row[perm[i]] > row[perm[i + 1]] or (row[perm[i]] == row[perm[i + 1]] and perm[i] < perm[i + 1])
               for i in range(E - 1)):
            return list(perm)
    raise AssertionError("no valid order")


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(300):
        E = int(rng.integers(1, 7))
        k = int(rng.integers(1, E + 1))
        T = 3
        # an integer grid of logits manufactures ties; signed zeros included
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
        logits[logits == 0] = np.where(rng.random(np.count_nonzero(logits == 0)) < 0.5, -0.0, 0.0)
        ids, _ = mo.route_topk(logits, k)
        for t in range(T):
            assert ids[t].tolist() == _brute_force_order(logits[t].tolist())[:k]


def test_softmax_matches_full_softmax_renormalised():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    k = 5
    ids, w = mo.route_topk(logits, k)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    for t in range(50):
        sel = full[t, ids[t]]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=1e-13, atol=0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)  # descending logits give descending weights


# ---------------------------------------------------------------------------
# histogram, prefix and permutation against counting loops and invariants
# ---------------------------------------------------------------------------

def _random_routing(rng, T, E, k, p_mask):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = mo.route_topk(logits, k)
    mask = (rng.random((T, k)) < p_mask).astype(np.uint8) if p_mask > 0 else None
    return logits, ids, w, mask


@pytest.mark.parametrize("T,E,k,p", [(1, 1, 1, 0.0), (7, 3, 2, 0.3), (40, 8, 2, 0.0), (33, 16, 6, 0.25),
                                     (5, 256, 6, 0.1), (64, 12, 12, 0.5)])
def test_histogram_offsets_permutation(T, E, k, p):
    rng = np.random.default_rng(T * 1000 + E)
    _, ids, _, mask = _random_routing(rng, T, E, k, p)
    counts = mo.route_histogram(ids, mask, E)
    # counting loop
    ref = [0] * E
    n_masked = 0
    for t in range(T):
        for s in range(k):
            if mask is not None and mask[t, s]:
                n_masked += 1
            else:
                ref[ids[t, s]] += 1
    assert counts.tolist() == ref
    assert counts.sum() == T * k - n_masked
    offsets = mo.prefix_offsets(counts)
    assert offsets[0] == 0 and offsets[-1] == T * k - n_masked
    assert np.all(np.diff(offsets) == counts) and np.all(np.diff(offsets) >= 0)
    row_of_route, route_of_row = mo.scatter_permutation(ids, mask)
    # nested-loop construction of the expert-major order
    order = []
    for e in range(E):
        for r in range(T * k):
            t, s = divmod(r, k)
            if ids[t, s] == e and not (mask is not None and mask[t, s]):
                order.append(r)
    R = len(order)
    assert route_of_row[:R].tolist() == order
    assert np.all(route_of_row[R:] == -1)
    for row, r in enumerate(order):
        assert row_of_route[r] == row
    assert np.count_nonzero(row_of_route == -1) == n_masked
    # the expert of each row is the one whose segment holds it
    flat = ids.reshape(-1)
    for e in range(E):
        assert np.all(flat[route_of_row[offsets[e]:offsets[e + 1]]] == e)


def test_scatter_then_gather_is_identity():
    rng = np.random.default_rng(3)
    T, E, k, d = 20, 6, 3, 5
    _, ids, _, mask = _random_routing(rng, T, E, k, 0.2)
    x = rng.standard_normal((T, d))
    row_of_route, route_of_row = mo.scatter_permutation(ids, mask)
    xs = mo.scatter_rows(x, route_of_row, k)
    for r in range(T * k):
        if row_of_route[r] >= 0:
            assert np.array_equal(xs[row_of_route[r]], x[r // k])
    R = xs.shape[0]
    assert np.array_equal(row_of_route[route_of_row[:R]], np.arange(R))


# ---------------------------------------------------------------------------
# the FFN and the whole path against special cases that reduce to library routines
# ---------------------------------------------------------------------------

def _dense_swiglu_torch(x, wg, wu, wd):
    x = torch.as_tensor(x, dtype=torch.float64)
    g = torch.nn.functional.linear(x, torch.as_tensor(wg, dtype=torch.float64))
    u = torch.nn.functional.linear(x, torch.as_tensor(wu, dtype=torch.float64))
    h = torch.nn.functional.silu(g) * u
    return torch.nn.functional.linear(h, torch.as_tensor(wd, dtype=torch.float64)).numpy()


def test_single_expert_is_dense_swiglu():
    """E=1, k=1: every token goes to the one expert with weight 1 -> a dense SwiGLU FFN."""
    rng = np.random.default_rng(9)
    T, d, f = 13, 6, 10  # d != f catches a transposed operand
    x = rng.standard_normal((T, d))
    wg, wu = rng.standard_normal((1, f, d)), rng.standard_normal((1, f, d))
    wd = rng.standard_normal((1, d, f))
    logits = rng.standard_normal((T, 1)).astype(np.float32)
    res = mo.moe_forward(logits, x, (wg, wu, wd), 1)
    np.testing.assert_allclose(res["out"], _dense_swiglu_torch(x, wg[0], wu[0], wd[0]), rtol=1e-13, atol=1e-13)


def test_k_equals_E_is_full_softmax_mixture():
    rng = np.random.default_rng(10)
    T, d, f, E = 9, 4, 7, 5
    x = rng.standard_normal((T, d))
    wg, wu = rng.standard_normal((E, f, d)), rng.standard_normal((E, f, d))
    wd = rng.standard_normal((E, d, f))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    res = mo.moe_forward(logits, x, (wg, wu, wd), E)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    ref = sum(p[:, e, None] * _dense_swiglu_torch(x, wg[e], wu[e], wd[e]) for e in range(E))
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-12)


def test_all_masked_gives_plus_zero():
    rng = np.random.default_rng(12)
    T, d, f, E, k = 6, 4, 8, 4, 2
    x = rng.standard_normal((T, d))
    w = (rng.standard_normal((E, f, d)), rng.standard_normal((E, f, d)), rng.standard_normal((E, d, f)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    mask = np.ones((T, k), dtype=np.uint8)
    res = mo.moe_forward(logits, x, w, k, mask)
    assert np.all(res["counts"] == 0) and np.all(res["offsets"] == 0)
    assert res["y"].shape == (0, d)
    assert np.all(res["out"] == 0.0) and not np.any(np.signbit(res["out"]))


def test_masked_expert_never_touched():
    """A NaN expert reached only through masked routes must not leak into the output."""
    rng = np.random.default_rng(13)
    T, d, f, E, k = 10, 4, 6, 4, 2
    x = rng.standard_normal((T, d))
    wg, wu, wd = rng.standard_normal((E, f, d)), rng.standard_normal((E, f, d)), rng.standard_normal((E, d, f))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = mo.route_topk(logits, k)
    mask = (ids == 2).astype(np.uint8)        # every route to expert 2 is owned elsewhere
    clean = mo.moe_forward(logits, x, (wg, wu, wd), k, mask)["out"]
    wg2, wu2, wd2 = wg.copy(), wu.copy(), wd.copy()
    wg2[2] = np.nan
    wu2[2] = np.nan
    wd2[2] = np.nan
    dirty = mo.moe_forward(logits, x, (wg2, wu2, wd2), k, mask)["out"]
    assert np.all(np.isfinite(dirty))
    assert np.array_equal(clean, dirty)
    # masking does not renormalise: the output is the partial sum over owned slots
    _, w = mo.route_topk(logits, k)
    full = mo.moe_forward(logits, x, (wg, wu, wd), k)
    for t in range(T):
        ref = np.zeros(d)
        for s in range(k):
            if not mask[t, s]:
                ref = ref + w[t, s] * _dense_swiglu_torch(x[t][None], wg[ids[t, s]], wu[ids[t, s]],
                                                          wd[ids[t, s]])[0]
        np.testing.assert_allclose(clean[t], ref, rtol=1e-12, atol=1e-12)
    assert not np.allclose(clean, full["out"])


def test_expert_blocks_and_row_blocks_change_no_bit(monkeypatch):
    """A bank fetched a block of experts at a time, and rows evaluated one at a time instead of four per
    pass, give the same output bit for bit (every dot product is the same ascending sum)."""
    rng = np.random.default_rng(14)
    T, d, f, E, k = 23, 5, 9, 6, 3
    x = rng.standard_normal((T, d))
    w = (rng.standard_normal((E, f, d)), rng.standard_normal((E, f, d)), rng.standard_normal((E, d, f)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    mask = (rng.random((T, k)) < 0.3).astype(np.uint8)
    whole = mo.moe_forward(logits, x, w, k, mask)
    monkeypatch.setattr(mo, "EXPERT_BLOCK", 4)
    fetched = []

    def fetch(e0, e1):
        fetched.append((e0, e1))
        return w[0][e0:e1], w[1][e0:e1], w[2][e0:e1]

    blocked = mo.moe_forward(logits, x, fetch, k, mask)
    assert set(fetched) <= {(0, 4), (4, 6)} and len(fetched) >= 2
    assert np.array_equal(blocked["out"], whole["out"])
    # one row at a time through the same grouped call
    xs, off = whole["xs"], whole["offsets"]
    rows = np.concatenate([mo.expert_ffn(xs[i:i + 1], w[0][e], w[1][e], w[2][e])
                           for e in range(E) for i in range(off[e], off[e + 1])])
    assert np.array_equal(rows, whole["y"])


def test_silu_closed_forms():
    assert mo.silu(0.0) == 0.0
    assert mo.silu(-1000.0) == 0.0          # underflows to (-)0, never NaN
    assert math.isclose(float(mo.silu(1000.0)), 1000.0)
    assert math.isclose(float(mo.silu(1.0)) - float(mo.silu(-1.0)), 1.0, rel_tol=1e-15)
