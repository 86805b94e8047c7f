"""Pins of the oracle's router projection (the step in front of top-k routing)."""

import json
import math
import os

import numpy as np

from oracle import moe_oracle as mo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_router_case():
    c = json.load(open(os.path.join(GOLDEN, "router_case.json")))
    logits, ids, w = mo.route_from_router(np.array(c["x"]), np.array(c["wr"]), c["k"])
    assert np.array_equal(logits, np.array(c["logits"]))
    assert ids.tolist() == c["ids"]
    # token 0: logits 3 and 2 -> weights e^0 / (1 + e^-1), e^-1 / (1 + e^-1)
    assert math.isclose(w[0][0], 1 / (1 + math.exp(-1)), rel_tol=1e-15)
    assert math.isclose(w[0][1], math.exp(-1) / (1 + math.exp(-1)), rel_tol=1e-15)


def test_one_hot_router_rows_select_input_columns():
    rng = np.random.default_rng(0)
    T, d, E = 5, 16, 7
    x = rng.standard_normal((T, d))
    cols = rng.integers(0, d, size=E)
    wr = np.zeros((E, d))
    wr[np.arange(E), cols] = 1.0
    assert np.array_equal(mo.router_logits(x, wr), x[:, cols])


def test_router_is_linear_and_permutation_equivariant():
    rng = np.random.default_rng(1)
    T, d, E = 6, 32, 9
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((E, d))
    a = mo.router_logits(x, wr)
    np.testing.assert_allclose(mo.router_logits(2.0 * x, wr), 2.0 * a, rtol=1e-14)
    np.testing.assert_allclose(mo.router_logits(x, wr + wr), 2.0 * a, rtol=1e-14)
    perm = rng.permutation(E)
    np.testing.assert_allclose(mo.router_logits(x, wr[perm]), a[:, perm], rtol=1e-14)
