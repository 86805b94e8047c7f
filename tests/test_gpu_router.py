"""GPU parity of the router projection with top-k routing in its epilogue (through the C-ABI).

The logits are bf16 products accumulated in fp32 on the tensor cores; the
oracle evaluates them in float64.  Each logit must lie within the rigorous
error bound of an fp32 dot product of d terms, d * 2^-24 * sum |x_j wr_j|.
The top-k is an integer decision taken on those fp32 logits: every chosen
expert must be a valid top-k choice of the oracle logits within twice that
bound; where the k-th and (k+1)-th oracle logits are farther apart than that
(the majority of tokens, checked) the chosen set must be the oracle's, in the
oracle's order wherever neighbours are farther apart too.  The kernel's
choice must also be exact on its own logits (checked with plain numpy).
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import to_np

pytestmark = pytest.mark.gpu


def _case(T, E, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wr = (torch.randn(E, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    return x, wr


def _run(x, wr, k, with_logits=True):
    T, E = x.shape[0], wr.shape[0]
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda") if with_logits else None
    M.moe_router_topk(x.cuda(), wr.cuda(), k, ids, w, logits)
    M.moe_check_device_error()
    return to_np(ids), to_np(w), None if logits is None else to_np(logits)


def _own_topk(logits, k):
    """Top-k of one float32 row by (value desc, id asc), -0.0 == +0.0, in plain numpy."""
    order = sorted(range(logits.shape[0]), key=lambda e: (-float(logits[e]), e))
    return order[:k]


@pytest.mark.parametrize("T,E,d,k", [
    (1, 8, 64, 2),
    (4, 256, 4096, 6),
    (64, 256, 256, 6),
    (100, 128, 512, 4),
    (401, 256, 4096, 6),
    (37, 200, 128, 8),     # two expert tiles, the second partly past E
    (130, 60, 192, 3),     # one expert tile, a ragged token tile
])
def test_router_matches_oracle(T, E, d, k):
    x, wr = _case(T, E, d, seed=T * 13 + E)
    ids, w, logits = _run(x, wr, k)
    xf, wf = to_np(x).astype(np.float64), to_np(wr).astype(np.float64)
    ref_logits, ref_ids, ref_w = mo.route_from_router(xf, wf, k)
    # Accumulation model: the products of bf16 operands are exact in fp32; the d products are then added in
    # fp32 in some order (the K split over the cluster reorders them) by an adder that either rounds to
    # nearest or truncates.  Any order of d - 1 such additions errs by at most
    # (d - 1) u / (1 - (d - 1) u) * sum |x_j w_j| with u = 2^-23, the unit roundoff of truncation (twice
    # that of rounding to nearest), so the bound holds whichever the tensor cores do.
    u = 2.0 ** -23
    bound = (d - 1) * u / (1 - (d - 1) * u) * (np.abs(xf) @ np.abs(wf).T)
    assert np.all(np.abs(logits - ref_logits) <= bound)

    n_sep = 0
    for t in range(T):
        # the kernel's choice is exact on its own fp32 logits
        assert ids[t].tolist() == _own_topk(logits[t], k)
        srt = np.sort(ref_logits[t])[::-1]
        band = 2 * bound[t].max()
        # every chosen expert is a valid top-k choice within the bound
        assert np.all(ref_logits[t][ids[t]] >= srt[k - 1] - band)
        if k == E or srt[k - 1] - srt[k] > band:
            # the set is decided: it must be the oracle's, in the oracle's
            # order wherever neighbours are farther apart than the band
            n_sep += 1
            assert set(ids[t].tolist()) == set(ref_ids[t].tolist())
            for s in range(k - 1):
                a, b = ref_ids[t][s], ref_ids[t][s + 1]
                if ref_logits[t][a] - ref_logits[t][b] > band:
                    assert ids[t].tolist().index(a) < ids[t].tolist().index(b)
            if ids[t].tolist() == ref_ids[t].tolist():
                # a logit error of at most delta moves each softmax weight by at most
                # 2 * delta relative; 2e-6 covers the fp32 exponentials and normalisation
                rtol = 2 * bound[t][ids[t]].max() + 2e-6
                np.testing.assert_allclose(w[t], ref_w[t], rtol=rtol, atol=0)
    if T >= 32:
        assert n_sep >= 0.5 * T


def test_router_without_logits_output():
    x, wr = _case(50, 256, 256, seed=3)
    ids_a, w_a, _ = _run(x, wr, 6)
    ids_b, w_b, _ = _run(x, wr, 6, with_logits=False)
    assert np.array_equal(ids_a, ids_b) and np.array_equal(w_a, w_b)


def test_router_rejects_bad_sizes():
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")   # d not a multiple of 64
    wr = torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(4, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(4, 2, dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoEError):
        M.moe_router_topk(x, wr, 2, ids, w)
