"""The allocation-free histogram entry point gives the workspace entry point's counts.

moe_route_histogram_noalloc serves callers that cannot allocate device
memory (for instance code inside a host framework that owns every device
allocation and passes no workspace).  Its scratch is a static device array
inside the library, shared by every call; these tests call it through the
C-ABI twice in a row and compare with moe_route_histogram, whose scratch is
the caller's workspace, and with the CPU oracle's histogram of the same
routes.  Counts are integers, so the comparisons are exact.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M

pytestmark = pytest.mark.gpu


def _ids(T, E, k, p_mask, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8).cuda() if p_mask > 0 else None
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    M.moe_route_topk(logits.cuda(), k, ids, w)
    return ids, mask


@pytest.mark.parametrize("T,E,k,p", [(2048, 256, 6, 0.1), (401, 256, 6, 0.0), (10000, 64, 6, 0.2), (1, 1, 1, 0.0),
                                     (4096, 16, 16, 0.5)])  # T*k = 65536: the limit itself
def test_noalloc_histogram_matches_workspace_histogram(T, E, k, p):
    ids, mask = _ids(T, E, k, p, seed=T + E)
    ref = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = torch.zeros(M.moe_workspace_size(T, k) // 4 + 4, dtype=torch.int32, device="cuda")
    M.moe_route_histogram(ids, mask, E, ref, ws)
    oracle_counts = mo.route_histogram(ids.cpu(), None if mask is None else mask.cpu(), E)
    assert np.array_equal(ref.cpu().numpy(), oracle_counts)
    for _ in range(2):  # two calls in a row share the static scratch
        got = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        M.moe_route_histogram_noalloc(ids, mask, E, got)
        M.moe_check_device_error()
        assert torch.equal(got, ref)
        assert np.array_equal(got.cpu().numpy(), oracle_counts)


def test_noalloc_histogram_rejects_chunks_beyond_its_scratch():
    T, E, k = 65537, 4, 1
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoEError) as exc:
        M.moe_route_histogram_noalloc(ids, None, E, counts)
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
