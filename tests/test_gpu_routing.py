"""GPU parity of the routing-side kernels against the oracle (through the C-ABI).

Top-k ids, counts, offsets and the permutation must match bit for bit; the
gate weights within 1e-6 relative; the scattered rows byte for byte; the
combine within the floating-point tolerance of its operand type.
"""

import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import WEIGHT_REL, assert_close, to_np

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _topk(logits, k):
    T, E = logits.shape
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_route_topk(logits.cuda().contiguous(), k, ids, w)
    torch.cuda.synchronize()
    return to_np(ids), to_np(w)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (4, 8, 2), (31, 64, 6), (33, 255, 8), (401, 256, 6), (2048, 256, 6),
                                   (7, 256, 16), (100, 32, 4), (64, 2, 2), (50, 100, 16), (3, 17, 17 - 1)])
def test_topk_matches_oracle(T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E)
    logits = torch.randn(T, E, generator=g)
    ids, w = _topk(logits, k)
    ref_ids, ref_w = mo.route_topk(logits.numpy(), k)
    assert np.array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, ref_w, rtol=WEIGHT_REL, atol=0)


def test_topk_ties_and_signed_zeros():
    """Integer-grid logits manufacture ties; half of the zeros are -0.0."""
    g = torch.Generator().manual_seed(5)
    logits = torch.randint(-3, 4, (512, 256), generator=g).float()
    zeros = logits == 0
    flip = torch.rand(logits.shape, generator=g) < 0.5
    logits[zeros & flip] = -0.0
    for k in (1, 6, 16):
        ids, w = _topk(logits, k)
        ref_ids, ref_w = mo.route_topk(logits.numpy(), k)
        assert np.array_equal(ids, ref_ids)
        np.testing.assert_allclose(w, ref_w, rtol=WEIGHT_REL, atol=0)


def test_topk_golden_fixtures():
    with open(os.path.join(GOLDEN, "topk_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        ids, _ = _topk(torch.tensor([c["logits"]], dtype=torch.float32), c["k"])
        assert ids[0].tolist() == c["ids"], c["name"]


def _routing_case(T, E, k, p_mask, seed, skew=0.0):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    if skew:
        logits += skew * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    return logits, mask


def _run_index_path(logits, mask, k, x):
    T, E = logits.shape
    cap = T * k
    dev = "cuda"
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.full((E,), -5, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -5, dtype=torch.int32, device=dev)
    ws = torch.zeros(M.moe_workspace_size(T, k) // 4 + 4, dtype=torch.int32, device=dev)
    xs = torch.full((cap, x.shape[1]), float("nan"), dtype=x.dtype, device=dev)
    ror = torch.full((cap,), -9, dtype=torch.int32, device=dev)
    rro = torch.full((cap,), -9, dtype=torch.int32, device=dev)
    lg, xd = logits.cuda(), x.cuda()
    md = None if mask is None else mask.cuda()
    M.moe_route_topk(lg, k, ids, w)
    M.moe_route_histogram(ids, md, E, counts, ws)
    M.moe_prefix_offsets(counts, T, k, offsets, ws)
    M.moe_scatter_rows(xd, ids, md, offsets, xs, ror, rro, ws)
    M.moe_check_device_error()
    return dict(ids=ids, w=w, counts=counts, offsets=offsets, xs=xs, row_of_route=ror, route_of_row=rro, ws=ws)


@pytest.mark.parametrize("T,E,k,p,d,dtype", [
    (1, 1, 1, 0.0, 8, torch.bfloat16),
    (5, 4, 2, 0.5, 64, torch.float32),
    (33, 8, 2, 0.0, 64, torch.float32),
    (300, 16, 4, 0.1, 256, torch.bfloat16),
    (401, 256, 6, 0.0, 4096, torch.bfloat16),
    (2048, 256, 6, 0.1, 512, torch.bfloat16),
    (3000, 256, 16, 0.3, 128, torch.bfloat16),   # several histogram chunks, ragged last chunk
    (700, 3, 3, 0.0, 16, torch.bfloat16),        # heavy experts
])
def test_histogram_prefix_scatter(T, E, k, p, d, dtype):
    logits, mask = _routing_case(T, E, k, p, seed=T + E)
    x = torch.randn(T, d).to(dtype)
    res = _run_index_path(logits, mask, k, x)
    ref = mo.moe_forward(logits.numpy(), to_np(x), (np.zeros((E, 1, d)), np.zeros((E, 1, d)), np.zeros((E, d, 1))),
                         k, None if mask is None else mask.numpy())
    assert np.array_equal(to_np(res["ids"]), ref["ids"])
    assert np.array_equal(to_np(res["counts"]), ref["counts"])
    assert np.array_equal(to_np(res["offsets"]), ref["offsets"])
    assert np.array_equal(to_np(res["row_of_route"]), ref["row_of_route"])
    assert np.array_equal(to_np(res["route_of_row"]), ref["route_of_row"])
    R = int(ref["offsets"][-1])
    xs = res["xs"].cpu()
    assert torch.equal(xs[:R], x[torch.as_tensor(ref["route_of_row"][:R] // k, dtype=torch.long)])
    # unused compact rows are zero-filled (+0.0 bit patterns)
    assert torch.all(xs[R:].view(torch.int16 if dtype == torch.bfloat16 else torch.int32) == 0)
    # the workspace is reusable: a second pass gives the same permutation
    res2 = _run_index_path(logits, mask, k, x)
    assert torch.equal(res2["route_of_row"], res["route_of_row"])
    assert torch.equal(res2["counts"], res["counts"])


@pytest.mark.parametrize("T,E,k,p,d", [
    (1, 8, 2, 0.0, 64),
    (63, 16, 4, 0.2, 64),
    (32, 256, 6, 0.1, 64),       # exactly one chunk
    (33, 256, 6, 0.1, 64),       # a one-token second chunk
    (401, 256, 6, 0.0, 256),
    (2048, 256, 6, 0.1, 128),    # 64 chunks of 32 tokens
    (3000, 256, 16, 0.3, 64),    # k = 16: 512 routes per pass
    (8192, 256, 6, 0.0, 64),     # 256 chunks, the most there are
    (8193, 256, 6, 0.1, 64),     # 64-token chunks: two passes per chunk
    (20000, 64, 8, 0.05, 64),    # 96-token chunks, ragged last chunk
    (300, 10, 3, 0.0, 64),       # E not a multiple of 4
])
def test_one_launch_routing_equals_the_step_kernels(T, E, k, p, d):
    """moe_route_topk_offsets gives the step kernels' ids, weights, counts, offsets and workspace (the scatter
    after it writes the same permutation), and the oracle's integer outputs."""
    logits, mask = _routing_case(T, E, k, p, seed=T * 7 + E, skew=1.0)
    x = torch.randn(T, d).to(torch.bfloat16)
    steps = _run_index_path(logits, mask, k, x)
    dev = "cuda"
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    counts = torch.full((E,), -5, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -5, dtype=torch.int32, device=dev)
    ws = torch.zeros(M.moe_workspace_size(T, k) // 4 + 4, dtype=torch.int32, device=dev)
    md = None if mask is None else mask.cuda()
    for _ in range(2):   # the workspace is left ready for the next call
        M.moe_route_topk_offsets(logits.cuda(), md, k, ids, w, counts, offsets, ws)
        M.moe_check_device_error()
        assert torch.equal(ids, steps["ids"])
        if E % 4 == 0:   # both sum the softmax in slot order
            assert torch.equal(w.view(torch.int32), steps["w"].view(torch.int32))
        else:            # the step kernel for other E sums it in butterfly order
            torch.testing.assert_close(w, steps["w"], rtol=1e-6, atol=0)
        assert torch.equal(counts, steps["counts"])
        assert torch.equal(offsets, steps["offsets"])
        assert torch.equal(ws, steps["ws"])
    cap = T * k
    xs = torch.empty(cap, d, dtype=torch.bfloat16, device=dev)
    ror = torch.full((cap,), -9, dtype=torch.int32, device=dev)
    rro = torch.full((cap,), -9, dtype=torch.int32, device=dev)
    M.moe_scatter_rows(x.cuda(), ids, md, offsets, xs, ror, rro, ws)
    M.moe_check_device_error()
    ref_ids, _ = mo.route_topk(logits, k)
    assert np.array_equal(to_np(ids), ref_ids)
    ref_counts = mo.route_histogram(ref_ids, mask, E)
    assert np.array_equal(to_np(counts), ref_counts)
    assert np.array_equal(to_np(offsets), mo.prefix_offsets(ref_counts))
    ref_ror, ref_rro = mo.scatter_permutation(ref_ids, mask)
    assert np.array_equal(to_np(ror), ref_ror)
    assert np.array_equal(to_np(rro), ref_rro)


def test_all_masked_routes():
    T, E, k = 40, 8, 2
    logits, _ = _routing_case(T, E, k, 0.0, seed=1)
    mask = torch.ones(T, k, dtype=torch.uint8)
    x = torch.randn(T, 16)
    res = _run_index_path(logits, mask, k, x)
    assert torch.all(res["counts"] == 0) and torch.all(res["offsets"] == 0)
    assert torch.all(res["row_of_route"] == -1) and torch.all(res["route_of_row"] == -1)
    assert torch.all(res["xs"].cpu().view(torch.int32) == 0)


def _combine(y, ror, w, T, k, d):
    out = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_combine(y.cuda(), ror.cuda(), w.cuda(), out)
    torch.cuda.synchronize()
    return out.cpu()


def test_combine_golden_fixtures():
    with open(os.path.join(GOLDEN, "combine_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        y = torch.tensor(np.array(c["y"], dtype=np.float64), dtype=torch.float32)
        y = torch.nn.functional.pad(y, (0, 4 - y.shape[1]))  # rows padded to a 16-byte multiple
        out = _combine(y, torch.tensor(c["row_of_route"], dtype=torch.int32),
                       torch.tensor(c["w"], dtype=torch.float32).reshape(c["T"], c["k"]), c["T"], c["k"], 4)
        expect = torch.nn.functional.pad(torch.tensor(c["out"], dtype=torch.float32), (0, 4 - len(c["out"][0])))
        assert torch.equal(out, expect), c["name"]
        assert torch.equal(torch.signbit(out), torch.signbit(expect)), c["name"]


@pytest.mark.parametrize("T,k,d,p", [(1, 1, 4, 0.0), (77, 2, 64, 0.3), (401, 6, 4096, 0.0), (2048, 6, 1024, 0.1)])
def test_combine_matches_oracle(T, k, d, p):
    g = torch.Generator().manual_seed(T)
    cap = T * k
    y = torch.randn(cap, d, generator=g)
    perm = torch.randperm(cap, generator=g).to(torch.int32)
    masked = torch.rand(cap, generator=g) < p
    ror = torch.where(masked, torch.full_like(perm, -1), perm)
    w = torch.rand(T, k, generator=g)
    out = _combine(y, ror, w, T, k, d)
    ref = mo.combine(y.numpy(), ror.numpy(), w.numpy(), T, k)
    assert_close(out, ref, "f32")


def test_prefix_can_be_repeated():
    """The prefix reads the histogram's chunk counts without changing them."""
    T, E, k = 3000, 256, 6
    logits, mask = _routing_case(T, E, k, 0.1, seed=4)
    x = torch.randn(T, 64).to(torch.bfloat16)
    once = _run_index_path(logits, mask, k, x)
    again = _run_index_path(logits, mask, k, x)
    M.moe_prefix_offsets(again["counts"], T, k, again["offsets"], again["ws"])
    M.moe_prefix_offsets(again["counts"], T, k, again["offsets"], again["ws"])
    M.moe_scatter_rows(x.cuda(), again["ids"], None if mask is None else mask.cuda(), again["offsets"],
                       again["xs"], again["row_of_route"], again["route_of_row"], again["ws"])
    M.moe_check_device_error()
    for key in ("offsets", "row_of_route", "route_of_row", "xs"):
        assert torch.equal(again[key], once[key]), key


def test_scatter_rejects_an_unprepared_workspace():
    """Ranks and bases that do not belong to these ids are caught before any write outside xs."""
    T, E, k, d = 64, 8, 2, 64
    logits, _ = _routing_case(T, E, k, 0.0, seed=6)
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    M.moe_route_topk(logits.cuda(), k, ids, w)
    offsets = torch.tensor([0] + [T * k] * E, dtype=torch.int32, device="cuda")
    ws = torch.full((M.moe_workspace_size(T, k) // 4 + 4,), 1_000_000, dtype=torch.int32, device="cuda")
    xs = torch.zeros(T * k, d, dtype=torch.float32, device="cuda")
    ror = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    rro = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    M.moe_scatter_rows(torch.randn(T, d, device="cuda"), ids, None, offsets, xs, ror, rro, ws)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    assert torch.all(ror == -1) and torch.all(xs == 0)


def test_combine_rejects_rows_beyond_the_buffer():
    T, k, d = 16, 2, 8
    y = torch.randn(T * k, d)
    ror = torch.arange(T * k, dtype=torch.int32)
    ror[5] = T * k + 7          # not a row of y
    w = torch.rand(T, k)
    out = _combine(y, ror, w, T, k, d)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    ror_ref = ror.clone()
    ror_ref[5] = -1             # the bad slot is skipped like a masked one
    assert_close(out, mo.combine(y.numpy(), ror_ref.numpy(), w.numpy(), T, k), "f32")


@pytest.mark.parametrize("k", [1, 6, 8, 9, 16])
def test_topk_streaming_and_warp_kernels_agree(k):
    """E = 256 with 16-byte-aligned logits takes the streaming kernel; a 4-byte offset view takes the warp kernel."""
    T, E = 777, 256
    g = torch.Generator().manual_seed(k)
    logits = torch.randint(-4, 5, (T, E), generator=g).float()   # many ties
    logits[logits == 0] = -0.0
    flat = torch.empty(T * E + 1, device="cuda")
    shifted = flat[1:].view(T, E)
    shifted.copy_(logits.cuda())
    assert shifted.data_ptr() % 16 != 0
    ids_a = torch.empty(T, k, dtype=torch.int32, device="cuda")
    ids_b = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w_a = torch.empty(T, k, device="cuda")
    w_b = torch.empty(T, k, device="cuda")
    M.moe_route_topk(logits.cuda(), k, ids_a, w_a)
    M.moe_route_topk(shifted, k, ids_b, w_b)
    ref_ids, ref_w = mo.route_topk(logits.numpy(), k)
    assert np.array_equal(to_np(ids_a), ref_ids)
    assert np.array_equal(to_np(ids_b), ref_ids)
    np.testing.assert_allclose(to_np(w_a), ref_w, rtol=WEIGHT_REL, atol=0)
    np.testing.assert_allclose(to_np(w_b), ref_w, rtol=WEIGHT_REL, atol=0)


# ---------------------------------------------------------------------------
# A1-A4 in one launch for small chunks: the same outputs as the four steps
# ---------------------------------------------------------------------------

class _Bufs:
    def __init__(self, T, E, k, d, xs_dtype):
        cap, dev = T * k, "cuda"
        self.ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
        self.w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
        self.counts = torch.full((E,), -5, dtype=torch.int32, device=dev)
        self.offsets = torch.full((E + 1,), -5, dtype=torch.int32, device=dev)
        self.xs = torch.full((cap, d), float("nan"), dtype=xs_dtype, device=dev)
        self.row_of_route = torch.full((cap,), -9, dtype=torch.int32, device=dev)
        self.route_of_row = torch.full((cap,), -9, dtype=torch.int32, device=dev)


@pytest.mark.parametrize("T,E,k,p,d,dtype,xs_f16", [
    (1, 256, 6, 0.0, 4096, torch.bfloat16, False),
    (4, 256, 6, 0.0, 4096, torch.bfloat16, False),
    (4, 256, 6, 0.0, 4096, torch.bfloat16, True),
    (7, 64, 4, 0.3, 128, torch.float32, False),
    (85, 256, 6, 0.2, 256, torch.bfloat16, False),
    (128, 256, 4, 0.0, 128, torch.bfloat16, True),   # T*k = 512, the largest small chunk
    (128, 8, 2, 0.5, 64, torch.float32, False),      # heavy experts, half the routes masked
    (33, 60, 3, 0.1, 64, torch.bfloat16, False),     # E not a multiple of 4
    (16, 4, 4, 1.0, 64, torch.bfloat16, False),      # every route masked
])
def test_small_chunk_routing_equals_the_four_steps(T, E, k, p, d, dtype, xs_f16):
    logits, mask = _routing_case(T, E, k, p, seed=3 * T + E, skew=1.0)
    if p == 1.0:
        mask = torch.ones(T, k, dtype=torch.uint8)
    x = torch.randn(T, d).to(dtype)
    ref = _run_index_path(logits, mask, k, x)
    b = _Bufs(T, E, k, d, torch.float16 if xs_f16 else dtype)
    M.moe_route_scatter_small(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), k, b)
    M.moe_check_device_error()
    for name in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(getattr(b, name), ref[name]), name
    if E % 4 == 0:
        assert torch.equal(b.w, ref["w"])
    else:
        torch.testing.assert_close(b.w, ref["w"], rtol=WEIGHT_REL, atol=0)
    want = ref["xs"].to(torch.float16) if xs_f16 else ref["xs"]
    bits = torch.int16 if want.element_size() == 2 else torch.int32
    assert torch.equal(b.xs.view(bits), want.view(bits))
    # and against the oracle's definition
    oref = mo.moe_forward(logits.numpy(), to_np(x), (np.zeros((E, 1, d)), np.zeros((E, 1, d)), np.zeros((E, d, 1))),
                          k, None if mask is None else mask.numpy())
    assert np.array_equal(to_np(b.ids), oref["ids"])
    assert np.array_equal(to_np(b.route_of_row), oref["route_of_row"])
    np.testing.assert_allclose(to_np(b.w), oref["w"], rtol=WEIGHT_REL, atol=0)


def test_small_chunk_routing_rejects_large_chunks():
    T, E, k, d = 129, 8, 2, 64
    logits, _ = _routing_case(T, E, k, 0.0, seed=1)
    x = torch.randn(T, d)
    b = _Bufs(T, E, k, d, torch.float32)
    with pytest.raises(M.MoEError):
        M.moe_route_scatter_small(logits.cuda(), x.cuda(), None, k, b)
