"""GPU parity of the 4-bit-activation path: 4-bit weights and activations on block-scaled tensor cores.

Every quantized operand is compared bit for bit with the oracle's 4-bit
quantizer: the codes, block scales and row scales of the token rows, of the
compact rows (their scatter) and of h (the quantizer applied to the GPU's own
bf16 h).  h is compared with the oracle's h within its bf16 rounding bound, y
with the oracle's down projection of the GPU's quantized h (the tensor cores
multiply the same 4-bit values exactly and accumulate in fp32), and out with
the oracle's whole 4-bit path.  The codes of h are decided from the kernel's
bf16 h on both sides.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_bf16_rounded, to_np
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _row_block_scales(q: "M.FP4Rows", r0=0, r1=None):
    """The GPU's tile-major block scales [K/64][ld][4] of rows r0 .. r1-1 in the oracle's layout [rows][K/16]."""
    r1 = q.rows if r1 is None else r1
    bs = q.block_scales[:, r0:r1, :].permute(1, 0, 2).contiguous()
    return to_np(bs.reshape(r1 - r0, -1))


def _check_rows(q: "M.FP4Rows", ob, r0=0, r1=None):
    r1 = q.rows if r1 is None else r1
    assert np.array_equal(to_np(q.codes[r0:r1]), ob.codes)
    assert np.array_equal(_row_block_scales(q, r0, r1), ob.block_scales)
    assert np.array_equal(to_np(q.scales[r0:r1]), ob.scales)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,K", [(1, 64), (37, 128), (300, 4096), (8, 2048)])
def test_quantize_rows_fp4_is_the_weight_quantizer(dtype, rows, K):
    g = torch.Generator().manual_seed(rows + K)
    a = torch.randn(rows, K, generator=g) * 3
    a[0, :16] = 0.0                                  # an all-zero block
    if rows > 2:
        a[2] = 0.0                                   # an all-zero row
        a[1, 5] = 900.0                              # one large value
    a = a.to(dtype)
    q = M.moe_quantize_rows_fp4(a.cuda())
    M.moe_check_device_error()
    _check_rows(q, mo.quantize_bank_fp4(a))


def _case(T, E, k, d, f, p_mask, seed, skew=1.5):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g) + skew * torch.linspace(0, 1, E)[None, :]
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    return logits, mask, x, wg, wu, wd


def _check_against_oracle(b, ref, k):
    for key in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(b, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    _check_rows(b.x_q, ref["x_q"])
    # compact rows: the scattered codes, block scales and scales; rows R .. T*k-1 zero
    tok = ref["route_of_row"][:R] // k
    assert np.array_equal(to_np(b.xs_q.codes[:R]), ref["x_q"].codes[tok])
    assert np.array_equal(_row_block_scales(b.xs_q, 0, R), ref["x_q"].block_scales[tok])
    assert np.array_equal(to_np(b.xs_q.scales[:R]), ref["x_q"].scales[tok])
    assert torch.all(b.xs_q.codes[R:] == 0) and torch.all(b.xs_q.block_scales[:, R:b.xs_q.rows] == 0)
    assert_close_bf16_rounded(b.h[:R], ref["h"])
    hq = mo.quantize_bank_fp4(b.h[:R].cpu())
    _check_rows(b.h_q, hq, 0, R)
    return R, hq


W4A4_CASES = [
    # T, E, k, d, f, p_mask
    (300, 8, 2, 256, 384, 0.0),
    (77, 4, 2, 128, 128, 0.2),
    (600, 16, 4, 512, 256, 0.1),
    (200, 1, 1, 128, 256, 0.0),
    (150, 3, 2, 384, 256, 0.0),     # d = 384: K = 128 mod 256 in the down projection's partner; half-empty stage
    (20, 16, 4, 512, 512, 0.1),
    (4, 64, 6, 256, 256, 0.0),      # a verification-width batch
    (12, 16, 4, 384, 384, 0.1),     # d and f = 128 mod 256 in a small chunk
    (30, 1, 1, 256, 512, 0.0),      # one expert
    (700, 8, 2, 256, 256, 0.0),     # heavy experts: many 64-row slices
]


@pytest.mark.parametrize("T,E,k,d,f,p", W4A4_CASES)
def test_w4a4_path_matches_oracle(T, E, k, d, f, p):
    logits, mask, x, wg, wu, wd = _case(T, E, k, d, f, p, seed=T * 5 + E)
    if T == 700:
        logits[:, 6] += 3.0
        logits[:, 7] += 2.5
    q = [M.moe_quantize_weights_fp4(w.cuda()) for w in (wg, wu, wd)]
    b = M.MoEBuffersW4A4(T, E, k, d, f)
    for t in (b.h, b.y, b.out):
        t.fill_(float("nan"))
    out = M.moe_forward_w4a4(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), *q, k, b)
    M.moe_check_device_error()
    qo = tuple(mo.quantize_bank_fp4(w) for w in (wg, wu, wd))
    R = int(b.offsets[-1])
    ref = mo.moe_forward_w4a4(logits, x, qo, k, mask, h_decided=b.h[:R].cpu())
    R, hq = _check_against_oracle(b, ref, k)
    # y: the oracle's down projection of the GPU's own quantized h
    y_ref = mo.grouped_down(mo.dequantize_weights_fp4(hq.codes, hq.block_scales, hq.scales), ref["offsets"], qo)
    assert_close(b.y[:R], y_ref, "bf16")
    assert torch.all(b.y[R:] == 0) and torch.all(b.h[R:].float() == 0)
    assert_close(out, ref["out"], "bf16")


def test_w4a4_steps_equal_the_whole_path():
    T, E, k, d, f = 100, 8, 2, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, 0.1, seed=6))
    q = [M.moe_quantize_weights_fp4(w) for w in (wg, wu, wd)]
    a = M.MoEBuffersW4A4(T, E, k, d, f)
    whole = M.moe_forward_w4a4(logits, x, mask, *q, k, a).clone()
    b = M.MoEBuffersW4A4(T, E, k, d, f)
    M.moe_route_topk_offsets(logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws)
    xq = M.moe_quantize_rows_fp4(x)
    M.moe_scatter_rows_fp4(xq, b.ids, mask, b.offsets, b.xs_q, b.row_of_route, b.route_of_row, b.ws)
    M.moe_grouped_gate_up_w4a4(b.xs_q, b.offsets, q[0], q[1], b.h)
    hq = M.moe_quantize_rows_fp4(b.h)
    M.moe_grouped_down_w4a4(hq, b.offsets, q[2], b.y)
    M.moe_combine(b.y, b.row_of_route, b.w, b.out)
    M.moe_check_device_error()
    assert torch.equal(b.out.view(torch.int32), whole.view(torch.int32))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_t4", "prefill_t401", "prefill_t2048", "prefill_t8192"])
def test_w4a4_full_size_workload(name):
    """Every output at full size: the integer outputs and every code bit for bit, h on every compact row, out on
    every token against the oracle's 4-bit path."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    q = [M.moe_quantize_weights_fp4(inp[n]) for n in ("w_gate", "w_up", "w_down")]
    b = M.MoEBuffersW4A4(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    out = M.moe_forward_w4a4(inp["logits"], inp["x"], inp["mask"], *q, cfg.k, b)
    M.moe_check_device_error()
    cache = {}

    def fetch(e0, e1):
        if (e0, e1) not in cache:
            banks = []
            for qq, name_w in zip(q, ("w_gate", "w_up", "w_down")):
                ob = mo.quantize_bank_fp4(inp[name_w][e0:e1].cpu())
                assert np.array_equal(to_np(qq.codes[e0:e1]), ob.codes)
                banks.append(ob)
            cache[(e0, e1)] = tuple(banks)
        return cache[(e0, e1)]

    R = int(b.offsets[-1])
    ref = mo.moe_forward_w4a4(inp["logits"].cpu(), inp["x"].cpu(), fetch, cfg.k,
                              None if inp["mask"] is None else inp["mask"].cpu(), h_decided=b.h[:R].cpu())
    _check_against_oracle(b, ref, cfg.k)
    st = assert_close(out, ref["out"], "bf16")
    print(f"{name} W4A4: rel_fro={st['rel_fro']:.2e} max/rms={st['max_abs'] / st['rms_ref']:.2e}")


@pytest.mark.parametrize("T,E,k,d,p", [(300, 16, 4, 512, 0.1), (40, 8, 6, 4096, 0.0), (33, 4, 2, 8192, 0.2),
                                       (20, 4, 2, 128, 0.0)])
def test_fused_quantize_scatter_equals_the_two_steps(T, E, k, d, p):
    """The scatter that quantizes the token rows gives the codes, block scales and scales of
    moe_quantize_rows_fp4 followed by moe_scatter_rows_fp4, bit for bit."""
    logits, mask, *_ = _case(T, E, k, 128, 128, p, seed=d + T)
    x = (torch.randn(T, d) * 2).to(torch.bfloat16).cuda()
    x[0, :16] = 0.0
    md = None if mask is None else mask.cuda()
    a = M.MoEBuffersW4A4(T, E, k, d, 128)
    M.moe_route_topk_offsets(logits.cuda(), md, k, a.ids, a.w, a.counts, a.offsets, a.ws)
    ref_x = M.moe_quantize_rows_fp4(x)
    ref_xs = M.FP4Rows.empty(T * k, d)
    ref_ror, ref_rro = torch.empty_like(a.row_of_route), torch.empty_like(a.route_of_row)
    M.moe_scatter_rows_fp4(ref_x, a.ids, md, a.offsets, ref_xs, ref_ror, ref_rro, a.ws)
    a.xs_q.codes.fill_(7)
    a.xs_q.scales.fill_(float("nan"))
    M.moe_scatter_rows_quant_fp4(x, a.ids, md, a.offsets, a.x_q, a.xs_q, a.row_of_route, a.route_of_row, a.ws)
    M.moe_check_device_error()
    for got, ref in ((a.x_q, ref_x), (a.xs_q, ref_xs)):
        n = got.rows
        assert torch.equal(got.codes, ref.codes)
        assert torch.equal(got.block_scales[:, :n], ref.block_scales[:, :n])
        assert torch.equal(got.scales.view(torch.int32), ref.scales.view(torch.int32))
    assert torch.equal(a.row_of_route, ref_ror) and torch.equal(a.route_of_row, ref_rro)
    _check_rows(a.x_q, mo.quantize_bank_fp4(x.cpu()))


def test_w4a4_kernels_reject_inconsistent_offsets():
    """offsets[E] beyond the capacity: the 4-bit kernels skip their work and flag it; nothing hangs."""
    E, d, f, cap = 4, 256, 256, 64
    w = [M.moe_quantize_weights_fp4(torch.zeros(E, f, d, dtype=torch.bfloat16, device="cuda")) for _ in range(2)]
    wd = M.moe_quantize_weights_fp4(torch.zeros(E, d, f, dtype=torch.bfloat16, device="cuda"))
    xs = M.moe_quantize_rows_fp4(torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"))
    h = torch.zeros(cap, f, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(cap, d, dtype=torch.float32, device="cuda")
    offsets = torch.tensor([0, 16, 32, 48, cap + 9], dtype=torch.int32, device="cuda")
    M.moe_grouped_gate_up_w4a4(xs, offsets, w[0], w[1], h)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    hq = M.moe_quantize_rows_fp4(h)
    M.moe_grouped_down_w4a4(hq, offsets, wd, y)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    M.moe_check_device_error()


@pytest.mark.parametrize("fmt", ["w4a4", "w8a8"])
def test_low_bit_paths_are_capturable_in_a_cuda_graph(fmt):
    """No allocation, synchronisation or host read inside the 4-bit and E4M3 paths: a CUDA graph of one
    call replays it bit for bit."""
    T, E, k, d, f = 300, 16, 4, 256, 256
    logits, mask, x, wg, wu, wd = (t.cuda() if t is not None else None
                                   for t in _case(T, E, k, d, f, 0.1, seed=43))
    if fmt == "w4a4":
        q = [M.moe_quantize_weights_fp4(w) for w in (wg, wu, wd)]
        b, fwd = M.MoEBuffersW4A4(T, E, k, d, f), M.moe_forward_w4a4
    else:
        q = [M.moe_quantize_weights_fp8(w) for w in (wg, wu, wd)]
        b, fwd = M.MoEBuffersW8A8(T, E, k, d, f), M.moe_forward_w8a8
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref = fwd(logits, x, mask, *q, k, b).clone()      # warm-up call off the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd(logits, x, mask, *q, k, b)
    b.out.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    M.moe_check_device_error()
    assert torch.equal(b.out.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("T,E,k,d,p", [(4, 64, 6, 256, 0.0), (100, 8, 2, 256, 0.1), (64, 10, 8, 512, 0.3),
                                       (128, 256, 4, 128, 0.0), (1, 4, 2, 4096, 0.0)])
def test_small_chunk_routing_quantize_scatter_in_one_launch(T, E, k, d, p):
    """moe_route_scatter_quant_small_fp4 gives the routing outputs of moe_route_topk_offsets and the rows of
    moe_scatter_rows_quant_fp4, bit for bit."""
    logits, mask, *_ = _case(T, E, k, 128, 128, p, seed=T + d)
    x = (torch.randn(T, d) * 2).to(torch.bfloat16).cuda()
    lg, md = logits.cuda(), None if mask is None else mask.cuda()
    a = M.MoEBuffersW4A4(T, E, k, d, 128)
    M.moe_route_topk_offsets(lg, md, k, a.ids, a.w, a.counts, a.offsets, a.ws)
    M.moe_scatter_rows_quant_fp4(x, a.ids, md, a.offsets, a.x_q, a.xs_q, a.row_of_route, a.route_of_row, a.ws)
    b = M.MoEBuffersW4A4(T, E, k, d, 128)
    b.xs_q.codes.fill_(5)
    b.xs_q.scales.fill_(float("nan"))
    b.route_of_row.fill_(77)
    M.moe_route_scatter_quant_small_fp4(lg, x, md, k, b)
    M.moe_check_device_error()
    for name in ("ids", "counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.w.view(torch.int32), b.w.view(torch.int32))
    for qa, qb in ((a.x_q, b.x_q), (a.xs_q, b.xs_q)):
        n = qa.rows
        assert torch.equal(qa.codes, qb.codes)
        assert torch.equal(qa.block_scales[:, :n], qb.block_scales[:, :n])
        assert torch.equal(qa.scales.view(torch.int32), qb.scales.view(torch.int32))
