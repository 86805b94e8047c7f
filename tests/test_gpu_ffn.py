"""GPU parity of the grouped expert FFN and of the whole path (through the C-ABI).

Sizes here run in seconds on the oracle and still span several 128-row
weight tiles, several 128-row compact slices of one expert, ragged tails
and empty experts.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, assert_close_bf16_rounded, full_size_reference, to_np
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed, p_mask=0.0, dead_experts=()):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    # a skew makes a few experts heavy (> 128 rows: several compact slices)
    logits += 1.5 * torch.linspace(0, 1, E)[None, :]
    for e in dead_experts:
        logits[:, e] = -50.0
    mask = (torch.rand(T, k, generator=g) < p_mask).to(torch.uint8) if p_mask > 0 else None
    return logits, mask


def _weights(E, d, f, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(dtype)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(dtype)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(dtype)
    return wg, wu, wd


FFN_CASES = [
    # E, d, f, T, k, p_mask, dtype
    (8, 256, 384, 300, 2, 0.0, torch.bfloat16),
    (4, 128, 128, 77, 2, 0.2, torch.bfloat16),
    (16, 512, 256, 600, 4, 0.1, torch.bfloat16),
    (1, 128, 256, 200, 1, 0.0, torch.bfloat16),
    (3, 384, 256, 150, 2, 0.0, torch.bfloat16),   # d = 384: the down projection's last feature pair is half a pair
    # T*k <= 128: narrow work items (64-feature gate/up items, single-tile down items)
    (16, 512, 384, 20, 4, 0.1, torch.bfloat16),
    (3, 384, 256, 30, 2, 0.0, torch.bfloat16),    # d = 384: three single-tile down items per expert
    (256, 256, 256, 4, 6, 0.0, torch.bfloat16),   # a 4-token verification batch
    (8, 64, 128, 32, 2, 0.0, torch.float32),
    (5, 96, 160, 50, 3, 0.3, torch.float32),
]


@pytest.mark.parametrize("E,d,f,T,k,p,dtype", FFN_CASES)
def test_grouped_ffn_matches_oracle(E, d, f, T, k, p, dtype):
    logits, mask = _routing(T, E, k, seed=E * 31 + T, p_mask=p, dead_experts=(1,) if E > 3 else ())
    x = torch.randn(T, d).to(dtype)
    wg, wu, wd = _weights(E, d, f, dtype, seed=d + f)
    bufs = M.MoEBuffers(T, E, k, d, f, dtype)
    for b in (bufs.h, bufs.y):
        b.fill_(float("nan"))
    out = M.moe_forward(logits.cuda(), x.cuda(), None if mask is None else mask.cuda(), wg.cuda(), wu.cuda(),
                        wd.cuda(), k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k,
                         None if mask is None else mask.numpy())
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    R = int(ref["offsets"][-1])
    assert np.array_equal(to_np(bufs.offsets), ref["offsets"])
    h_ref = mo.grouped_swiglu(ref["xs"], ref["offsets"], (to_np(wg), to_np(wu), to_np(wd)))
    if dtype == torch.bfloat16:
        assert_close_bf16_rounded(bufs.h[:R], h_ref)
    else:
        assert_close(bufs.h[:R], h_ref, tol)
    # the down step is checked against the oracle applied to the GPU's own h,
    # so that h's bf16 rounding is not counted twice
    y_ref_from_h = np.zeros((R, d))
    off = ref["offsets"]
    h_gpu = to_np(bufs.h[:R]).astype(np.float64)
    for e in range(E):
        if off[e + 1] > off[e]:
            y_ref_from_h[off[e]:off[e + 1]] = mo.expert_down(h_gpu[off[e]:off[e + 1]], to_np(wd[e]))
    assert_close(bufs.y[:R], y_ref_from_h, tol)
    assert_close(out, ref["out"], tol)
    # unused compact rows are zero-filled
    assert torch.all(bufs.h[R:].float() == 0) and torch.all(bufs.y[R:] == 0)


def test_expert_with_many_compact_slices():
    """One expert owns all routes: ~5 compact slices of 128 rows plus a ragged one."""
    E, d, f, T, k = 2, 128, 256, 700, 1
    logits = torch.zeros(T, E)
    logits[:, 1] = 1.0
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, torch.bfloat16, seed=3)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    out = M.moe_forward(logits.cuda(), x.cuda(), None, wg.cuda(), wu.cuda(), wd.cuda(), k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k)
    assert to_np(bufs.counts).tolist() == [0, 700]
    assert_close(out, ref["out"], "bf16")


def test_tiny_fp32_workload():
    cfg = CONFIGS["tiny_fp32"]
    inp = make_inputs(cfg)
    bufs = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.float32)
    out = M.moe_forward(inp["logits"].cuda(), inp["x"].cuda(), None, inp["w_gate"].cuda(), inp["w_up"].cuda(),
                        inp["w_down"].cuda(), cfg.k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(inp["logits"].numpy(), inp["x"].numpy(),
                         (inp["w_gate"].numpy(), inp["w_up"].numpy(), inp["w_down"].numpy()), cfg.k)
    assert np.array_equal(to_np(bufs.ids), ref["ids"])
    assert np.array_equal(to_np(bufs.route_of_row), ref["route_of_row"])
    assert_close(out, ref["out"], "f32")


def test_nan_sentinel_and_determinism():
    """Stale NaN in every compact buffer cannot reach the output; two runs are byte-identical."""
    E, d, f, T, k = 8, 256, 256, 257, 3
    logits, mask = _routing(T, E, k, seed=77, p_mask=0.25)
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, torch.bfloat16, seed=9))
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    for b in (bufs.xs, bufs.h, bufs.y, bufs.out):
        b.fill_(float("nan"))
    out1 = M.moe_forward(logits.cuda(), x, mask.cuda(), wg, wu, wd, k, bufs).clone()
    assert torch.all(torch.isfinite(out1))
    R = int(bufs.offsets[-1])
    assert R < T * k
    for b in (bufs.xs, bufs.h, bufs.y):
        assert torch.all(b[R:].float() == 0)
    out2 = M.moe_forward(logits.cuda(), x, mask.cuda(), wg, wu, wd, k, bufs).clone()
    assert torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    M.moe_check_device_error()


def test_all_masked_output_is_plus_zero():
    E, d, f, T, k = 4, 128, 128, 20, 2
    logits, _ = _routing(T, E, k, seed=5)
    mask = torch.ones(T, k, dtype=torch.uint8).cuda()
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, torch.bfloat16, seed=2))
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    bufs.out.fill_(float("nan"))
    out = M.moe_forward(logits.cuda(), x, mask, wg, wu, wd, k, bufs)
    M.moe_check_device_error()
    assert torch.all(out.view(torch.int32) == 0)  # +0.0 bit pattern everywhere


def test_inconsistent_offsets_are_rejected_on_the_device():
    """offsets[E] beyond the buffer capacity: the kernels skip their work and flag it; nothing hangs."""
    E, d, f, cap = 4, 128, 128, 16
    xs = torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros(E, f, d, dtype=torch.bfloat16, device="cuda")
    h = torch.zeros(cap, f, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(cap, d, dtype=torch.float32, device="cuda")
    offsets = torch.tensor([0, 4, 8, 12, 40], dtype=torch.int32, device="cuda")
    M.moe_grouped_ffn(xs, offsets, wg, wg, wg.transpose(1, 2).contiguous(), h, y)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    assert exc.value.status == M.MOE_ERR_INVALID_ARG
    M.moe_check_device_error()  # the error word was cleared


def test_empty_chunk():
    bufs = M.MoEBuffers(0, 8, 2, 128, 128, torch.bfloat16)
    z = torch.empty(0, 8, device="cuda")
    w = torch.zeros(8, 128, 128, dtype=torch.bfloat16, device="cuda")
    out = M.moe_forward(z, torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"), None, w, w, w, 2, bufs)
    assert out.shape == (0, 128)
    M.moe_check_device_error()


# ---------------------------------------------------------------------------
# full-size workloads: every output of the path against the oracle -- the
# integer outputs bit for bit, h on every compact row within its bf16 rounding
# bound, out on every token within the bf16 tolerance
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_t4", "prefill_t401", "prefill_t2048", "prefill_t8192"])
def test_full_size_workload(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device="cuda")
    bufs = M.MoEBuffers(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f, torch.bfloat16)
    bufs.h.fill_(float("nan"))
    out = M.moe_forward(inp["logits"], inp["x"], inp["mask"], inp["w_gate"], inp["w_up"], inp["w_down"], cfg.k,
                        bufs)
    M.moe_check_device_error()
    ref = full_size_reference(inp)
    assert np.array_equal(to_np(bufs.ids), ref["ids"])
    np.testing.assert_allclose(to_np(bufs.w), ref["w"], rtol=1e-6, atol=0)
    for key in ("counts", "offsets", "row_of_route", "route_of_row"):
        assert np.array_equal(to_np(getattr(bufs, key)), ref[key]), key
    R = int(ref["offsets"][-1])
    assert_close_bf16_rounded(bufs.h[:R], ref["h"])
    assert torch.all(bufs.h[R:].float() == 0)
    st = assert_close(out, ref["out"], "bf16")
    print(f"{name}: all {cfg.T} tokens, {R} compact rows: rel_fro={st['rel_fro']:.2e} "
          f"max/rms={st['max_abs'] / st['rms_ref']:.2e}")


@pytest.mark.parametrize("d,f", [(256, 256), (384, 256)])
def test_big_item_mode_with_light_and_big_items(d, f):
    """Most rows go to two experts (slices of up to 256 rows, the big-item carve-up); the rest stay light."""
    E, T, k = 8, 700, 2
    g = torch.Generator().manual_seed(d)
    logits = torch.randn(T, E, generator=g)
    logits[:, 6] += 3.0
    logits[:, 7] += 2.5
    x = torch.randn(T, d).to(torch.bfloat16)
    wg, wu, wd = _weights(E, d, f, torch.bfloat16, seed=f)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    out = M.moe_forward(logits.cuda(), x.cuda(), None, wg.cuda(), wu.cuda(), wd.cuda(), k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k)
    counts = ref["counts"]
    assert np.maximum(counts - 128, 0).sum() * 2 >= counts.sum()      # the big-item carve-up applies
    assert (counts > 256).sum() >= 2 and ((counts > 0) & (counts <= 128)).sum() >= 2
    h_ref = mo.grouped_swiglu(ref["xs"], ref["offsets"], (to_np(wg), to_np(wu), to_np(wd)))
    R = int(ref["offsets"][-1])
    assert_close_bf16_rounded(bufs.h[:R], h_ref)
    assert_close(out, ref["out"], "bf16")


def test_bound_calls_replay_the_same_path():
    """moe.bind marshals a call once; replaying it gives the direct call's output bit for bit."""
    E, d, f, T, k = 8, 128, 256, 100, 2
    logits, mask = _routing(T, E, k, seed=5, p_mask=0.1)
    x = torch.randn(T, d).to(torch.bfloat16).cuda()
    wg, wu, wd = (w.cuda() for w in _weights(E, d, f, torch.bfloat16, seed=6))
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    m = mask.cuda()
    direct = M.moe_forward(logits.cuda(), x, m, wg, wu, wd, k, bufs).clone()
    bufs.out.zero_()
    # a temporary argument: bind must keep it alive for the replay
    run = M.bind(M.moe_forward, logits.cuda(), x, m, wg, wu, wd, k, bufs)
    torch.empty(T, E, device="cuda").fill_(float("nan"))   # would reuse a freed logits block
    assert torch.all(bufs.out == 0)          # binding does not launch anything
    run()
    run()
    M.moe_check_device_error()
    assert torch.equal(bufs.out, direct)


def test_swiglu_of_large_negative_gates_is_zero_not_nan():
    """Gate pre-activations far below -88 overflow e^-g to infinity: silu must give -0, not NaN."""
    E, d, f, T, k = 2, 128, 128, 40, 1
    logits, _ = _routing(T, E, k, seed=21)
    x = (torch.randn(T, d) * 100.0).to(torch.bfloat16)       # |gate| up to several hundred
    wg, wu, wd = _weights(E, d, f, torch.bfloat16, seed=22)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    out = M.moe_forward(logits.cuda(), x.cuda(), None, wg.cuda(), wu.cuda(), wd.cuda(), k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k)
    h_ref = mo.grouped_swiglu(ref["xs"], ref["offsets"], (to_np(wg), to_np(wu), to_np(wd)))
    assert (h_ref < -1e-30).sum() + (np.abs(h_ref) < 1e-30).sum() > 0
    xs = ref["xs"]
    g = np.concatenate([xs[ref["offsets"][e]:ref["offsets"][e + 1]] @ to_np(wg[e]).astype(np.float64).T
                        for e in range(E) if ref["offsets"][e + 1] > ref["offsets"][e]])
    assert (g < -88).sum() > 100                               # the overflow case is exercised
    assert torch.isfinite(bufs.h[:T].float()).all()
    assert_close_bf16_rounded(bufs.h[:T], h_ref)
    assert_close(out, ref["out"], "bf16")
