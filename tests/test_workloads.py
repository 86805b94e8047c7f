"""The seeded input generator: reproducible draws with the workloads' structure."""

import numpy as np
import torch

from oracle import moe_oracle as mo
from workloads import CONFIGS, make_inputs, make_logits, make_mask, make_tokens


def test_draws_are_reproducible_and_independent_per_tensor():
    cfg = CONFIGS["tiny_fp32"]
    a, b = make_inputs(cfg), make_inputs(cfg)
    for key in ("logits", "x", "w_gate", "w_up", "w_down"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["w_gate"], a["w_up"])
    assert a["mask"] is None
    assert a["w_gate"].shape == (8, 128, 64) and a["w_down"].shape == (8, 64, 128)
    assert a["x"].dtype == torch.float32 and a["logits"].dtype == torch.float32


def test_bf16_shapes_and_scale():
    cfg = CONFIGS["prefill_t401"].replace(E=4, d=256, f=128)
    inp = make_inputs(cfg)
    assert inp["x"].dtype == torch.bfloat16 and inp["w_gate"].dtype == torch.bfloat16
    # N(0, 1/fan_in): the sample variance times fan_in is close to 1
    assert abs(inp["w_gate"].float().var().item() * 256 - 1.0) < 0.05
    assert abs(inp["w_down"].float().var().item() * 128 - 1.0) < 0.05
    assert abs(inp["x"].float().var().item() - 1.0) < 0.05


def test_mask_rate_of_the_medium_chunk():
    cfg = CONFIGS["prefill_t2048"]
    m = make_mask(cfg)
    assert m.shape == (2048, 6) and m.dtype == torch.uint8
    assert 0.08 < m.float().mean().item() < 0.12


def test_zipf_chunk_has_empty_and_heavy_experts():
    cfg = CONFIGS["prefill_t8192"]
    ids, _ = mo.route_topk(make_logits(cfg).numpy(), cfg.k)
    counts = mo.route_histogram(ids, None, cfg.E)
    assert np.count_nonzero(counts == 0) > 50
    assert np.count_nonzero(counts > 1000) >= 3


def test_tiny_logits_are_the_router_projection():
    cfg = CONFIGS["tiny_fp32"]
    x = make_tokens(cfg)
    lg = make_logits(cfg, x)
    assert lg.shape == (32, 8) and lg.dtype == torch.float32
    assert torch.equal(lg, make_logits(cfg))
