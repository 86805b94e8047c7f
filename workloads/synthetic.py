"""Seeded synthetic workloads shaped like the prefill chunks of the MoE pages.

The pages ("perf(ds4): batch heterogeneous MoE prefill by expert", Summary and
"Original matched qualification") measure a DeepSeek-V4 Flash model on
401-, 2048- and 8192-token prefill chunks with 256 routed experts and top-6
routing.  No model, prompt or weights are available, so every tensor here is a
seeded random draw with those shapes.

Distribution conventions (each one is a reading of the workload text):

* ``N(0, v)`` names the VARIANCE ``v``; expert weights are ``N(0, 1/fan_in)``
  so a unit-variance input keeps unit-scale projections.
* Token rows ``X`` are ``N(0, 1)``, rounded to bf16 for the bf16 workloads.
* Router logits are ``N(0, 1)`` per (token, expert).  The 2048-token workload
  adds a per-expert bias ``b_e ~ N(0, 0.5)``.  The 8192-token workload adds
  ``ln p_{pi(e)}`` with ``p_r ~ r^-1.1`` over a seeded permutation ``pi`` of
  the experts, which leaves some experts with no route and a few with more
  than a thousand.
* The tiny fp32 workload draws a router matrix ``Wr ~ N(0, 1/d)`` and hands
  the router projection ``X @ Wr`` (evaluated in float64, stored as float32)
  to both sides as the logits: the router projection is an input of the routed
  path, not one of its steps.
* The owner mask of the 2048-token workload is a Bernoulli(0.1) draw over the
  ``T x k`` (token, slot) routes; ``1`` means "masked: not owned here".

Weight storage is K-contiguous (the nn.Linear convention): ``w_gate`` and
``w_up`` are ``[E][f][d]`` and ``w_down`` is ``[E][d][f]``.

Every tensor is drawn from its own ``torch.Generator`` seeded from
(workload seed, tensor tag), so a tensor does not depend on which other
tensors were drawn first.  Draws made on a CUDA device use torch's CUDA
generator and differ from CPU draws with the same seed; a caller that needs
the same values on both sides draws once and copies.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# Tags that separate the per-tensor random streams of one workload.
_TAG_LOGITS = 1
_TAG_TOKENS = 2
_TAG_GATE = 3
_TAG_UP = 4
_TAG_DOWN = 5
_TAG_MASK = 6
_TAG_BIAS = 7
_TAG_PERM = 8
_TAG_ROUTER = 9
_TAG_ROUTER_ROWS = 10


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """Shape and draw recipe of one workload."""

    name: str
    T: int          # tokens in the chunk
    d: int          # hidden size
    f: int          # expert FFN size
    E: int          # routed experts
    k: int          # experts per token
    dtype: str      # "f32" or "bf16": operand type of X and the expert weights
    seed: int
    logits: str     # "router" | "normal" | "normal_bias" | "zipf"
    bias_var: float = 0.0
    zipf_s: float = 0.0
    mask_p: float = 0.0

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def routes(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny_fp32": MoEConfig("tiny_fp32", T=32, d=64, f=128, E=8, k=2, dtype="f32", seed=0, logits="router"),
    "prefill_t401": MoEConfig("prefill_t401", T=401, d=4096, f=2048, E=256, k=6, dtype="bf16", seed=1,
                              logits="normal"),
    "prefill_t2048": MoEConfig("prefill_t2048", T=2048, d=4096, f=2048, E=256, k=6, dtype="bf16", seed=2,
                               logits="normal_bias", bias_var=0.5, mask_p=0.1),
    "prefill_t8192": MoEConfig("prefill_t8192", T=8192, d=4096, f=2048, E=256, k=6, dtype="bf16", seed=3,
                               logits="zipf", zipf_s=1.1),
    "verify_t4": MoEConfig("verify_t4", T=4, d=4096, f=2048, E=256, k=6, dtype="bf16", seed=4, logits="normal"),
}


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tag * 7919 + 17)
    return g


def _torch_dtype(dtype: str) -> torch.dtype:
    if dtype == "f32":
        return torch.float32
    if dtype == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown operand dtype {dtype!r}")


def make_tokens(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Token rows X [T][d], N(0, 1), in the workload's operand dtype."""
    g = _gen(cfg.seed, _TAG_TOKENS, device)
    x = torch.randn(cfg.T, cfg.d, generator=g, device=device, dtype=torch.float32)
    return x.to(_torch_dtype(cfg.dtype))


def make_logits(cfg: MoEConfig, x: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Router logits [T][E] float32 on the CPU (see the module docstring)."""
    T, E = cfg.T, cfg.E
    if cfg.logits == "router":
        if x is None:
            x = make_tokens(cfg, "cpu")
        g = _gen(cfg.seed, _TAG_ROUTER, "cpu")
        wr = torch.randn(cfg.d, E, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(cfg.d))
        return (x.cpu().double() @ wr.double()).float()
    g = _gen(cfg.seed, _TAG_LOGITS, "cpu")
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    if cfg.logits == "normal":
        return logits
    if cfg.logits == "normal_bias":
        gb = _gen(cfg.seed, _TAG_BIAS, "cpu")
        bias = torch.randn(E, generator=gb, dtype=torch.float32) * math.sqrt(cfg.bias_var)
        return logits + bias[None, :]
    if cfg.logits == "zipf":
        gp = _gen(cfg.seed, _TAG_PERM, "cpu")
        rank = torch.randperm(E, generator=gp) + 1  # rank of expert e in 1..E
        log_p = -cfg.zipf_s * torch.log(rank.double())
        log_p = log_p - torch.logsumexp(log_p, 0)
        return (logits.double() + log_p[None, :]).float()
    raise ValueError(f"unknown logits recipe {cfg.logits!r}")


def make_mask(cfg: MoEConfig) -> Optional[torch.Tensor]:
    """Owner mask u8 [T][k] (1 = route masked), or None when nothing is masked."""
    if cfg.mask_p <= 0.0:
        return None
    g = _gen(cfg.seed, _TAG_MASK, "cpu")
    return (torch.rand(cfg.T, cfg.k, generator=g) < cfg.mask_p).to(torch.uint8)


def _randn_scaled(shape, scale: float, dtype: torch.dtype, g: torch.Generator, device, chunk: int) -> torch.Tensor:
    """N(0, scale^2) draw of ``shape`` (leading dim chunked to bound float32 temporaries)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    for lo in range(0, shape[0], chunk):
        hi = min(shape[0], lo + chunk)
        tmp = torch.randn((hi - lo,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        tmp.mul_(scale)
        out[lo:hi].copy_(tmp)
    return out


def make_weights(cfg: MoEConfig, device="cpu", chunk: int = 8):
    """Expert weights (w_gate [E][f][d], w_up [E][f][d], w_down [E][d][f]) ~ N(0, 1/fan_in)."""
    dt = _torch_dtype(cfg.dtype)
    E, d, f = cfg.E, cfg.d, cfg.f
    wg = _randn_scaled((E, f, d), 1.0 / math.sqrt(d), dt, _gen(cfg.seed, _TAG_GATE, device), device, chunk)
    wu = _randn_scaled((E, f, d), 1.0 / math.sqrt(d), dt, _gen(cfg.seed, _TAG_UP, device), device, chunk)
    wd = _randn_scaled((E, d, f), 1.0 / math.sqrt(f), dt, _gen(cfg.seed, _TAG_DOWN, device), device, chunk)
    return wg, wu, wd


def make_router_matrix(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Router matrix Wr [E][d] ~ N(0, 1/d) in the workload's operand dtype, stored
    K-contiguous like the expert weights, for runs that compute the router
    projection X . Wr^T themselves (unit-variance logits for unit-variance X)."""
    g = _gen(cfg.seed, _TAG_ROUTER_ROWS, device)
    return _randn_scaled((cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d), _torch_dtype(cfg.dtype), g, device, 64)


def make_inputs(cfg: MoEConfig, device="cpu", weights_device=None) -> dict:
    """All inputs of one workload.

    ``logits``, ``mask`` and ``x`` are drawn on the CPU and moved to ``device``;
    the expert weights are drawn directly on ``weights_device`` (default
    ``device``) because the full-size bank is 12.9 GB.
    """
    x = make_tokens(cfg, "cpu")
    logits = make_logits(cfg, x)
    mask = make_mask(cfg)
    wdev = device if weights_device is None else weights_device
    wg, wu, wd = make_weights(cfg, wdev)
    return {
        "cfg": cfg,
        "logits": logits.to(device),
        "x": x.to(device),
        "mask": None if mask is None else mask.to(device),
        "w_gate": wg,
        "w_up": wu,
        "w_down": wd,
    }
