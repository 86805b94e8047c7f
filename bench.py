"""Benchmark of grouped MoE prefill on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole path (top-k routing, histogram, prefix,
scatter, grouped gate/up+SwiGLU, grouped down, combine) over one synthetic
prefill chunk already resident in HBM.  The default workload is the
2048-token chunk (E=256, top-6, d=4096, f=2048, 10% of routes masked).
Under torchrun each rank runs an independent replica on its own GPU with its
own seed (no data-path collective); value = tokens of all ranks / the
slowest rank's time.

--impl reference times the CPU oracle (C++, float64, OpenMP) on the host cores
on a bounded sample of the same workload, as the reference arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

# chunks up to this size take the fused A1-A4 launch (moe_route_scatter_small)
SMALL_TOKENS, SMALL_ROUTES = 128, 512
METRIC = "grouped MoE prefill tokens/s (T=401/2048/8192, E=256, top-6); % of roofline"
UNIT = "tokens/s"


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples taken every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None
        self.t_start = self.t_end = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu_index), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.45)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        # samples while the GPU was busy (clock above idle) are the "under load" ones
        busy = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time); identity on one rank."""
    if world <= 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def algorithmic_work(counts, T: int, E: int, k: int, d: int, f: int, es: int, fp8: bool = False,
                     fused: bool = False, gather: bool = False, w8a8: bool = False, fp4: bool = False,
                     w4a4: bool = False) -> dict:
    """Algorithmic bytes and FLOPs of one step, from the realised expert counts.

    Only touched experts' weights count; activations are counted once per
    read or write.  es = operand bytes (2 for bf16, 4 for fp32); y and out are
    fp32.  fp8: the expert weights are 1-byte codes plus one fp32 scale per
    output channel (activations stay bf16).  fused: the down kernel writes
    out directly (the combine's y round trip is not counted); with gather the
    gate/up kernel also reads the token rows x itself (no compact copy).
    """
    counts = np.asarray(counts)
    R = int(counts.sum())
    touched = int(np.count_nonzero(counts))
    if w4a4:
        # 4-bit weights and activations: per row of K values, K/2 code bytes, K/16 block-scale bytes and an
        # fp32 scale; h is written in bf16, read back by its quantizer, and read by the down kernel as codes
        rd, rf = d // 2 + d // 16 + 4, f // 2 + f // 16 + 4
        wgu, wdn = touched * 2 * f * rd, touched * d * rf
        gate_up = wgu + R * rd + R * f * 2
        down = wdn + R * rf + R * d * 4
        quant = R * f * 2 + R * rf                           # the rows of h
        scatter = T * d * 2 + T * rd + R * rd                # token rows read, quantized, scattered
        routing = T * E * 4 + T * k * 8
        combine = R * d * 4 + T * d * 4
        return {"R": R, "touched": touched, "gate_up_bytes": gate_up, "down_bytes": down,
                "path_bytes": routing + quant + scatter + gate_up + down + combine, "flops": 6.0 * R * d * f}
    if w8a8:
        # E4M3 weights (codes + channel scales) and E4M3 activations (codes + row scales); h is written in
        # bf16, read back by its quantizer, and read by the down kernel as codes
        wgu, wdn = touched * 2 * f * (d + 4), touched * d * (f + 4)
        gate_up = wgu + R * (d + 4) + R * f * 2
        down = wdn + R * (f + 4) + R * d * 4
        quant = R * f * 2 + R * (f + 4)                     # the rows of h
        scatter = T * d * 2 + T * (d + 4) + R * (d + 4)      # token rows read, quantized, scattered
        routing = T * E * 4 + T * k * 8
        combine = R * d * 4 + T * d * 4
        return {"R": R, "touched": touched, "gate_up_bytes": gate_up, "down_bytes": down,
                "path_bytes": routing + quant + scatter + gate_up + down + combine, "flops": 6.0 * R * d * f}
    wgu = touched * 2 * f * (d + 4) if fp8 else touched * 2 * f * d * es
    wdn = touched * d * (f + 4) if fp8 else touched * d * f * es
    if fp4:   # two codes per byte, an E4M3 scale per 16 values, an fp32 scale per row
        wgu = touched * 2 * f * (d // 2 + d // 16 + 4)
        wdn = touched * d * (f // 2 + f // 16 + 4)
    gate_up = wgu + R * d * es + R * f * es
    down = wdn + R * f * es + R * d * 4
    routing = T * E * 4 + T * k * 8
    scatter = T * d * es + R * d * es
    combine = R * d * 4 + T * d * 4
    if fused:
        down = wdn + R * f * es + T * d * 4
        if gather:
            gate_up = wgu + T * d * es + R * f * es
            scatter = T * k * 8
        return {"R": R, "touched": touched, "gate_up_bytes": gate_up, "down_bytes": down,
                "path_bytes": routing + scatter + gate_up + down, "flops": 6.0 * R * d * f}
    return {"R": R, "touched": touched, "gate_up_bytes": gate_up, "down_bytes": down,
            "path_bytes": routing + scatter + gate_up + down + combine, "flops": 6.0 * R * d * f}


def _workload(name: str, rank: int, tokens: int = 0, experts: int = 0):
    from workloads import CONFIGS
    cfg = CONFIGS[name]
    if tokens or experts:
        cfg = cfg.replace(name=f"{name}[T={tokens or cfg.T},E={experts or cfg.E}]", T=tokens or cfg.T,
                          E=experts or cfg.E)
    if rank:
        cfg = cfg.replace(seed=cfg.seed + 1000 * rank)
    return cfg


def _oracle_inputs(inp, tokens):
    """Host copies of what the oracle needs for a token sample: its logits, rows and mask, and the expert
    banks (bf16, read exactly by the oracle; with FP8 weights (inp["fp8"]) the oracle's own E4M3 codes and
    per-channel scales of the bank).  The bank is copied (and quantized) once per run, outside any timing."""
    from oracle import moe_oracle as mo
    logits = inp["logits"].cpu()[tokens]
    x = inp["x"].cpu()[tokens]
    mask = None if inp["mask"] is None else inp["mask"].cpu()[tokens]
    if "_oracle_bank" not in inp:
        bank = tuple(inp[n].cpu() for n in ("w_gate", "w_up", "w_down"))
        if inp.get("fp4"):
            bank = tuple(mo.quantize_bank_fp4(b) for b in bank)
        elif inp.get("fp8"):
            bank = tuple(mo.quantize_bank_fp8(b) for b in bank)
        inp["_oracle_bank"] = bank
    return logits, x, mask, inp["_oracle_bank"]


def _time_oracle(inp, n_tokens: int):
    """Seconds the oracle takes for the whole path over the first n_tokens tokens."""
    from oracle import moe_oracle as mo
    cfg = inp["cfg"]
    cache = inp.setdefault("_oracle_sample", {})
    if n_tokens not in cache:
        cache.clear()
        cache[n_tokens] = _oracle_inputs(inp, list(range(n_tokens)))
    logits, x, mask, bank = cache[n_tokens]
    forward = (mo.moe_forward_w8a8 if inp.get("w8a8") else mo.moe_forward_w4a4 if inp.get("w4a4") else
               mo.moe_forward)
    t0 = time.perf_counter()
    forward(logits, x, bank, cfg.k, mask)
    return time.perf_counter() - t0


def _oracle_threads():
    from oracle import moe_oracle as mo
    return mo.threads()


def _size_oracle_sample(inp, budget_s: float):
    """Tokens of the oracle sample: sized from a 1-token run, then refined (the
    per-token cost falls as the sampled tokens share experts).

    The oracle reads the host copy of the bank (bf16, or its FP8 codes):
    one copy per run.
    """
    T = inp["cfg"].T
    t1 = _time_oracle(inp, 1)
    n = int(max(1, min(T, budget_s / max(t1, 1e-3))))
    for _ in range(3):
        if n >= T:
            break
        tn = _time_oracle(inp, n)
        if tn >= 0.5 * budget_s:
            break
        n = int(max(1, min(T, n * budget_s / max(tn, 1e-3))))
    return n, t1


def _cpu_desc():
    model = ""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return model


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    from workloads import make_inputs
    cfg = _workload(args.workload, 0, args.tokens, args.experts)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(cfg, device="cpu", weights_device=dev)
    inp["fp8"] = args.weights in ("fp8", "w8a8")
    inp["fp4"] = args.weights in ("fp4", "w4a4")
    inp["w8a8"] = args.weights == "w8a8"
    inp["w4a4"] = args.weights == "w4a4"
    per_step_budget = max(0.05, args.reference_budget_s / max(1, args.steps + args.warmup))
    n, _ = _size_oracle_sample(inp, per_step_budget)
    for _ in range(args.warmup):
        _time_oracle(inp, n)
    total = 0.0
    for _ in range(args.steps):
        total += _time_oracle(inp, n)
    value = n * args.steps / total
    cores = _oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "f": cfg.f, "E": cfg.E, "k": cfg.k,
                   "weights": "fp8_e4m3 codes + fp32 per-channel scales (quantized by the oracle)"
                   if inp["fp8"] else "as drawn"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {n} tokens of the {cfg.T}-token chunk per step (C++ oracle, float64, "
                                   f"OpenMP over {cores} threads)",
                         "cpu": _cpu_desc()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _code_only(text: str) -> str:
    """Source text without comments and blank lines: what the kernels are compiled from."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _src_hash(*names):
    """Hash of the kernel sources (comments ignored) that a stored ncu traffic record belongs to."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sparse_moe_expert_top_gb300", "csrc", n)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    ent = rec.get(kernel, {}).get(workload)
    if not ent or ent.get("src_hash") != _src_hash(*ent.get("sources", [])):
        return None
    return ent["dram_bytes_per_launch"]


def _run_e2e(args, M, world, dev, logits, x, mask, wg, wu, wd, k, bufs, T, d, forward):
    """End to end through the public API: every step copies its inputs from pinned host memory,
    runs the whole path (one moe_forward call) and copies its output back to pinned host memory.

    Chunks are pipelined the way a serving loop would run them: step i+1's inputs are copied in on
    a copy stream while step i computes, and step i's output is copied out on another stream while
    step i+1 computes (inputs and outputs double-buffered; intermediates shared, since the compute
    of consecutive steps is ordered on one stream).
    """
    import copy as _copy
    h_logits = logits.cpu().pin_memory()
    h_x = x.cpu().pin_memory()
    h_mask = None if mask is None else mask.cpu().pin_memory()
    h_out = [torch.empty(T, d, dtype=torch.float32).pin_memory() for _ in range(2)]
    d_logits = [torch.empty_like(logits) for _ in range(2)]
    d_x = [torch.empty_like(x) for _ in range(2)]
    d_mask = [None if mask is None else torch.empty_like(mask) for _ in range(2)]
    bset = [bufs, _copy.copy(bufs)]
    bset[1].out = torch.empty_like(bufs.out)
    h2d = h_logits.numel() * 4 + h_x.numel() * h_x.element_size() + (0 if h_mask is None else h_mask.numel())
    d2h = h_out[0].numel() * 4
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        sl = i & 1
        with torch.cuda.stream(cin):
            cin.wait_event(ev_done[sl])          # step i-2 has consumed this input slot
            d_logits[sl].copy_(h_logits, non_blocking=True)
            d_x[sl].copy_(h_x, non_blocking=True)
            if h_mask is not None:
                d_mask[sl].copy_(h_mask, non_blocking=True)
            ev_in[sl].record(cin)
        comp.wait_event(ev_in[sl])
        comp.wait_event(ev_out[sl])              # step i-2's output has left this slot
        forward(d_logits[sl], d_x[sl], d_mask[sl], wg, wu, wd, k, bset[sl])
        ev_done[sl].record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_done[sl])
            h_out[sl].copy_(bset[sl].out, non_blocking=True)
            ev_out[sl].record(cout)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    last = (args.steps - 1) & 1
    assert torch.equal(h_out[last], bset[last].out.cpu()), "end-to-end output differs from the device result"
    forward(logits, x, mask, wg, wu, wd, k, bufs)
    assert torch.equal(h_out[last], bufs.out.cpu()), "end-to-end output differs from the device-resident run"

    return {"value": world * T * args.steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "pipelining": "inputs of step i+1 copied in and output of step i "
                                                     "copied out while step i / i+1 computes"}


def run_ours(args, rank: int, world: int):
    from sparse_moe_expert_top_gb300 import build as _build
    _build.build()
    from sparse_moe_expert_top_gb300 import moe as M
    from workloads import make_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = _workload(args.workload, rank, args.tokens, args.experts)
    inp = make_inputs(cfg, device=dev)
    T, E, k, d, f = cfg.T, cfg.E, cfg.k, cfg.d, cfg.f
    dtype = inp["x"].dtype
    fp4 = args.weights == "fp4"
    fp8 = args.weights == "fp8" or fp4      # the 4-bit path shares the FP8 path's fp16 activations and kernel
    w8a8 = args.weights == "w8a8"
    w4a4 = args.weights == "w4a4"
    fused = args.fused
    if fused and (fp8 or w8a8 or w4a4 or args.router or dtype != torch.bfloat16):
        raise SystemExit("--fused runs the bf16 path with the workload's logits")
    if (w8a8 or w4a4) and (args.router or dtype != torch.bfloat16):
        raise SystemExit("--weights w8a8 / w4a4 run the bf16 workloads with their logits")
    # the FP8-weight path keeps its compact activations (xs, h) in fp16
    bufs = (M.MoEBuffersW8A8(T, E, k, d, f, device=dev) if w8a8 else
            M.MoEBuffersW4A4(T, E, k, d, f, device=dev) if w4a4 else
            M.MoEBuffers(T, E, k, d, f, torch.float16 if fp8 else dtype, device=dev))
    logits, x, mask = inp["logits"], inp["x"], inp["mask"]
    if w4a4:
        # load-time step, outside the timed region: the 4-bit banks
        inp["fp4"] = inp["w4a4"] = True
        wg, wu, wd = (M.moe_quantize_weights_fp4(inp[n]) for n in ("w_gate", "w_up", "w_down"))
        torch.cuda.synchronize()
        forward = M.moe_forward_w4a4
    elif w8a8:
        # load-time step, outside the timed region: E4M3 codes + per-channel scales
        inp["fp8"] = inp["w8a8"] = True
        wg, wu, wd = (M.moe_quantize_weights_fp8(inp[n]) for n in ("w_gate", "w_up", "w_down"))
        torch.cuda.synchronize()
        forward = M.moe_forward_w8a8
    elif fp8:
        if dtype != torch.bfloat16:
            raise SystemExit("--weights fp8 needs a bf16 workload")
        # load-time step, outside the timed region: FP8 E4M3 codes + per-channel scales
        inp["fp8"] = True
        inp["fp4"] = fp4
        if fp4:
            wg, wu, wd = (M.moe_quantize_weights_fp4(inp[n]) for n in ("w_gate", "w_up", "w_down"))
            gate_up_call, down_call, forward = M.moe_grouped_gate_up_fp4, M.moe_grouped_down_fp4, M.moe_forward_fp4
        else:
            wg, wu, wd = (M.moe_quantize_weights_fp8(inp[n]) for n in ("w_gate", "w_up", "w_down"))
            gate_up_call, down_call, forward = M.moe_grouped_gate_up_fp8, M.moe_grouped_down_fp8, M.moe_forward_fp8
        torch.cuda.synchronize()
        scatter_call = M.moe_scatter_rows_f16
    else:
        wg, wu, wd = inp["w_gate"], inp["w_up"], inp["w_down"]
        gate_up_call, down_call, forward = M.moe_grouped_gate_up, M.moe_grouped_down, M.moe_forward
        scatter_call = M.moe_scatter_rows

    b = bufs
    # every call is marshalled once (M.bind); the timed loop replays the C calls.
    # Small chunks take A1-A4 in one launch, as moe_forward does.
    small = T <= SMALL_TOKENS and T * k <= SMALL_ROUTES and not args.router and not w8a8 and not w4a4
    # fused: moe_forward_fused's automatic choice -- gather the token rows in
    # the gate/up kernel while experts get few rows, else the compact copy;
    # the combine in the down kernel while y fits in twice the L2, else the
    # unfused path
    if fused and args.fused_mode == "auto":
        args.fused_mode = {M.MOE_FUSED_GATHER: "gather", M.MOE_FUSED_COMPACT: "compact",
                           M.MOE_FUSED_NONE: "none"}[M.moe_forward_fused_mode(T, E, k, d)]
    if args.fused_mode == "none":
        fused = False
    gather = fused and args.fused_mode == "gather"
    small = small and not fused
    if w8a8:
        # E4M3 activations: the token rows and h quantized per row, E4M3 x E4M3 tensor-core MMAs; small chunks
        # take the routing, quantization and scatter in one launch, as moe_forward_w8a8 does
        small8 = T <= SMALL_TOKENS and T * k <= SMALL_ROUTES
        names = (("route_scatter_quant_small",) if small8 else ("route", "scatter_quant")) + (
            "gate_up", "quantize_h", "down", "combine")
        routing = []
    elif w4a4:
        # 4-bit activations: the token rows and h quantized by the 4-bit quantizer, block-scaled MMAs; small
        # chunks take the routing, quantization and scatter in one launch, as moe_forward_w4a4 does
        small4 = T <= SMALL_TOKENS and T * k <= SMALL_ROUTES
        names = (("route_scatter_quant_small",) if small4 else ("route", "scatter_quant")) + (
            "gate_up", "quantize_h", "down", "combine")
        routing = []
    elif fused and T <= SMALL_TOKENS and T * k <= SMALL_ROUTES:
        names = ("route_scatter_small", "gate_up", "down_combine")
        routing = [M.bind(M.moe_route_scatter_small_fused, logits, x, mask, k, b, gather)]
    elif fused:
        # the combine runs inside the down kernel
        names = ("route", "scatter_index", "gate_up", "down_combine")
        routing = [
            M.bind(M.moe_route_topk_offsets, logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws),
            M.bind(M.moe_scatter_index, b.ids, mask, b.offsets, d, b.row_of_route, b.route_of_row, b.tile_counts,
                   b.out, b.ws, None if gather else x, None if gather else b.xs),
        ]
    elif args.router:
        # the router projection on the tensor cores replaces the given logits
        if dtype != torch.bfloat16:
            raise SystemExit("--router needs a bf16 workload")
        from workloads.synthetic import make_router_matrix
        wr = make_router_matrix(cfg, dev)
        names = ("router_topk", "histogram", "prefix", "scatter", "gate_up", "down", "combine")
        routing = [
            M.bind(M.moe_router_topk, x, wr, k, b.ids, b.w),
            M.bind(M.moe_route_histogram, b.ids, mask, E, b.counts, b.ws),
            M.bind(M.moe_prefix_offsets, b.counts, T, k, b.offsets, b.ws),
            M.bind(scatter_call, x, b.ids, mask, b.offsets, b.xs, b.row_of_route, b.route_of_row, b.ws),
        ]
    elif small:
        names = ("route_scatter_small", "gate_up", "down", "combine")
        routing = [M.bind(M.moe_route_scatter_small, logits, x, mask, k, b)]
    else:
        # A1-A3 in one launch (moe_route_topk_offsets), then the scatter
        names = ("route", "scatter", "gate_up", "down", "combine")
        routing = [
            M.bind(M.moe_route_topk_offsets, logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws),
            M.bind(scatter_call, x, b.ids, mask, b.offsets, b.xs, b.row_of_route, b.route_of_row, b.ws),
        ]
    GU = names.index("gate_up")
    if fused:
        fmode = M.MOE_FUSED_GATHER if gather else M.MOE_FUSED_COMPACT

        def forward(*a):
            return M.moe_forward_fused(*a, mode=fmode)

        calls = routing + [
            M.bind(M.moe_grouped_gate_up_gather, x, k, b.route_of_row, b.offsets, wg, wu, b.h) if gather else
            M.bind(M.moe_grouped_gate_up, b.xs, b.offsets, wg, wu, b.h),
            M.bind(M.moe_grouped_down_combine, b.h, b.offsets, wd, b.route_of_row, b.row_of_route, b.w, b.y,
                   b.tile_counts, b.out),
        ]
    elif w4a4:
        calls = ([M.bind(M.moe_route_scatter_quant_small_fp4, logits, x, mask, k, b)] if small4 else [
            M.bind(M.moe_route_topk_offsets, logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws),
            M.bind(M.moe_scatter_rows_quant_fp4, x, b.ids, mask, b.offsets, b.x_q, b.xs_q, b.row_of_route,
                   b.route_of_row, b.ws)]) + [
            M.bind(M.moe_grouped_gate_up_w4a4, b.xs_q, b.offsets, wg, wu, b.h),
            M.bind(M.moe_quantize_rows_fp4, b.h, b.h_q),
            M.bind(M.moe_grouped_down_w4a4, b.h_q, b.offsets, wd, b.y),
            M.bind(M.moe_combine, b.y, b.row_of_route, b.w, b.out),
        ]
    elif w8a8:
        calls = ([M.bind(M.moe_route_scatter_quant_small_e4m3, logits, x, mask, k, b)] if small8 else [
            M.bind(M.moe_route_topk_offsets, logits, mask, k, b.ids, b.w, b.counts, b.offsets, b.ws),
            M.bind(M.moe_scatter_rows_quant_e4m3, x, b.ids, mask, b.offsets, b.x_q, b.x_scales, b.xs, b.xs_scales,
                   b.row_of_route, b.route_of_row, b.ws)]) + [
            M.bind(M.moe_grouped_gate_up_w8a8, b.xs, b.xs_scales, b.offsets, wg, wu, b.h),
            M.bind(M.moe_quantize_rows_e4m3, b.h, b.offsets, b.h_q, b.h_scales),
            M.bind(M.moe_grouped_down_w8a8, b.h_q, b.h_scales, b.offsets, wd, b.y),
            M.bind(M.moe_combine, b.y, b.row_of_route, b.w, b.out),
        ]
    elif fp8:
        calls = routing + [
            M.bind(gate_up_call, b.xs, b.offsets, wg, wu, b.h),
            M.bind(down_call, b.h, b.offsets, wd, b.y),
            M.bind(M.moe_combine, b.y, b.row_of_route, b.w, b.out),
        ]
    else:
        # a plan holds the FFN launches' tensor maps, encoded once
        plan = M.moe_plan_create(wg, wu, wd, b)
        calls = routing + [
            M.bind(M.moe_plan_grouped_gate_up, plan),
            M.bind(M.moe_plan_grouped_down, plan),
            M.bind(M.moe_combine, b.y, b.row_of_route, b.w, b.out),
        ]
        if not args.router:
            def forward(lg, xx, mm, _wg, _wu, _wd, _k, bb):
                return M.moe_plan_forward(plan, lg, xx, mm, out=bb.out)

    def step(gu_events=None):
        for i, c in enumerate(calls):
            if gu_events is not None and i == GU:
                gu_events[0].record()
            c()
            if gu_events is not None and i == GU:
                gu_events[1].record()

    for _ in range(args.warmup):
        step()
    M.moe_check_device_error()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    # timed region: the whole path per step; CUDA events around the dominant
    # kernel (grouped gate/up) on its stream give its live launch duration
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    # step boundaries: bnd[s] .. bnd[s+1] is step s; bnd[0] .. bnd[-1] the whole timed region
    bnd = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    bnd[0].record()
    for s in range(args.steps):
        step(ev[s])
        bnd[s + 1].record()
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    M.moe_check_device_error()
    elapsed_ms = max_over_ranks(bnd[0].elapsed_time(bnd[-1]), world, dev)
    step_ms = [bnd[s].elapsed_time(bnd[s + 1]) for s in range(args.steps)]
    step_median = statistics.median(step_ms)
    step_mad = statistics.median(abs(t - step_median) for t in step_ms)
    gu_ms = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps))

    # per-kernel breakdown: a separate loop after the timed region, with events around every call
    n_bd = min(args.steps, 20)
    evk = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in names] for _ in range(n_bd)]
    for s in range(n_bd):
        for i, c in enumerate(calls):
            evk[s][i][0].record()
            c()
            evk[s][i][1].record()
    torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(evk[s][i][0].elapsed_time(evk[s][i][1]) for s in range(n_bd))
                  for i, n in enumerate(names)}

    # host cost of one whole-path call, with the argument checks and tensor-map encoding
    # of moe_forward against a prepared plan (calls marshalled once; the GPU queue
    # absorbs the launches, so the host time per call is what is measured)
    host_us = None
    if not (fused or fp8 or w8a8 or w4a4 or args.router):
        host_us = {}
        for label, call in (("moe_forward", M.bind(M.moe_forward, logits, x, mask, wg, wu, wd, k, b)),
                            ("moe_plan_forward", M.bind(M.moe_plan_forward, plan, logits, x, mask))):
            call()
            torch.cuda.synchronize()
            n_calls = 50
            t0 = time.perf_counter()
            for _ in range(n_calls):
                call()
            host_us[label] = 1e6 * (time.perf_counter() - t0) / n_calls
            torch.cuda.synchronize()
        M.moe_check_device_error()

    # the end-to-end leg runs moe_forward, which takes the logits as input: not with --router
    e2e = None if (args.no_e2e or args.router) else _run_e2e(args, M, world, dev, logits, x, mask, wg, wu, wd, k,
                                                             bufs, T, d, forward)

    if rank != 0:
        return

    # kernels per step: one per call; the fp32 SIMT FFN launches two kernels per projection
    launches_per_step = len(calls) + (2 if dtype == torch.float32 else 0)

    # ---- roofline of the dominant kernel (grouped gate/up + SwiGLU)
    es = 2 if dtype == torch.bfloat16 else 4
    work = algorithmic_work(bufs.counts.cpu().numpy(), T, E, k, d, f, es, fp8, fused, gather, w8a8, fp4, w4a4)
    R, touched = work["R"], work["touched"]
    gate_up_bytes = work["gate_up_bytes"]
    peaks = _peaks()
    achieved = gate_up_bytes / (gu_ms * 1e-3) / 1e9
    # chunks of many routes run the bf16 and E4M3 projections on pairs of SMs (the library's choice)
    paired = dtype == torch.bfloat16 and not (fp8 or fp4 or gather or w4a4) and M.moe_ffn_paired(T * k)
    traffic = _profiled_traffic(("gate_up_w4a4" if w4a4 else "gate_up_w8a8" if w8a8 else "gate_up_fp4" if fp4 else
                                 "gate_up_fp8" if fp8 else "gate_up_gather" if gather else "gate_up") +
                                ("_pair" if paired else ""), cfg.name)
    kname = ("moe_grouped_gate_up_w4a4 (ffn_nvf4_kernel<gated>)" if w4a4 else
             "moe_grouped_gate_up_w8a8 (ffn_pair_kernel<gated, E4M3>)" if w8a8 and paired else
             "moe_grouped_gate_up_w8a8 (ffn_tc_kernel<gated, E4M3>)" if w8a8 else
             "moe_grouped_gate_up_fp4 (ffn_fp8_kernel<gated, FP4>)" if fp4 else
             "moe_grouped_gate_up_fp8 (ffn_fp8_kernel<gated>)" if fp8 else
             "moe_grouped_gate_up_gather (ffn_tc_kernel<gated, fused>)" if gather else
             "moe_grouped_gate_up (ffn_pair_kernel<gated>)" if paired else
             "moe_grouped_gate_up (ffn_tc_kernel<gated>)")
    roofline = {"kernel": kname, "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic, "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": gate_up_bytes, "avg_launch_ms": gu_ms}
    # whole-path roofline: the slower of FLOPs at the dense bf16 tensor peak
    # and the path's algorithmic bytes at HBM bandwidth
    flops, path_bytes = work["flops"], work["path_bytes"]
    if args.router:
        flops += 2.0 * T * E * d
        path_bytes += T * d * 2 + E * d * 2 - T * E * 4   # x and wr read instead of the logits
    # E4M3 x E4M3 MMAs run at twice the bf16 rate (the nominal dense fp8 / bf16 ratio, 4.5 / 2.25 PFLOP/s),
    # 4-bit block-scaled MMAs at six times (13.5 / 2.25)
    tensor_peak = peaks["bf16_tflops_sustained"] * (2.0 if w8a8 else 6.0 if w4a4 else 1.0)
    t_roof = max(flops / (tensor_peak * 1e12), path_bytes / (peaks["hbm_gbs"] * 1e9))
    ms_per_step = elapsed_ms / args.steps
    value = world * T * args.steps / (elapsed_ms * 1e-3)

    # ---- CPU baseline: the oracle on the host cores, bounded sample
    cpu = None
    if not args.no_cpu_baseline and not args.router:
        n, _ = _size_oracle_sample(inp, args.cpu_budget_s)
        secs = _time_oracle(inp, n)
        cores = _oracle_threads()
        cpu = {"value": n / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {n} of {T} tokens, whole path in float64 (C++ oracle, OpenMP over {cores} "
                         f"threads), {secs:.1f} s", "cpu": _cpu_desc()}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": step_median, "ms_per_step_mad": step_mad,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if w8a8 else "e2m1" if w4a4 else ("bf16" if dtype == torch.bfloat16 else "f32"),
        "data": "synthetic",
        "config": {"workload": cfg.name, "T": T, "d": d, "f": f, "E": E, "k": k, "mask_p": cfg.mask_p,
                   "routes_unmasked": R, "experts_touched": touched,
                   "weights": "e2m1 codes + e4m3 scale per 16 + fp32 per-channel scales" if (fp4 or w4a4) else
                              "fp8_e4m3 codes + fp32 per-channel scales" if (fp8 or w8a8) else
                              ("bf16" if dtype == torch.bfloat16 else "f32"),
                   "activations": "fp8_e4m3 codes + fp32 per-row scales (x and h)" if w8a8 else
                                  "e2m1 codes + e4m3 scale per 16 + fp32 per-row scales (x and h)" if w4a4 else
                                  ("fp16 (exact widening of bf16 x)" if fp8 else None),
                   "permutation": ("fused: token rows gathered by the gate/up kernel, weighted combine in the "
                                   "down kernel" if gather else "compact copy xs, weighted combine in the down "
                                   "kernel") if fused else "compact copy xs + separate combine",
                   "router": "x . Wr^T on the tensor cores (moe_router_topk, Wr ~ N(0, 1/d) bf16) in front of "
                             "the histogram; the workload's own logits unused" if args.router else None,
                   "l2": f"inputs larger than L2: "
                         f"{touched * 3 * d * f * (0.5625 if (fp4 or w4a4) else 1 if fp8 else es) / 1e9:.1f} GB of "
                         "touched expert weights streamed per step (L2 129 MB), no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "roofline": roofline,
        "path_roofline": {"flops": flops, "bytes": path_bytes, "t_roof_ms": t_roof * 1e3,
                          "frac": t_roof * 1e3 / ms_per_step,
                          "tflops": flops / (ms_per_step * 1e-3) / 1e12},
        "kernels_ms": per_kernel,
        "host_us_per_call": host_us,
        "kernels_ms_note": "separate loop after the timed region, CUDA events around every call; the timed "
                           "region records events around gate/up only (roofline.avg_launch_ms)",
        "cpu_baseline": cpu,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_routing_sweep(args):
    """Routing-side kernels (top-k, histogram, prefix, scatter, combine) over a T-sweep.

    E = 256, k = 6, 10 % of routes masked; the row width d shrinks as T grows
    so that every case fits a few GB.  Prints one JSON line per T with each
    kernel's time and its achieved bandwidth (algorithmic bytes / time).
    """
    from sparse_moe_expert_top_gb300 import build as _build
    _build.build()
    from sparse_moe_expert_top_gb300 import moe as M

    def timeit(fn, n=args.sweep_reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1e-3

    E, k, dev = 256, 6, "cuda"
    peak = _peaks()["hbm_gbs"]
    sizes = [(2048, 4096), (8192, 4096), (32768, 2048), (131072, 512), (262144, 256)]
    if args.sweep_tokens:
        keep = {int(t) for t in args.sweep_tokens.split(",")}
        sizes = [(T, d) for T, d in sizes if T in keep]
    for T, d in sizes:
        g = torch.Generator(device=dev).manual_seed(T)
        logits = torch.randn(T, E, device=dev, generator=g)
        x = torch.randn(T, d, device=dev, generator=g).to(torch.bfloat16)
        mask = (torch.rand(T, k, device=dev, generator=g) < 0.1).to(torch.uint8)
        cap = T * k
        i32 = dict(dtype=torch.int32, device=dev)
        ids, w = torch.empty(T, k, **i32), torch.empty(T, k, device=dev)
        counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
        ws = torch.zeros(M.moe_workspace_size(T, k) // 4 + 4, **i32)
        xs = torch.empty(cap, d, dtype=torch.bfloat16, device=dev)
        ror, rro = torch.empty(cap, **i32), torch.empty(cap, **i32)
        y = torch.randn(cap, d, device=dev, generator=g)
        out = torch.empty(T, d, device=dev)
        M.moe_route_topk(logits, k, ids, w)
        M.moe_route_histogram(ids, mask, E, counts, ws)
        M.moe_prefix_offsets(counts, T, k, offsets, ws)
        M.moe_scatter_rows(x, ids, mask, offsets, xs, ror, rro, ws)
        M.moe_check_device_error()
        R = int(counts.sum())
        times = {
            "route_topk_offsets": timeit(lambda: M.moe_route_topk_offsets(logits, mask, k, ids, w, counts, offsets,
                                                                          ws)),
            "topk": timeit(lambda: M.moe_route_topk(logits, k, ids, w)),
            "histogram": timeit(lambda: M.moe_route_histogram(ids, mask, E, counts, ws)),
            "prefix": timeit(lambda: M.moe_prefix_offsets(counts, T, k, offsets, ws)),
            "scatter": timeit(lambda: M.moe_scatter_rows(x, ids, mask, offsets, xs, ror, rro, ws)),
            "combine": timeit(lambda: M.moe_combine(y, ror, w, out)),
        }
        M.moe_check_device_error()
        nbytes = {
            "route_topk_offsets": T * E * 4 + T * k * 8 + T * k * 5,
            "topk": T * E * 4 + T * k * 8,
            "histogram": T * k * 9,
            "scatter": T * d * 2 + cap * d * 2 + T * k * 12,
            "combine": R * d * 4 + T * d * 4 + T * k * 8,
        }
        line = {"routing_sweep": True, "T": T, "E": E, "k": k, "d": d, "R": R}
        for name, t in times.items():
            line[name + "_us"] = round(t * 1e6, 2)
            if name in nbytes:
                gbs = nbytes[name] / t / 1e9
                line[name + "_GBs"] = round(gbs)
                line[name + "_frac_of_hbm"] = round(gbs / peak, 3)
        print(json.dumps(line), flush=True)
        del logits, x, xs, y, out, ws
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="prefill_t2048")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller profiling cases)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller profiling cases)")
    ap.add_argument("--weights", choices=("bf16", "fp8", "w8a8", "fp4", "w4a4"), default="bf16",
                    help="expert weight format: the workload's own (bf16); FP8 E4M3 codes with per-channel "
                         "scales quantized at load time, with fp16 activations (fp8) or with E4M3 activations "
                         "quantized per row on the FP8 tensor cores (w8a8); or 4-bit E2M1 codes with an E4M3 "
                         "scale per 16 values and per-channel scales, with fp16 activations (fp4) or with "
                         "activations in the same 4-bit format on the block-scaled tensor cores (w4a4)")
    ap.add_argument("--fused", action="store_true",
                    help="the fused permutation (bf16): rows gathered in the gate/up kernel, combine in the down "
                         "kernel (moe_forward_fused)")
    ap.add_argument("--fused-mode", choices=("auto", "gather", "compact", "none"), default="auto",
                    help="with --fused: rows gathered in the gate/up kernel, the compact copy, or the unfused "
                         "path (auto: moe_forward_fused's choice)")
    ap.add_argument("--router", action="store_true",
                    help="compute the router projection x . Wr^T on the GPU in front of the path (moe_router_topk)")
    ap.add_argument("--routing-sweep", action="store_true",
                    help="time the routing-side kernels over a T-sweep instead (JSON line per T)")
    ap.add_argument("--sweep-tokens", default="", help="with --routing-sweep: the chunk sizes to run (comma list)")
    ap.add_argument("--sweep-reps", type=int, default=20, help="with --routing-sweep: timed launches per kernel")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)
    try:
        if args.routing_sweep:
            run_routing_sweep(args)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
