"""The multi-rank (replica) logic of bench.py, on CPU with the gloo backend.

The path does not shard across GPUs (one GPU, no collectives): under
torchrun every rank runs an independent replica with its own seed, and the
only collective is the max over ranks of the measured times.  These tests
run two gloo ranks on the CPU.
"""

import json
import os
import socket
import subprocess
import sys
import textwrap

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, {root!r})
    import torch, torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank={rank}, world_size=2)
    rank = dist.get_rank()
    slowest = bench.max_over_ranks(1.5 + 2.0 * rank, 2, "cpu")
    cfg = bench._workload("prefill_t2048", rank)
    dist.barrier()
    dist.destroy_process_group()
    print(json.dumps({{"rank": rank, "slowest": slowest, "seed": cfg.seed, "T": cfg.T}}))
""")


def test_two_gloo_ranks_agree_on_the_slowest_time_and_use_distinct_seeds():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.format(root=ROOT, port=port, rank=r)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert [o["slowest"] for o in outs] == [3.5, 3.5]
    assert outs[0]["seed"] != outs[1]["seed"] and outs[0]["T"] == outs[1]["T"] == 2048


def test_reference_arm_other_ranks_exit_without_work(capsys):
    class A:
        workload = "tiny_fp32"
        steps = 1
        warmup = 3
        reference_budget_s = 1.0
        tokens = 0
        experts = 0
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5


def test_algorithmic_work_counts_touched_experts_only():
    # E = 3 experts, expert 0 untouched; T = 3 tokens, k = 2, one route masked -> R = 5
    counts = np.array([0, 3, 2])
    T, E, k, d, f, es = 3, 3, 2, 128, 256, 2
    w = bench.algorithmic_work(counts, T, E, k, d, f, es)
    assert w["R"] == 5 and w["touched"] == 2
    assert w["gate_up_bytes"] == 2 * (2 * 256 * 128 * 2) + 5 * 128 * 2 + 5 * 256 * 2
    assert w["down_bytes"] == 2 * (128 * 256 * 2) + 5 * 256 * 2 + 5 * 128 * 4
    assert w["flops"] == 6.0 * 5 * 128 * 256
    routing = 3 * 3 * 4 + 3 * 2 * 8
    scatter = 3 * 128 * 2 + 5 * 128 * 2
    combine = 5 * 128 * 4 + 3 * 128 * 4
    assert w["path_bytes"] == routing + scatter + w["gate_up_bytes"] + w["down_bytes"] + combine


def test_algorithmic_work_of_the_fused_permutation():
    """--fused: no combine pass and no y round trip; with the gather, x is read once instead of xs."""
    counts = np.array([0, 3, 2])
    T, E, k, d, f, es = 3, 3, 2, 128, 256, 2
    plain = bench.algorithmic_work(counts, T, E, k, d, f, es)
    compact = bench.algorithmic_work(counts, T, E, k, d, f, es, fused=True)
    gather = bench.algorithmic_work(counts, T, E, k, d, f, es, fused=True, gather=True)
    routing = 3 * 3 * 4 + 3 * 2 * 8
    down = 2 * (128 * 256 * 2) + 5 * 256 * 2 + 3 * 128 * 4          # out written once, y not counted
    assert compact["down_bytes"] == gather["down_bytes"] == down
    assert compact["gate_up_bytes"] == plain["gate_up_bytes"]
    assert gather["gate_up_bytes"] == 2 * (2 * 256 * 128 * 2) + 3 * 128 * 2 + 5 * 256 * 2
    assert compact["path_bytes"] == routing + (3 * 128 * 2 + 5 * 128 * 2) + plain["gate_up_bytes"] + down
    assert gather["path_bytes"] == routing + 3 * 2 * 8 + gather["gate_up_bytes"] + down
    assert gather["flops"] == compact["flops"] == plain["flops"]


def test_workload_overrides_for_profiling_cases():
    cfg = bench._workload("prefill_t2048", 0, tokens=128, experts=32)
    assert (cfg.T, cfg.E, cfg.d, cfg.f, cfg.k) == (128, 32, 4096, 2048, 6)
    assert cfg.name.startswith("prefill_t2048[")
