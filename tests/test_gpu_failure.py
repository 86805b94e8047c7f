"""Failure detection on the GPU without a fault.

A bounded wait that runs out must turn into MOE_ERR_TIMEOUT on the host,
clear on the next check, and leave the CUDA context usable.
"""

import time

import numpy as np
import pytest
import torch

from oracle import moe_oracle as mo
from sparse_moe_expert_top_gb300 import moe as M
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu


def test_a_bounded_wait_that_runs_out_reports_a_timeout():
    M.moe_check_device_error()  # start clean
    t0 = time.perf_counter()
    M.moe_selftest_bounded_wait(50)
    with pytest.raises(M.MoEError) as exc:
        M.moe_check_device_error()
    elapsed = time.perf_counter() - t0
    assert exc.value.status == M.MOE_ERR_TIMEOUT
    assert 0.04 < elapsed < 10.0
    M.moe_check_device_error()  # the word was cleared


def test_the_context_stays_usable_after_a_timeout():
    M.moe_selftest_bounded_wait(10)
    with pytest.raises(M.MoEError):
        M.moe_check_device_error()
    T, E, k, d, f = 40, 4, 2, 128, 128
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(T, E, generator=g)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, f, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, d, f, generator=g) / f ** 0.5).to(torch.bfloat16)
    bufs = M.MoEBuffers(T, E, k, d, f, torch.bfloat16)
    out = M.moe_forward(logits.cuda(), x.cuda(), None, wg.cuda(), wu.cuda(), wd.cuda(), k, bufs)
    M.moe_check_device_error()
    ref = mo.moe_forward(logits.numpy(), to_np(x), (to_np(wg), to_np(wu), to_np(wd)), k)
    assert np.array_equal(to_np(bufs.ids), ref["ids"])
    assert_close(out, ref["out"], "bf16")


def test_selftest_rejects_limits_out_of_range():
    for bad in (0, 5001):
        with pytest.raises(M.MoEError) as exc:
            M.moe_selftest_bounded_wait(bad)
        assert exc.value.status == M.MOE_ERR_INVALID_ARG
