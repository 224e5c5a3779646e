"""Failure detection on the GPU without a fault: a bounded inter-block wait
whose predecessor never publishes must give up, report
EF_ERR_DEVICE_TIMEOUT through the workspace status word, and leave the
context usable for the next call."""

import time

import pytest
import torch

import error_feedback_gradient_gb300 as efg
from error_feedback_gradient_gb300 import binding
from efcheck import check_topk_step
from error_feedback_gradient_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
EF_ERR_DEVICE_TIMEOUT = 12


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.empty(512, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    binding.selftest_wait_timeout(ws, 50_000_000)          # 50 ms
    assert efg.workspace_status(ws) == EF_ERR_DEVICE_TIMEOUT
    dt = time.perf_counter() - t0
    assert 0.04 < dt < 5.0
    # the next call still works and is still exact
    n = 70_001
    check_topk_step(wl.student_t3(n, 1e-3, 1, "cuda"), torch.zeros(n, device="cuda"), [0, n], [70])


def test_selftest_rejects_bad_arguments():
    ws = torch.empty(512, dtype=torch.uint8, device="cuda")
    with pytest.raises(efg.EFError):
        binding.selftest_wait_timeout(ws, 10)              # below 1 ms
    with pytest.raises(efg.EFError):
        binding.selftest_wait_timeout(ws[:100], 50_000_000)
