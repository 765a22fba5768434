"""Device-side failure detection without a GPU fault: a bounded wait that can
never complete gives up, records MOE_ERR_DEVICE_TIMEOUT in the status word,
and the context stays usable for the next layer call."""
import time

import pytest
import torch

from gpu_cases import assert_close, prepared, run_forward
from sparse_moe_ffn_gb300 import binding

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 6


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    binding.moe_selftest_wait_timeout(ws, limit_ns=2_000_000)  # 2 ms
    assert binding.moe_read_device_status(ws) == MOE_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the context is intact: a full layer call still runs and is correct
    import oracle
    shape, dev, bits = prepared("tiny")
    out, _ = run_forward(shape, dev)
    assert_close(out, oracle.moe_forward(bits, shape.k, shape.norm_topk_prob), "after timeout")


def test_status_is_reset_by_the_next_call():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.moe_selftest_wait_timeout(ws, limit_ns=1_000_000)
    assert binding.moe_read_device_status(ws) == MOE_ERR_DEVICE_TIMEOUT
    shape, dev, _ = prepared("tiny")
    big = binding.alloc_workspace(shape.N, shape.H, shape.E, shape.I, shape.k)
    big[:4].copy_(ws[:4])  # a stale error in the status word ...
    run_forward(shape, dev, workspace=big)  # ... is cleared by moe_forward (asserts status 0)
