"""Failure detection without a GPU fault: a pipeline wait that nothing completes
ends after its time bound with a status the host reads, and the context stays
usable for a normal decode step afterwards."""
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import assert_close, run_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hpa.hpa_selftest_wait_timeout(status, 50_000_000)       # 50 ms
    torch.cuda.synchronize()
    assert int(status.item()) & 8
    b = W.make_batch([700, 90], seed=1)
    g = run_gpu(b, num_ctas=3)
    ref, _ = oracle.attention(b)
    assert_close(g["out"], ref, "bf16")
