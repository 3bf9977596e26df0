"""Device-side failure detection without a GPU fault: a bounded wait that runs
out reports NA_ERR_DEVICE_TIMEOUT in the caller's status word, the kernel
returns, and the context keeps working.  This file runs last so that a failure
here leaves every other test already run."""
import time

import pytest
import torch

import workloads as W
from harness import gpu_decode

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    import causal_gqa_attention_rope_gb300 as na
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    na.na_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == na.NA_ERR_DEVICE_TIMEOUT
    assert elapsed < 60, f"the wait took {elapsed:.1f} s"
    # the context is intact: a decode afterwards runs and matches a second run
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128), [100, 37], capacity=128, seed=3)
    a, _, st_a = gpu_decode(dec, with_probs=False)
    b, _, st_b = gpu_decode(dec, with_probs=False)
    assert st_a == 0 and st_b == 0
    assert torch.equal(a, b)
