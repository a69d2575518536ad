"""The failure path of the pipeline waits, on the GPU, without a fault: a
kernel whose mbarrier is never arrived at gives up after its limit, reports
KVC_DEV_TIMEOUT through the status word, and leaves the context usable (a
step right after it matches the oracle)."""
import time

import pytest
import torch

import kv_cache_append_gb300 as kvc
import workloads
from test_gpu_parity import DEV, SMALL, _built, compare_full, run_gpu  # noqa: F401

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvc.selftest_wait_timeout(status, limit_ns=5_000_000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == kvc.DEV_TIMEOUT
    assert 0.005 <= elapsed < 5.0
    # the context still runs kernels correctly
    x = workloads.generate(SMALL["decode_bf16_ragged_M"], 0)
    out, st = run_gpu(x.to(DEV))
    compare_full(x, out, st)


def test_status_bits_accumulate_and_limits_are_checked():
    status = torch.full((1,), kvc.DEV_MASK, dtype=torch.int32, device=DEV)
    kvc.selftest_wait_timeout(status, limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == kvc.DEV_MASK | kvc.DEV_TIMEOUT
    with pytest.raises(kvc.KvcError):
        kvc.selftest_wait_timeout(status, limit_ns=10)
    with pytest.raises(kvc.KvcError):
        kvc.selftest_wait_timeout(status, limit_ns=10**9)
