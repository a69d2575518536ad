"""The two-pass tensor-core step, a compile-time alternative of the
one-pass step with stored P rows (built with -DKVC_TC_TWO_PASS=1).

For one row group (at most 128 query rows per KV head), out of place, with
M a multiple of 8, the two-pass form works every unit twice: a first pass
over the key prefix keeps each row's softmax maximum and sum, and the second
pass copies the caches and writes the normalised attention rows directly, so
no P rows are stored and read back. On one GB300 it measured slower than the
default one-pass form, so the default build does not take it; this test
builds that variant of libkvc and runs the tensor-core parity tests, the
long-context full-size check and the guard-band tests against it in a child
process (the binding loads one library per process, named by KVC_LIBRARY).
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_two_pass_variant_parity():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, ROOT)
    from kv_cache_append_gb300 import build as kbuild
    lib = kbuild.build_variant("2pass", ["KVC_TC_TWO_PASS=1"])
    env = dict(os.environ, KVC_LIBRARY=lib, KVC_EXPECT_TWO_PASS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
           os.path.join(HERE, "test_gpu_parity.py"), os.path.join(HERE, "test_gpu_guard_bands.py"),
           "-k", "tensor or two_pass or long_mqa or poison or step_writes"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "passed" in r.stdout
