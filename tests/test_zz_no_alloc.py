"""kvc_step_static: the step for callers that cannot allocate device memory.

Such callers (a serving loop whose device memory is all reserved up front, a
plugin whose host framework owns the allocator, code that cannot accept
cudaMalloc's device-wide synchronisation) pass inputs and outputs but no
workspace; the library keeps the scratch in one static device array. These
tests call that entry point through the C ABI, several times in a row on
different shapes and inputs (CUDA-core and tensor-core paths, whose scratch
layouts differ), so scratch left by one call must not leak into the next.
Each result must equal kvc_step's on the same inputs bit for bit (both run
the same deterministic kernels), one of them is also checked against the
oracle, and calls after the first on a device must not change the device's
free memory. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import kv_cache_append_gb300 as kvc
import workloads
from workloads import Spec

pytestmark = pytest.mark.gpu

STATIC_LIMIT = 96 << 20
KVC_E_STATIC_LIMIT = -9


@pytest.fixture(scope="module")
def lib():
    from kv_cache_append_gb300 import build as kbuild
    kbuild.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kvc.library()


def _p(t):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _bits(t):
    if not t.is_floating_point():
        return t
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def call_static(lib, x, out, status):
    q, nk, nv, kc, vc, ln, mk = x.args()
    mk = mk.view(torch.uint8)
    dims = kvc.dims_of(q, kc, vc)
    scale = x.options.get("scale", kvc.default_scale(q.shape[-1]))
    rc = lib.kvc_step_static(ctypes.byref(dims), _p(q), _p(nk), _p(nv), _p(kc), _p(vc), _p(ln),
                             _p(mk), ctypes.c_double(scale), _p(out["key_cache"]),
                             _p(out["value_cache"]), _p(out["lengths"]), _p(out["attention"]),
                             _p(out["context"]), _p(status),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, kvc.status_string(rc)


SPECS = [
    # CUDA-core path (8 rows per KV head), Zipf lengths, some rows append nothing
    Spec(B=8, Hq=8, Hk=2, Q=2, D=128, Dv=128, M=777, dtype="bf16", lengths=("zipf", 1.2),
         counts=("uniform", 0, 2)),
    # tensor-core path (128 rows per KV head): fp16 P rows and partials in the scratch
    Spec(B=2, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=3000, dtype="f16",
         lengths=("uniform", 2000, 2992), std=0.5, scale=0.05),
    # decode shape (CUDA-core path), after the tensor-core call's leftovers
    Spec(B=4, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=2000, dtype="bf16",
         lengths=("uniform", 100, 1999)),
    # tensor-core path again, two row groups, after a call of another shape
    Spec(B=2, Hq=8, Hk=2, Q=40, D=64, Dv=64, M=600, dtype="bf16",
         lengths=("uniform", 100, 500)),
]


def test_static_entry_matches_kvc_step_call_after_call(lib):
    dev = torch.device("cuda:0")
    for i, spec in enumerate(SPECS):
        x = workloads.generate(spec, 40 + i, device=dev)
        dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
        assert kvc.workspace_bytes(dims) <= STATIC_LIMIT
        ref = kvc.kv_cache_attention_step(*x.args(), x.options)   # kvc_step (loads its kernels)
        out = kvc.allocate_outputs(x.query, x.key_cache, x.value_cache)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info(dev)[0]
        call_static(lib, x, out, status)
        torch.cuda.synchronize()
        if i > 0:   # the first call on the device is the set-up
            assert torch.cuda.mem_get_info(dev)[0] == free0
        assert int(status.item()) == 0
        for k in ("key_cache", "value_cache", "lengths", "attention", "context"):
            assert torch.equal(_bits(out[k]), _bits(ref[k])), (i, k)
        if i == 1:
            from test_gpu_parity import compare_full
            compare_full(x.to("cpu"), out, int(status.item()))
        del ref, out, x


def test_static_entry_rejects_sizes_beyond_its_scratch(lib):
    # ragged_specdec needs ~2 GB of scratch: rejected before anything runs
    dims = kvc.make_dims(256, 32, 8, 4, 128, 128, 16384, torch.bfloat16)
    assert kvc.workspace_bytes(dims) > STATIC_LIMIT
    rc = lib.kvc_step_static(ctypes.byref(dims), *([ctypes.c_void_p(4096)] * 7),
                             ctypes.c_double(0.1), *([ctypes.c_void_p(8192)] * 5), None, None)
    assert rc == KVC_E_STATIC_LIMIT
    assert "KVC_STATIC_SCRATCH_BYTES" in kvc.status_string(rc)
