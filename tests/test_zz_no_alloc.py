"""kvc_step_static: the step for callers that cannot allocate device memory.

Such callers (a serving loop whose device memory is all reserved up front, a
plugin whose host framework owns the allocator, code that cannot accept
cudaMalloc's device-wide synchronisation) pass inputs and outputs but no
workspace; the library keeps the scratch in one static device array. These
tests call that entry point through the C ABI and check it against kvc_step
on the same inputs, on two calls in a row with different inputs, so scratch
left by the first call must not leak into the second. This file is collected
last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import kv_cache_append_gb300 as kvc
import workloads
from workloads import Spec

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-5, 1e-4), torch.bfloat16: (4e-3, 2e-2), torch.float16: (4e-3, 2e-2)}
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
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def call_static(lib, x):
    q, nk, nv, kc, vc, ln, mk = x.args()
    mk = mk.view(torch.uint8)
    dims = kvc.dims_of(q, kc, vc)
    out = kvc.allocate_outputs(q, kc, vc)
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    scale = x.options.get("scale", kvc.default_scale(q.shape[-1]))
    rc = lib.kvc_step_static(ctypes.byref(dims), _p(q), _p(nk), _p(nv), _p(kc), _p(vc), _p(ln),
                             _p(mk), ctypes.c_double(scale), _p(out["key_cache"]),
                             _p(out["value_cache"]), _p(out["lengths"]), _p(out["attention"]),
                             _p(out["context"]), _p(status),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, kvc.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


SPECS = [
    Spec(B=8, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=777, dtype="bf16", lengths=("zipf", 1.2),
         counts=("uniform", 0, 4)),
    Spec(B=4, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=2000, dtype="bf16",
         lengths=("uniform", 100, 1999)),
]


def test_static_entry_matches_kvc_step_on_two_calls(lib):
    dev = torch.device("cuda:0")
    for seed, spec in enumerate(SPECS):
        x = workloads.generate(spec, seed + 40, device=dev)
        assert kvc.workspace_bytes(kvc.dims_of(x.query, x.key_cache, x.value_cache)) <= STATIC_LIMIT
        ref = kvc.kv_cache_attention_step(*x.args(), x.options)   # kvc_step
        got = call_static(lib, x)
        torch.cuda.synchronize()
        assert torch.equal(_bits(got["key_cache"]), _bits(ref["key_cache"]))
        assert torch.equal(_bits(got["value_cache"]), _bits(ref["value_cache"]))
        assert torch.equal(got["lengths"], ref["lengths"])
        atol_a, atol_c = TOL[x.query.dtype]
        np.testing.assert_allclose(got["attention"].double().cpu().numpy(),
                                   ref["attention"].double().cpu().numpy(), rtol=0, atol=atol_a)
        np.testing.assert_allclose(got["context"].double().cpu().numpy(),
                                   ref["context"].double().cpu().numpy(), rtol=0, atol=atol_c)


def test_static_entry_rejects_sizes_beyond_its_scratch(lib):
    # ragged_specdec needs ~2 GB of scratch: rejected before anything runs
    dims = kvc.make_dims(256, 32, 8, 4, 128, 128, 16384, torch.bfloat16)
    assert kvc.workspace_bytes(dims) > STATIC_LIMIT
    rc = lib.kvc_step_static(ctypes.byref(dims), *([ctypes.c_void_p(4096)] * 7),
                             ctypes.c_double(0.1), *([ctypes.c_void_p(8192)] * 5), None, None)
    assert rc == KVC_E_STATIC_LIMIT
    assert "KVC_STATIC_SCRATCH_BYTES" in kvc.status_string(rc)
