"""libkvc's C ABI on the CPU: the library loads, exports every symbol that
include/*.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import glob
import os
import re

import pytest

import kv_cache_append_gb300 as kvc
from kv_cache_append_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvc.library()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", text, re.M))
    return sorted(names)


def test_header_declares_entry_points():
    assert {"kvc_step", "kvc_workspace_bytes", "kvc_status_string"} <= set(declared_symbols())


@pytest.mark.parametrize("name", declared_symbols())
def test_symbol_exported(lib, name):
    assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert lib.kvc_version() >= 100
    for code in range(-8, 1):
        assert kvc.status_string(code)
    assert kvc.status_string(-99) == "unknown status"


def _dims(**kw):
    base = dict(B=2, Hq=4, Hk=2, Q=3, D=16, Dv=16, M=32, dtype=0)
    base.update(kw)
    return kvc.make_dims(**base)


def test_workspace_bytes_host_only(lib):
    d = _dims()
    ws = kvc.workspace_bytes(d)
    # one fp32 score per (b, h, t, slot) at least, plus the partials
    assert ws >= 2 * 4 * 3 * 32 * 4 + 2 * 2 * 6 * (16 + 2) * 4
    assert ws % 256 == 0
    assert kvc.workspace_bytes(_dims(Q=0)) == 256           # the fused kernel's work counter
    assert kvc.workspace_bytes(_dims(Hq=3)) == 0          # invalid: Hk does not divide Hq
    big = _dims(B=64, Hq=32, Hk=8, Q=1, D=128, Dv=128, M=8192, dtype=1)
    assert kvc.workspace_bytes(big) >= 64 * 32 * 8192 * 4
    generic = _dims(D=3)                                     # 12-byte rows: generic path
    assert kvc.workspace_bytes(generic) >= 2 * 4 * 3 * 32 * 4


def _call(lib, dims, scale=0.25, null=()):
    ptrs = {n: ctypes.c_void_p(4096 * (i + 1)) for i, n in enumerate(
        ["q", "nk", "nv", "kc", "vc", "len", "mask", "ok", "ov", "ol", "oa", "oc", "ws"])}
    for n in null:
        ptrs[n] = None
    return lib.kvc_step(ctypes.byref(dims) if dims is not None else None,
                        ptrs["q"], ptrs["nk"], ptrs["nv"], ptrs["kc"], ptrs["vc"],
                        ptrs["len"], ptrs["mask"], ctypes.c_double(scale), ptrs["ok"],
                        ptrs["ov"], ptrs["ol"], ptrs["oa"], ptrs["oc"], ptrs["ws"],
                        1 << 30, None, None)


def test_argument_errors_return_before_any_launch(lib):
    assert _call(lib, None) == -1                          # KVC_E_NULL
    assert _call(lib, _dims(dtype=7)) == -3                # KVC_E_DTYPE
    assert _call(lib, _dims(Hq=3)) == -2                   # KVC_E_SHAPE
    assert _call(lib, _dims(Q=-1)) == -2
    assert _call(lib, _dims(M=0)) == -2
    assert _call(lib, _dims(B=0)) == -2
    assert _call(lib, _dims(), null=("kc",)) == -1
    assert _call(lib, _dims(), null=("q",)) == -1          # query needed when Q > 0
    assert _call(lib, _dims(), scale=0.0) == -4            # KVC_E_SCALE
    assert _call(lib, _dims(), scale=-1.0) == -4
    assert _call(lib, _dims(), scale=float("nan")) == -4
    assert _call(lib, _dims(), scale=float("inf")) == -4


def test_binding_rejects_cpu_tensors():
    import torch
    z = torch.zeros(1, 1, 1, 4)
    with pytest.raises(ValueError, match="CUDA"):
        kvc.kv_cache_attention_step(z, z, z, torch.zeros(1, 1, 4, 4), torch.zeros(1, 1, 4, 4),
                                    torch.zeros(1, dtype=torch.int64),
                                    torch.ones(1, 1, dtype=torch.bool), {})


def test_binding_rejects_unknown_option():
    with pytest.raises(ValueError, match="only key"):
        kvc.kvc._scale_from({"scale": 0.5, "dropout": 0.1}, 16)
    assert kvc.kvc._scale_from({}, 16) == 0.25


def _call_inplace(lib, dims, scale=0.25, null=()):
    ptrs = {n: ctypes.c_void_p(4096 * (i + 1)) for i, n in enumerate(
        ["q", "nk", "nv", "kc", "vc", "len", "mask", "ol", "oa", "oc", "ws"])}
    for n in null:
        ptrs[n] = None
    return lib.kvc_step_inplace(ctypes.byref(dims) if dims is not None else None,
                                ptrs["q"], ptrs["nk"], ptrs["nv"], ptrs["kc"], ptrs["vc"],
                                ptrs["len"], ptrs["mask"], ctypes.c_double(scale), ptrs["ol"],
                                ptrs["oa"], ptrs["oc"], ptrs["ws"], 1 << 30, None, None)


def test_inplace_argument_errors_return_before_any_launch(lib):
    assert _call_inplace(lib, None) == -1                   # KVC_E_NULL
    assert _call_inplace(lib, _dims(dtype=7)) == -3         # KVC_E_DTYPE
    assert _call_inplace(lib, _dims(Hq=3)) == -2            # KVC_E_SHAPE
    assert _call_inplace(lib, _dims(), null=("kc",)) == -1  # the donated caches are required
    assert _call_inplace(lib, _dims(), null=("vc",)) == -1
    assert _call_inplace(lib, _dims(), null=("ol",)) == -1
    assert _call_inplace(lib, _dims(), null=("q",)) == -1
    assert _call_inplace(lib, _dims(), scale=0.0) == -4     # KVC_E_SCALE


def test_attend_cache_workspace_and_argument_errors(lib):
    d = _dims(Q=4)
    ws = lib.kvc_attend_cache_workspace_bytes(ctypes.byref(d))
    assert ws >= kvc.workspace_bytes(d) + 2 * 4 * 4 * (16 + 16) * 4
    assert lib.kvc_attend_cache_workspace_bytes(ctypes.byref(_dims(Hq=3))) == 0
    p = [ctypes.c_void_p(4096 * (i + 1)) for i in range(8)]

    def call(dims, num_slots=4, total_q=5, scale=0.5, null=(), k_cum=0):
        a = list(p)
        for i in null:
            a[i] = None
        # q, key_cache, value_cache, cu_q, seqlens_k, slot_ids, out, workspace
        return lib.kvc_attend_cache(ctypes.byref(dims) if dims is not None else None,
                                    num_slots, total_q, a[0], a[1], a[2], a[3], a[4], k_cum,
                                    a[5], ctypes.c_double(scale), a[6], a[7], 1 << 30, None,
                                    None)
    assert call(None) == -1                       # KVC_E_NULL
    assert call(_dims(Hq=3)) == -2                # KVC_E_SHAPE
    assert call(d, num_slots=0) == -2
    assert call(d, total_q=-1) == -2
    assert call(d, k_cum=2) == -2
    assert call(d, num_slots=1, null=(5,)) == -2  # identity slots need num_slots >= B
    assert call(d, null=(1,)) == -1               # key_cache
    assert call(d, null=(0,)) == -1               # q
    assert call(d, null=(6,)) == -1               # out
    assert call(d, scale=-2.0) == -4              # KVC_E_SCALE
