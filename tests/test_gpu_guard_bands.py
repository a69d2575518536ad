"""Write-bounds checks: every buffer a call receives sits inside guard bands.

A kernel that writes past the end (or before the start) of an output, the
workspace, the status word or an input would pass the parity tests as long as
the bytes it hit were not compared. Here every buffer each entry point gets
-- inputs, outputs, workspace, status -- is carved out of a larger device
allocation whose 4 KB bands on both sides hold a known byte pattern; after
the call the bands must be unchanged ("inputs are never modified", Required
behavior, bullet 4, and no write outside the buffers the caller passed). Every
face and path is covered on small odd shapes: the out-of-place step (fused,
tensor with one and two row groups, the two-pass tensor form, generic, fp32), in place (decode
tensor-core, fused, tensor), paged (decode tensor-core, fused, tensor),
read-only re-attention, the gradients (each slot kernel) and the
no-allocation entry. The guarded run's results must equal an unguarded run's
(bit for bit; the gradients, whose query sums use atomics, within their
bound), so the guarded call did the real work.
"""
import ctypes

import pytest
import torch

import bounds
import kv_cache_append_gb300 as kvc
import workloads
from test_gpu_parity import DEV, SMALL, TC, _built  # noqa: F401
from workloads import Spec

pytestmark = pytest.mark.gpu

PAD = 4096
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` between two PAD-byte bands of PATTERN."""

    def __init__(self, shape, dtype, src=None):
        numel = 1
        for s in shape:
            numel *= int(s)
        es = torch.empty((), dtype=dtype).element_size()
        self.nbytes = numel * es
        self.raw = torch.full((self.nbytes + 2 * PAD,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.raw[PAD:PAD + self.nbytes].view(dtype).view(tuple(shape))
        if src is not None:
            self.t.copy_(src)

    def intact(self) -> bool:
        return bool((self.raw[:PAD] == PATTERN).all()) and \
            bool((self.raw[PAD + self.nbytes:] == PATTERN).all())


def guard(t):
    return Guarded(t.shape, t.dtype, t)


def _bits(t):
    if not t.is_floating_point():
        return t
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_intact(bufs):
    bad = [name for name, g in bufs.items() if not g.intact()]
    assert not bad, f"guard bands overwritten around: {bad}"


def guarded_inputs(x):
    names = ("query", "new_key", "new_value", "key_cache", "value_cache", "lengths")
    g = {n: guard(t) for n, t in zip(names, x.args()[:6])}
    g["append_mask"] = guard(x.append_mask.view(torch.uint8))
    return g


def scale_of(x):
    return float(x.options.get("scale", kvc.default_scale(x.query.shape[-1])))


STEP = {
    "fused_specdec_bf16": SMALL["specdec_bf16"].replace(Q=2, counts=("uniform", 0, 2)),
    "tensor_specdec_bf16_r16": SMALL["specdec_bf16"],
    "fused_fp32_Q40": SMALL["chunk_fp32_Q40"],
    "tensor_f16_D192": TC["r128_fp16_D192_Dv128"].replace(M=1001, lengths=("uniform", 500, 993)),
    # one row group, M a multiple of 8: the two-pass form, which writes the
    # attention rows from the step kernel
    "tensor2_f16_D192": TC["r128_fp16_D192_Dv128"].replace(M=1000, lengths=("uniform", 500, 992)),
    "tensor_bf16_rg2": TC["r160_bf16_chunk40"],
    "generic_D5_Dv7": Spec(B=3, Hq=4, Hk=2, Q=3, D=5, Dv=7, M=51, dtype="bf16",
                           counts=("uniform", 0, 3)),
    "q0": Spec(B=3, Hq=4, Hk=2, Q=0, D=64, Dv=64, M=100, dtype="bf16"),
}


@pytest.mark.parametrize("name", sorted(STEP))
def test_step_writes_stay_in_bounds(name):
    x = workloads.generate(STEP[name], 31).to(DEV)
    want = kvc.kv_cache_attention_step(*x.args(), x.options)
    gi = guarded_inputs(x)
    go = {k: guard(torch.zeros_like(v)) for k, v in want.items()}
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    ws = Guarded((kvc.workspace_bytes(dims),), torch.uint8)
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    kvc.step_into(dims, *(gi[n].t for n in ("query", "new_key", "new_value", "key_cache",
                                            "value_cache", "lengths", "append_mask")),
                  scale_of(x), {k: g.t for k, g in go.items()}, ws.t, st.t)
    torch.cuda.synchronize()
    assert_intact({**gi, **{"out_" + k: g for k, g in go.items()}, "workspace": ws, "status": st})
    for k in want:
        assert torch.equal(_bits(go[k].t), _bits(want[k])), k


INPLACE = {
    "decode_tc_bf16_hot": Spec(B=4, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=515, dtype="bf16",
                               lengths=("uniform", 100, 511), hot_frac=0.05, hot_scale=50.0),
    "fused_fp32": SMALL["chunk_fp32_Q40"],
    "tensor_f16_D192": STEP["tensor_f16_D192"],
    # 24 rows per KV head: the decode kernel's 32-row instance
    "decode_tc32_f16": Spec(B=3, Hq=8, Hk=1, Q=3, D=128, Dv=128, M=333, dtype="f16",
                            counts=("uniform", 0, 3)),
}


@pytest.mark.parametrize("name", sorted(INPLACE))
def test_inplace_writes_stay_in_bounds(name):
    x = workloads.generate(INPLACE[name], 32).to(DEV)
    kc, vc = x.key_cache.clone(), x.value_cache.clone()
    want = kvc.kv_cache_attention_step_inplace(x.query, x.new_key, x.new_value, kc, vc,
                                               x.lengths, x.append_mask, x.options)
    gi = guarded_inputs(x)
    go = {k: guard(torch.zeros_like(want[k])) for k in ("lengths", "attention", "context")}
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    ws = Guarded((kvc.workspace_bytes(dims),), torch.uint8)
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    kvc.step_inplace_into(dims, *(gi[n].t for n in ("query", "new_key", "new_value", "key_cache",
                                                    "value_cache", "lengths", "append_mask")),
                          scale_of(x), {k: g.t for k, g in go.items()}, ws.t, st.t)
    torch.cuda.synchronize()
    assert_intact({**gi, **{"out_" + k: g for k, g in go.items()}, "workspace": ws, "status": st})
    assert torch.equal(_bits(gi["key_cache"].t), _bits(kc))
    assert torch.equal(_bits(gi["value_cache"].t), _bits(vc))
    for k in go:
        assert torch.equal(_bits(go[k].t), _bits(want[k])), k


PAGED = {
    "decode_tc_bs16": (INPLACE["decode_tc_bf16_hot"].replace(M=512), 16),
    "decode_tc32_bs16": (INPLACE["decode_tc32_f16"].replace(M=336), 16),
    "fused_fp32_bs8": (SMALL["chunk_fp32_Q40"], 8),
    "tensor_f16_bs64": (STEP["tensor_f16_D192"].replace(M=1024), 64),
    "fused_bs40": (TC["r160_bf16_chunk40"], 40),
}


def _pool(c, table, nblocks, bs):
    B, Hk, M, W = c.shape
    mb = M // bs
    blocks = c.reshape(B, Hk, mb, bs, W).permute(0, 2, 1, 3, 4).reshape(B * mb, Hk, bs, W)
    pool = torch.zeros(nblocks, Hk, bs, W, dtype=c.dtype, device=c.device)
    pool[table.reshape(-1).long()] = blocks
    return pool


@pytest.mark.parametrize("name", sorted(PAGED))
def test_paged_writes_stay_in_bounds(name):
    spec, bs = PAGED[name]
    x = workloads.generate(spec, 33).to(DEV)
    B, M = spec.B, spec.M
    mb = M // bs
    nblocks = B * mb + 3
    table = torch.randperm(nblocks, generator=torch.Generator().manual_seed(4))[:B * mb]
    table = table.reshape(B, mb).to(torch.int32).to(DEV)
    kp, vp = _pool(x.key_cache, table, nblocks, bs), _pool(x.value_cache, table, nblocks, bs)
    kp2, vp2 = kp.clone(), vp.clone()
    want = kvc.kv_cache_attention_step_paged(x.query, x.new_key, x.new_value, kp2, vp2, table,
                                             x.lengths, x.append_mask, x.options)
    gi = guarded_inputs(x)
    gk, gv, gt = guard(kp), guard(vp), guard(table)
    go = {k: guard(torch.zeros_like(want[k])) for k in ("lengths", "attention", "context")}
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    ws = Guarded((kvc.paged_workspace_bytes(dims),), torch.uint8)
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    kvc.step_paged_into(dims, gt.t, gi["query"].t, gi["new_key"].t, gi["new_value"].t, gk.t,
                        gv.t, gi["lengths"].t, gi["append_mask"].t, scale_of(x),
                        {k: g.t for k, g in go.items()}, ws.t, st.t)
    torch.cuda.synchronize()
    assert_intact({**gi, "key_pool": gk, "value_pool": gv, "table": gt,
                   **{"out_" + k: g for k, g in go.items()}, "workspace": ws, "status": st})
    assert torch.equal(_bits(gk.t), _bits(kp2)) and torch.equal(_bits(gv.t), _bits(vp2))
    for k in go:
        assert torch.equal(_bits(go[k].t), _bits(want[k])), k


READONLY = {
    # (B, Hq, Hk, D, Dv, M, dtype, smax)
    "decode_tc": (6, 16, 4, 128, 128, 700, "bf16", 4),
    "decode_tc32": (4, 32, 4, 128, 128, 500, "bf16", 4),
    "fused_fp32": (5, 8, 2, 64, 64, 300, "f32", 5),
    "tensor": (3, 16, 1, 192, 128, 900, "f16", 8),
}


@pytest.mark.parametrize("name", sorted(READONLY))
def test_readonly_writes_stay_in_bounds(name):
    from test_gpu_attend_cache import make_case
    B, Hq, Hk, D, Dv, M, dt, smax = READONLY[name]
    q, kc, vc, cu, K, slot = make_case(B, Hq, Hk, D, Dv, M, dt, 6, smax)
    q, kc, vc, cu, K, slot = (t.to(DEV) for t in (q, kc, vc, cu, K, slot))
    want = kvc.attention_over_cache(q, kc, vc, cu, K, slot)
    gq, gk, gv, gcu, gK, gs = (guard(t) for t in (q, kc, vc, cu, K, slot))
    smax_seen = int((cu[1:] - cu[:-1]).max().item())
    dims = kvc.make_dims(B, Hq, Hk, max(1, smax_seen), D, Dv, M, q.dtype)
    go = guard(torch.zeros_like(want))
    ws = Guarded((kvc.attend_cache_workspace_bytes(dims),), torch.uint8)
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    kvc.attend_cache_into(dims, kc.shape[0], gq.t, gk.t, gv.t, gcu.t, gK.t, False, gs.t,
                          kvc.default_scale(D), go.t, ws.t, st.t)
    torch.cuda.synchronize()
    assert_intact({"q": gq, "key_cache": gk, "value_cache": gv, "cu_seqlens_q": gcu,
                   "seqlens_k": gK, "slot_ids": gs, "out": go, "workspace": ws, "status": st})
    assert torch.equal(_bits(go.t), _bits(want))


BACKWARD = {
    "rows_bf16": SMALL["decode_bf16_ragged_M"].replace(M=333),
    "tiled_fp32": SMALL["chunk_fp32_Q40"],
    "tc_f16_D192": SMALL["mqa_fp16_D192"].replace(M=700, lengths=("uniform", 100, 690)),
    "generic_bf16": STEP["generic_D5_Dv7"],
    # statistics on the decode kernel's 32-row instance, slots on the tensor-core kernel
    "dec32_tc_bf16": Spec(B=3, Hq=8, Hk=1, Q=3, D=128, Dv=128, M=300, dtype="bf16",
                          lengths=("uniform", 20, 290)),
}


@pytest.mark.parametrize("name", sorted(BACKWARD))
def test_backward_writes_stay_in_bounds(name):
    x = workloads.generate(BACKWARD[name], 34).to(DEV)
    g = torch.Generator(device=DEV).manual_seed(3)
    B, Hq, Q, _ = x.query.shape
    M, Dv = x.key_cache.shape[2], x.value_cache.shape[-1]
    grads = {"key_cache": torch.randn(x.key_cache.shape, generator=g, device=DEV),
             "value_cache": torch.randn(x.value_cache.shape, generator=g, device=DEV),
             "attention": torch.randn(B, Hq, Q, M, generator=g, device=DEV),
             "context": torch.randn(B, Hq, Q, Dv, generator=g, device=DEV)}
    grads = {k: v.to(x.query.dtype) for k, v in grads.items()}
    want = kvc.kv_cache_attention_step_backward(*x.args(), x.options,
                                                **{f"d_{k}": v for k, v in grads.items()})
    gi = guarded_inputs(x)
    gg = {k: guard(v) for k, v in grads.items()}
    go = {k: guard(torch.zeros_like(v)) for k, v in want.items()}
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    ws = Guarded((kvc.backward_workspace_bytes(dims),), torch.uint8)
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    kvc.step_backward_into(dims, *(gi[n].t for n in ("query", "new_key", "new_value",
                                                     "key_cache", "value_cache", "lengths",
                                                     "append_mask")),
                           scale_of(x), {k: v.t for k, v in gg.items()},
                           {k: v.t for k, v in go.items()}, ws.t, st.t)
    torch.cuda.synchronize()
    assert_intact({**gi, **{"grad_" + k: v for k, v in gg.items()},
                   **{"out_" + k: v for k, v in go.items()}, "workspace": ws, "status": st})
    # the query gradient's fp32 sums are added with atomics, so its last bit
    # may differ between runs: compared within the gradient bound
    for k in want:
        r = bounds.grad_ratio(go[k].t.double().cpu().numpy(), want[k].double().cpu().numpy(),
                              x.query.dtype)
        assert r <= 1.0, (k, r)


def test_static_entry_writes_stay_in_bounds():
    x = workloads.generate(STEP["tensor_f16_D192"], 35).to(DEV)
    want = kvc.kv_cache_attention_step(*x.args(), x.options)
    gi = guarded_inputs(x)
    go = {k: guard(torch.zeros_like(v)) for k, v in want.items()}
    st = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32, device=DEV))
    lib = kvc.library()
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    p = [ctypes.c_void_p(gi[n].t.data_ptr()) for n in ("query", "new_key", "new_value",
                                                        "key_cache", "value_cache", "lengths",
                                                        "append_mask")]
    rc = lib.kvc_step_static(ctypes.byref(dims), *p, ctypes.c_double(scale_of(x)),
                             *(ctypes.c_void_p(go[k].t.data_ptr()) for k in
                               ("key_cache", "value_cache", "lengths", "attention", "context")),
                             ctypes.c_void_p(st.t.data_ptr()),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, kvc.status_string(rc)
    torch.cuda.synchronize()
    assert_intact({**gi, **{"out_" + k: g for k, g in go.items()}, "status": st})
    for k in want:
        assert torch.equal(_bits(go[k].t), _bits(want[k])), k
