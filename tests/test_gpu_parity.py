"""GPU parity: libkvc (through its C ABI) against the fp64 oracle on the same
seeded inputs.

Bars: caches and lengths bit-exact; fp32 attention within 1e-5 and context
within 1e-4 (absolute); bf16/fp16 attention within 4e-3 and context within
2e-2 (absolute), the oracle's exact double result being the reference.
Every comparison also applies the per-row error bounds of tests/bounds.py
(derived from the kernels' arithmetic, relative to each row's own magnitude),
which can fail on long rows where the absolute bars cannot, and asserts that
wrong variants of the oracle's own output (scaled by 0.9, all zero) exceed
them. Small cases compare every element; the full-size workloads, run in the
same launch configuration as bench.py, compare every cache element through the
append property and sampled batch rows against the oracle.
"""
import hashlib
import os

import numpy as np
import pytest
import torch

import bounds
import kv_cache_append_gb300 as kvc
import oracle
import workloads
from workloads import Spec

pytestmark = pytest.mark.gpu

TOL = {torch.float32: (1e-5, 1e-4), torch.bfloat16: (4e-3, 2e-2), torch.float16: (4e-3, 2e-2)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_append_gb300 import build as kbuild
    kbuild.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


DEV = torch.device("cuda:0")


def run_gpu(x: workloads.StepInputs):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = kvc.kv_cache_attention_step(*x.args(), x.options, status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def compare_full(xc: workloads.StepInputs, out, status, expect_flags=0):
    """Every element against the oracle (inputs on the CPU)."""
    ref = oracle.step(*xc.args(), xc.options)
    assert torch.equal(_bits(out["key_cache"].cpu()), _bits(ref["key_cache"]))
    assert torch.equal(_bits(out["value_cache"].cpu()), _bits(ref["value_cache"]))
    assert torch.equal(out["lengths"].cpu(), ref["lengths"])
    flags = int(np.bitwise_or.reduce(ref["flags"])) if len(ref["flags"]) else 0
    assert status == flags == expect_flags
    atol_a, atol_c = TOL[xc.query.dtype]
    att = out["attention"].double().cpu().numpy()
    ctx = out["context"].double().cpu().numpy()
    np.testing.assert_allclose(att, ref["attention"], rtol=0, atol=atol_a)
    np.testing.assert_allclose(ctx, ref["context"], rtol=0, atol=atol_c)
    # masked / invalid entries are exactly +0
    zero = ref["attention"] == 0.0
    assert np.all(att[zero] == 0.0) and not np.any(np.signbit(att[zero]))
    # per-row bounds relative to each row's magnitude
    bounds.check_step(xc, ref["key_cache"], ref["value_cache"], att, ctx, ref["attention"],
                      ref["context"], scale_of(xc))
    return ref


def scale_of(x):
    return float(x.options.get("scale", kvc.default_scale(x.query.shape[-1])))


def check_append_property(x, out):
    """Full-size bit-exactness: the output cache equals the input cache except
    rows [length, length + n), which equal the first n new rows."""
    counts = x.append_mask.to(torch.int64).sum(1).cpu()
    lengths = x.lengths.cpu()
    for name, cache, new in (("key_cache", x.key_cache, x.new_key),
                             ("value_cache", x.value_cache, x.new_value)):
        got = _bits(out[name])
        want = _bits(cache).clone()
        nb = _bits(new)
        for b in range(cache.shape[0]):
            L, n = int(lengths[b]), int(counts[b])
            if n:
                want[b, :, L:L + n] = nb[b, :, :n]
        assert torch.equal(got, want), name
    assert torch.equal(out["lengths"].cpu(), lengths + counts)


def compare_batch_rows(x, out, bsel):
    """Attention/context of every (h, t) of the selected batch rows against the
    oracle, on the sub-batch those rows form (the rows of a batch are
    independent by definition)."""
    bsel = sorted(set(int(b) for b in bsel))
    idx = torch.tensor(bsel, device=x.query.device)
    sub = [t.index_select(0, idx).cpu() for t in x.args()]
    B, Hq, Q, _ = sub[0].shape
    rows = [(b, h, t) for b in range(B) for h in range(Hq) for t in range(Q)]
    att_ref, ctx_ref = oracle.rows(*sub, rows, x.options)
    att = out["attention"].index_select(0, idx).double().cpu().numpy().reshape(len(rows), -1)
    ctx = out["context"].index_select(0, idx).double().cpu().numpy().reshape(len(rows), -1)
    atol_a, atol_c = TOL[x.query.dtype]
    np.testing.assert_allclose(att, att_ref, rtol=0, atol=atol_a)
    np.testing.assert_allclose(ctx, ctx_ref, rtol=0, atol=atol_c)
    assert np.all(att[att_ref == 0.0] == 0.0)
    # per-row bounds on the updated caches the step returned (already checked
    # bit for bit against the append property)
    xs = workloads.StepInputs(*sub, x.options)
    upd_k = out["key_cache"].index_select(0, idx).cpu()
    upd_v = out["value_cache"].index_select(0, idx).cpu()
    M, Dv = att.shape[-1], ctx.shape[-1]
    return bounds.check_step(xs, upd_k, upd_v, att.reshape(B, Hq, Q, M),
                             ctx.reshape(B, Hq, Q, Dv), att_ref.reshape(B, Hq, Q, M),
                             ctx_ref.reshape(B, Hq, Q, Dv), scale_of(x), "sampled")


# ------------------------------------------------------------------ small cases
SMALL = {
    "tiny_fp32": workloads.SPECS["tiny_fp32"],
    "decode_bf16_ragged_M": Spec(B=4, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=1000, dtype="bf16",
                                 lengths=("uniform", 0, 999)),
    "specdec_bf16": Spec(B=8, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=777, dtype="bf16",
                         lengths=("zipf", 1.2), counts=("uniform", 0, 4), hot_frac=0.05,
                         hot_scale=50.0),
    "mqa_fp16_D192": Spec(B=2, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=3000, dtype="f16",
                          lengths=("uniform", 2000, 2992), std=0.5, scale=0.05),
    "chunk_fp32_Q40": Spec(B=2, Hq=8, Hk=2, Q=40, D=64, Dv=64, M=600, dtype="f32",
                           lengths=("uniform", 100, 500)),
    "mha_fp16_Dv256": Spec(B=2, Hq=2, Hk=2, Q=3, D=64, Dv=256, M=200, dtype="f16",
                           counts=("uniform", 0, 3)),
    "gqa_fp32_small_rows": Spec(B=3, Hq=6, Hk=3, Q=2, D=4, Dv=8, M=70, dtype="f32",
                                counts=("uniform", 0, 2)),
    "bf16_D8_M1": Spec(B=3, Hq=2, Hk=1, Q=1, D=8, Dv=8, M=1, dtype="bf16",
                       lengths=("fixed", 0)),
    # rows longer than one finalize segment (8192 slots), M not a multiple of 8
    "fp32_three_segments": Spec(B=1, Hq=2, Hk=1, Q=2, D=16, Dv=16, M=2 * 8192 + 13,
                                dtype="f32", lengths=("uniform", 9000, 16395)),
    # more than 32 rows per unit on small caches: row blocks of 32 rows, the
    # last one partial (42 = 32 + 10 rows; 48 = 32 + 16 rows, 16-bit D = 96)
    "rowblocks_fp32_R42": Spec(B=3, Hq=6, Hk=1, Q=7, D=64, Dv=64, M=300, dtype="f32",
                               counts=("uniform", 0, 7)),
    "rowblocks_bf16_D96_R48": Spec(B=2, Hq=12, Hk=2, Q=8, D=96, Dv=64, M=257, dtype="bf16",
                                   lengths=("uniform", 0, 249), counts=("uniform", 1, 8)),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("seed", [0, 1])
def test_small_full_parity(name, seed):
    x = workloads.generate(SMALL[name], seed)
    out, status = run_gpu(x.to(DEV))
    compare_full(x, out, status)


@pytest.mark.parametrize("seed", range(5))
def test_tiny_oracle_case_all_seeds(seed):
    x = workloads.generate(workloads.SPECS["tiny_fp32"], seed)
    out, status = run_gpu(x.to(DEV))
    compare_full(x, out, status)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunked_chain_40_32_24(dtype):
    """Three chained appends, each consuming the previous step's outputs."""
    spec = workloads.SPECS["chunked_append"].replace(dtype=dtype)
    first, rest = workloads.chain_chunks(spec, seed=2)
    xc = first
    xg = first.to(DEV)
    for i in range(len(workloads.CHUNKS)):
        out, status = run_gpu(xg)
        ref = compare_full(xc, out, status)
        if i == len(rest):
            break
        q, nk, nv, mask = rest[i]
        xc = workloads.StepInputs(q, nk, nv, ref["key_cache"], ref["value_cache"],
                                  ref["lengths"], mask, {})
        xg = workloads.StepInputs(q.to(DEV), nk.to(DEV), nv.to(DEV), out["key_cache"],
                                  out["value_cache"], out["lengths"], mask.to(DEV), {})


# ------------------------------------------------------------------ edge cases
def test_q_zero():
    spec = Spec(B=3, Hq=4, Hk=2, Q=0, D=64, Dv=64, M=100, dtype="bf16")
    x = workloads.generate(spec, 0)
    out, status = run_gpu(x.to(DEV))
    assert out["attention"].shape == (3, 4, 0, 100) and out["context"].shape == (3, 4, 0, 64)
    compare_full(x, out, status)


def test_all_rows_append_nothing():
    spec = Spec(B=4, Hq=8, Hk=2, Q=3, D=128, Dv=128, M=300, dtype="bf16", counts=("fixed", 0))
    x = workloads.generate(spec, 1)
    out, status = run_gpu(x.to(DEV))
    compare_full(x, out, status)
    assert torch.count_nonzero(out["attention"]) == 0


def test_first_token_and_full_cache():
    spec = Spec(B=4, Hq=4, Hk=1, Q=2, D=64, Dv=64, M=130, dtype="f32")
    x = workloads.generate(spec, 3)
    x.lengths = torch.tensor([0, 128, 64, 127])
    x.append_mask = workloads.prefix_mask([1, 2, 2, 1], 2)
    out, status = run_gpu(x.to(DEV))
    compare_full(x, out, status)


def test_contract_violations_are_flagged_and_append_nothing():
    spec = Spec(B=5, Hq=4, Hk=2, Q=3, D=64, Dv=64, M=96, dtype="bf16")
    x = workloads.generate(spec, 4)
    x.lengths = torch.tensor([10, 95, 200, -3, 40])
    x.append_mask = torch.tensor([[1, 0, 1], [1, 1, 0], [1, 0, 0], [1, 0, 0], [1, 1, 1]],
                                 dtype=torch.bool)
    out, status = run_gpu(x.to(DEV))
    compare_full(x, out, status, expect_flags=kvc.DEV_MASK | kvc.DEV_OVERFLOW)


@pytest.mark.parametrize("D,Dv,dtype", [(3, 5, "f32"), (5, 7, "bf16"), (64, 264, "bf16")])
def test_generic_path_shapes(D, Dv, dtype):
    spec = Spec(B=3, Hq=4, Hk=2, Q=3, D=D, Dv=Dv, M=50, dtype=dtype, counts=("uniform", 0, 3))
    x = workloads.generate(spec, 5)
    xg = x.to(DEV)
    n, path = kvc.plan_info(kvc.dims_of(xg.query, xg.key_cache, xg.value_cache), xg.key_cache,
                            xg.value_cache, xg.new_key, xg.new_value, xg.key_cache,
                            xg.value_cache)
    assert path == "generic" and n == 4  # copy, attend, merge, row writer
    out, status = run_gpu(xg)
    compare_full(x, out, status)


def test_unaligned_pointers_take_generic_path():
    spec = Spec(B=2, Hq=4, Hk=2, Q=2, D=64, Dv=64, M=40, dtype="bf16")
    x = workloads.generate(spec, 6)
    xg = x.to(DEV)
    kc = torch.empty(xg.key_cache.numel() + 1, dtype=torch.bfloat16, device=DEV)
    kc[1:] = xg.key_cache.reshape(-1)
    xg.key_cache = kc[1:].view(x.key_cache.shape)
    out, status = run_gpu(xg)
    compare_full(x, out, status)


def test_inputs_unchanged_and_repeatable():
    x = workloads.generate(SMALL["specdec_bf16"], 7).to(DEV)
    digest = [hashlib.sha256(t.cpu().numpy().tobytes() if t.dtype != torch.bfloat16 else
                             t.view(torch.int16).cpu().numpy().tobytes()).hexdigest()
              for t in x.args()]
    a, _ = run_gpu(x)
    b, _ = run_gpu(x)
    after = [hashlib.sha256(t.cpu().numpy().tobytes() if t.dtype != torch.bfloat16 else
                            t.view(torch.int16).cpu().numpy().tobytes()).hexdigest()
             for t in x.args()]
    assert digest == after
    for k in a:
        assert torch.equal(_bits(a[k]) if a[k].is_floating_point() else a[k],
                           _bits(b[k]) if b[k].is_floating_point() else b[k]), k


def test_large_scores_stay_finite():
    spec = Spec(B=2, Hq=4, Hk=2, Q=2, D=128, Dv=128, M=256, dtype="bf16")
    x = workloads.generate(spec, 8)
    x.query = (x.query.float() * 60.0).to(torch.bfloat16)   # raw dots well above 1000
    out, status = run_gpu(x.to(DEV))
    assert torch.isfinite(out["attention"]).all() and torch.isfinite(out["context"]).all()
    compare_full(x, out, status)


# ------------------------------------------------------------------ full-size workloads
FULL = ["gqa_decode", "ragged_specdec", "long_mqa"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    spec = workloads.SPECS[name]
    x = workloads.generate(spec, seed=1, device=DEV)
    out, status = run_gpu(x)
    assert status == 0
    check_append_property(x, out)
    # sampled batch rows: the longest and shortest rows, one with the most
    # appended rows, plus seeded random rows
    lengths = x.lengths.cpu().numpy()
    counts = x.append_mask.sum(1).cpu().numpy()
    rng = np.random.default_rng(99)
    bsel = {int(lengths.argmax()), int(lengths.argmin()), int(counts.argmax())}
    bsel |= set(rng.choice(spec.B, size=min(3, spec.B), replace=False).tolist())
    if name == "long_mqa":
        bsel = set(sorted(bsel)[:4])
    compare_batch_rows(x, out, bsel)
    del out, x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["gqa_decode", "ragged_specdec"])
def test_full_size_workload_fp32(name):
    """The decode shapes at full size in fp32 (the CUDA-core kernel), checked at
    the fp32 bars (1e-5 / 1e-4) and the per-row bounds on sampled batch rows."""
    spec = workloads.SPECS[name].replace(dtype="f32")
    x = workloads.generate(spec, seed=3, device=DEV)
    out, status = run_gpu(x)
    assert status == 0
    check_append_property(x, out)
    lengths = x.lengths.cpu().numpy()
    counts = x.append_mask.sum(1).cpu().numpy()
    rng = np.random.default_rng(7)
    bsel = {int(lengths.argmax()), int(lengths.argmin()), int(counts.argmax())}
    bsel |= set(rng.choice(spec.B, size=3, replace=False).tolist())
    compare_batch_rows(x, out, bsel)
    del out, x
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ tensor-core path
TC = {
    "r128_fp16_D192_Dv128": Spec(B=2, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=3000, dtype="f16",
                                 lengths=("uniform", 2000, 2992), std=0.5, scale=0.05),
    "r64_bf16_ragged": Spec(B=3, Hq=16, Hk=2, Q=8, D=128, Dv=128, M=700, dtype="bf16",
                            lengths=("uniform", 0, 692), counts=("uniform", 0, 8)),
    "r64_bf16_D64_Dv256": Spec(B=2, Hq=8, Hk=1, Q=8, D=64, Dv=256, M=333, dtype="bf16",
                               lengths=("uniform", 100, 325)),
    "r64_fp16_D256_Dv64": Spec(B=2, Hq=4, Hk=1, Q=16, D=256, Dv=64, M=512, dtype="f16",
                               lengths=("uniform", 0, 496), counts=("uniform", 1, 16)),
    "r96_bf16_hot": Spec(B=2, Hq=12, Hk=1, Q=8, D=128, Dv=128, M=1024, dtype="bf16",
                         hot_frac=0.2, hot_scale=50.0),
    # several finalize segments per row; padded fp16 P rows (M % 8 != 0)
    "r64_fp16_segments": Spec(B=1, Hq=8, Hk=1, Q=8, D=64, Dv=64, M=20000, dtype="f16",
                              lengths=("uniform", 17000, 19990)),
    "r64_bf16_segments_M9005": Spec(B=1, Hq=8, Hk=1, Q=8, D=64, Dv=64, M=9005, dtype="bf16",
                                    lengths=("uniform", 8000, 8995)),
    # more than 128 query rows per unit: two row groups
    "r160_bf16_chunk40": Spec(B=2, Hq=8, Hk=2, Q=40, D=64, Dv=64, M=600, dtype="bf16",
                              lengths=("uniform", 100, 500)),
    "r200_fp16_ragged": Spec(B=3, Hq=8, Hk=1, Q=25, D=128, Dv=128, M=777, dtype="f16",
                             lengths=("uniform", 0, 752), counts=("uniform", 0, 25)),
    "r256_bf16_D192": Spec(B=1, Hq=16, Hk=1, Q=16, D=192, Dv=128, M=1000, dtype="bf16",
                           lengths=("uniform", 500, 984), counts=("uniform", 1, 16)),
    # 9 to 63 rows per unit (the rest of the 128 tensor-memory lanes are padding):
    # the least, a decode-like GQA spec step, D = 256 with Dv = 64, a ragged 48
    "r9_f16_min": Spec(B=3, Hq=9, Hk=1, Q=1, D=128, Dv=128, M=500, dtype="f16",
                       lengths=("uniform", 0, 498)),
    "r16_bf16_specdec": Spec(B=4, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=700, dtype="bf16",
                             lengths=("uniform", 10, 690), counts=("uniform", 0, 4),
                             hot_frac=0.05, hot_scale=50.0),
    "r12_bf16_D256_Dv64": Spec(B=2, Hq=12, Hk=4, Q=4, D=256, Dv=64, M=400, dtype="bf16",
                               lengths=("uniform", 100, 390)),
    "r48_fp16_ragged": Spec(B=3, Hq=16, Hk=1, Q=3, D=64, Dv=64, M=650, dtype="f16",
                            lengths=("uniform", 0, 640), counts=("uniform", 0, 3)),
    # rows of 320 elements and more at any row count (decode shapes of wide heads)
    "r4_bf16_D256_Dv128": Spec(B=3, Hq=8, Hk=2, Q=1, D=256, Dv=128, M=450, dtype="bf16",
                               lengths=("uniform", 0, 449)),
    "r1_f16_D192_Dv128": Spec(B=4, Hq=2, Hk=2, Q=1, D=192, Dv=128, M=300, dtype="f16",
                              lengths=("uniform", 50, 299)),
    "r6_bf16_D64_Dv256_ragged": Spec(B=3, Hq=2, Hk=1, Q=3, D=64, Dv=256, M=200, dtype="bf16",
                                     lengths=("uniform", 0, 197), counts=("uniform", 0, 3)),
}


# the tensor-core step: one pass with stored P rows and the row writer, or
# (one row group, out of place, M a multiple of 8) two passes writing the
# attention rows directly
TENSOR_PATHS = ("tensor", "tensor_2pass")


def _path(x):
    """The path kvc_step takes for x (out of place: output caches of their own)."""
    ok, ov = torch.empty_like(x.key_cache), torch.empty_like(x.value_cache)
    return kvc.plan_info(kvc.dims_of(x.query, x.key_cache, x.value_cache), x.key_cache,
                         x.value_cache, x.new_key, x.new_value, ok, ov)[1]


@pytest.mark.skipif(os.environ.get("KVC_EXPECT_TWO_PASS") != "1",
                    reason="the two-pass form is built only with KVC_TC_TWO_PASS=1")
def test_two_pass_taken_where_it_applies():
    """The two-pass form for one row group with M a multiple of 8 (out of
    place), the one-pass form otherwise (two row groups, M = 700 or 9005, in
    place)."""
    want = {"r128_fp16_D192_Dv128": "tensor_2pass", "r64_fp16_D256_Dv64": "tensor_2pass",
            "r96_bf16_hot": "tensor_2pass", "r64_fp16_segments": "tensor_2pass",
            "r64_bf16_ragged": "tensor", "r64_bf16_segments_M9005": "tensor",
            "r160_bf16_chunk40": "tensor", "r200_fp16_ragged": "tensor"}
    for name, path in want.items():
        xg = workloads.generate(TC[name], 0).to(DEV)
        assert _path(xg) == path, name
        dims = kvc.dims_of(xg.query, xg.key_cache, xg.value_cache)
        assert kvc.plan_info_inplace(dims, xg.key_cache, xg.value_cache, xg.new_key,
                                     xg.new_value)[1] == "tensor"


@pytest.mark.parametrize("name", sorted(TC))
@pytest.mark.parametrize("seed", [0, 1])
def test_tensor_core_path(name, seed):
    x = workloads.generate(TC[name], seed)
    xg = x.to(DEV)
    assert _path(xg) in TENSOR_PATHS
    out, status = run_gpu(xg)
    compare_full(x, out, status)


def test_tensor_core_path_growing_scores():
    """Scores that grow along the slots raise the reference maximum on many
    tiles, so the context accumulator is rescaled again and again."""
    spec = Spec(B=2, Hq=16, Hk=2, Q=8, D=128, Dv=128, M=640, dtype="bf16",
                lengths=("fixed", 600))
    x = workloads.generate(spec, 9)
    ramp = (1.0 + torch.arange(spec.M, dtype=torch.float32) / 24.0)[None, None, :, None]
    x.key_cache = (x.key_cache.float() * ramp).to(torch.bfloat16)
    x.query = (x.query.float() * 4.0).to(torch.bfloat16)
    xg = x.to(DEV)
    assert _path(xg) in TENSOR_PATHS
    out, status = run_gpu(xg)
    compare_full(x, out, status)


def test_tensor_core_path_contract_violations():
    spec = Spec(B=4, Hq=16, Hk=2, Q=8, D=64, Dv=64, M=256, dtype="f16")
    x = workloads.generate(spec, 11)
    x.lengths = torch.tensor([10, 250, 300, 100])
    m = workloads.prefix_mask([8, 8, 3, 8], 8)
    m[3, 6] = False
    m[3, 7] = True   # not a prefix
    x.append_mask = m
    xg = x.to(DEV)
    assert _path(xg) in TENSOR_PATHS
    out, status = run_gpu(xg)
    compare_full(x, out, status, expect_flags=kvc.DEV_MASK | kvc.DEV_OVERFLOW)


# ------------------------------------------------------------------ poisoned tails
def _poison_tails(x):
    """Slots from each row's new length on hold +Inf keys and NaN values: the
    step must neither read them into any result nor change them."""
    counts = x.append_mask.to(torch.int64).sum(1)
    for b in range(x.key_cache.shape[0]):
        N = int(x.lengths[b]) + int(counts[b])
        x.key_cache[b, :, N:] = float("inf")
        x.value_cache[b, :, N:] = float("nan")
    return x


POISON = {
    "fused_bf16": Spec(B=4, Hq=8, Hk=2, Q=3, D=128, Dv=128, M=500, dtype="bf16",
                       lengths=("uniform", 10, 400), counts=("uniform", 1, 3)),
    "tensor_f16": Spec(B=3, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=700, dtype="f16",
                       lengths=("uniform", 10, 600), counts=("uniform", 1, 8)),
    "tensor_bf16_rg2": Spec(B=2, Hq=8, Hk=2, Q=40, D=64, Dv=64, M=600, dtype="bf16",
                            lengths=("uniform", 100, 500)),
}


@pytest.mark.parametrize("name", sorted(POISON))
@pytest.mark.parametrize("inplace", [False, True])
def test_poisoned_tail_slots(name, inplace):
    x = _poison_tails(workloads.generate(POISON[name], 12))
    xg = x.to(DEV)
    if inplace:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        kc, vc = xg.key_cache.clone(), xg.value_cache.clone()
        out = kvc.kv_cache_attention_step_inplace(xg.query, xg.new_key, xg.new_value, kc, vc,
                                                  xg.lengths, xg.append_mask, xg.options,
                                                  status=status)
        torch.cuda.synchronize()
        status = int(status.item())
    else:
        out, status = run_gpu(xg)
    compare_full(x, out, status)
