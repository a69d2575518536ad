"""GPU parity of the in-place step (kvc_step_inplace) against the fp64 oracle.

The caches are donated and updated in place: afterwards they must equal the
oracle's updated caches bit for bit, the lengths must be exact, attention and
context must meet the same tolerances as the out-of-place step, and caches and
lengths must equal the out-of-place step's bit for bit. Attention and context
are compared with the out-of-place step within the step's tolerance only: the
in-place step may cut the cache into larger tiles (it copies nothing), so its
partial sums can round differently. Inputs other than the caches stay
untouched.
"""
import numpy as np
import pytest
import torch

import kv_cache_append_gb300 as kvc
import workloads
from test_gpu_parity import (DEV, SMALL, TC, TOL, _bits, _built, check_append_property,  # noqa: F401
                             compare_batch_rows, compare_full, run_gpu)
from workloads import Spec

pytestmark = pytest.mark.gpu


def run_inplace(x: workloads.StepInputs):
    """kvc_step_inplace on clones of x's caches; returns (outputs, status)."""
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kc, vc = x.key_cache.clone(), x.value_cache.clone()
    out = kvc.kv_cache_attention_step_inplace(x.query, x.new_key, x.new_value, kc, vc,
                                              x.lengths, x.append_mask, x.options,
                                              status=status)
    torch.cuda.synchronize()
    assert out["key_cache"] is kc and out["value_cache"] is vc
    return out, int(status.item())


def same_as_out_of_place(xg, out):
    ref, _ = run_gpu(xg)
    for k in ("key_cache", "value_cache"):
        assert torch.equal(_bits(out[k]), _bits(ref[k])), k
    assert torch.equal(out["lengths"], ref["lengths"])
    atol_a, atol_c = TOL[xg.query.dtype]
    for k, atol in (("attention", atol_a), ("context", atol_c)):
        np.testing.assert_allclose(out[k].double().cpu().numpy(), ref[k].double().cpu().numpy(),
                                   rtol=0, atol=atol, err_msg=k)


CASES = {
    "tiny_fp32": SMALL["tiny_fp32"],
    "decode_bf16_ragged_M": SMALL["decode_bf16_ragged_M"],
    "specdec_bf16": SMALL["specdec_bf16"],
    "chunk_fp32_Q40": SMALL["chunk_fp32_Q40"],
    "fp32_three_segments": SMALL["fp32_three_segments"],
    "gqa_fp32_small_rows": SMALL["gqa_fp32_small_rows"],        # generic path (16-byte rows)
    "tc_r128_fp16_D192": TC["r128_fp16_D192_Dv128"],
    "tc_r64_bf16_ragged": TC["r64_bf16_ragged"],
    "tc_r160_bf16_chunk40": TC["r160_bf16_chunk40"],
    "generic_D5_Dv7": Spec(B=3, Hq=4, Hk=2, Q=3, D=5, Dv=7, M=50, dtype="bf16",
                           counts=("uniform", 0, 3)),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 3])
def test_inplace_parity(name, seed):
    x = workloads.generate(CASES[name], seed)
    xg = x.to(DEV)
    before = [t.clone() for t in (xg.query, xg.new_key, xg.new_value, xg.lengths,
                                  xg.append_mask)]
    out, status = run_inplace(xg)
    compare_full(x, out, status)
    same_as_out_of_place(xg, out)
    for a, b in zip(before, (xg.query, xg.new_key, xg.new_value, xg.lengths, xg.append_mask)):
        assert torch.equal(_bits(a) if a.is_floating_point() else a,
                           _bits(b) if b.is_floating_point() else b)


def test_inplace_q_zero_copies_lengths_only():
    spec = Spec(B=3, Hq=4, Hk=2, Q=0, D=64, Dv=64, M=100, dtype="bf16")
    x = workloads.generate(spec, 0)
    out, status = run_inplace(x.to(DEV))
    compare_full(x, out, status)


def test_inplace_nothing_appended_writes_nothing():
    spec = Spec(B=4, Hq=8, Hk=2, Q=3, D=128, Dv=128, M=300, dtype="bf16", counts=("fixed", 0))
    x = workloads.generate(spec, 1)
    xg = x.to(DEV)
    out, status = run_inplace(xg)
    compare_full(x, out, status)
    assert torch.equal(_bits(out["key_cache"]), _bits(xg.key_cache))
    assert torch.count_nonzero(out["attention"]) == 0


@pytest.mark.parametrize("tensor", [False, True])
def test_inplace_contract_violations(tensor):
    """Rows outside the contract append nothing, so their cache rows stay."""
    if tensor:
        spec = Spec(B=4, Hq=16, Hk=2, Q=8, D=64, Dv=64, M=256, dtype="f16")
        lengths, counts, bad_t = [10, 250, 300, 100], [8, 8, 3, 8], 6
    else:
        spec = Spec(B=5, Hq=4, Hk=2, Q=3, D=64, Dv=64, M=200, dtype="bf16")
        lengths, counts, bad_t = [10, 199, 250, -3, 40], [3, 3, 1, 1, 3], 1
    x = workloads.generate(spec, 11)
    x.lengths = torch.tensor(lengths)
    m = workloads.prefix_mask(counts, spec.Q)
    m[-1, bad_t] = False  # not a prefix
    x.append_mask = m
    out, status = run_inplace(x.to(DEV))
    compare_full(x, out, status, expect_flags=kvc.DEV_MASK | kvc.DEV_OVERFLOW)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_inplace_chunked_chain_40_32_24(dtype):
    """Three chained appends into one donated cache."""
    spec = workloads.SPECS["chunked_append"].replace(dtype=dtype)
    first, rest = workloads.chain_chunks(spec, seed=2)
    xc = first
    kc, vc = first.key_cache.to(DEV), first.value_cache.to(DEV)
    lengths = first.lengths.to(DEV)
    q, nk, nv, mask = first.query, first.new_key, first.new_value, first.append_mask
    for i in range(len(workloads.CHUNKS)):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = kvc.kv_cache_attention_step_inplace(q.to(DEV), nk.to(DEV), nv.to(DEV), kc, vc,
                                                  lengths, mask.to(DEV), {}, status=status)
        torch.cuda.synchronize()
        ref = compare_full(xc, out, int(status.item()))
        if i == len(rest):
            break
        q, nk, nv, mask = rest[i]
        lengths = out["lengths"]
        xc = workloads.StepInputs(q, nk, nv, ref["key_cache"], ref["value_cache"],
                                  ref["lengths"], mask, {})


def test_inplace_rejects_overlap_with_caches():
    spec = Spec(B=2, Hq=4, Hk=2, Q=2, D=64, Dv=64, M=40, dtype="bf16")
    x = workloads.generate(spec, 6).to(DEV)
    q, nk, nv, kc, vc, ln, mk = x.args()
    dims = kvc.dims_of(q, kc, vc)
    out = kvc.allocate_outputs(q, kc, vc)
    ws = torch.empty(kvc.workspace_bytes(dims), dtype=torch.uint8, device=DEV)
    alias = kc.view(-1)[:q.numel()].view(q.shape)   # the query inside the key cache
    with pytest.raises(kvc.KvcError) as err:
        kvc.step_inplace_into(dims, alias, nk, nv, kc, vc, ln, mk.view(torch.uint8), 0.125,
                              out, ws)
    assert err.value.status == -6  # KVC_E_ALIAS


@pytest.mark.parametrize("name", ["gqa_decode", "long_mqa"])
def test_inplace_full_size(name):
    spec = workloads.SPECS[name]
    x = workloads.generate(spec, seed=1, device=DEV)
    out, status = run_inplace(x)
    assert status == 0
    check_append_property(x, out)
    lengths = x.lengths.cpu().numpy()
    rng = np.random.default_rng(7)
    bsel = {int(lengths.argmax()), int(lengths.argmin())}
    if name != "long_mqa":
        bsel |= set(rng.choice(spec.B, size=3, replace=False).tolist())
    compare_batch_rows(x, out, bsel)
    del out, x
    torch.cuda.empty_cache()
