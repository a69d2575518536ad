"""GPU parity of the read-only re-attention (kvc_attend_cache) against the
fp64 oracle (oracle.attend_cache): packed queries attend the cache rows their
slots name, causally up to each sequence's total cached length; the cache is
never written. Output within the context tolerance of the step; sequences
outside the contract give zero rows and the overflow flag; and re-attending
a cache that the in-place step just appended reproduces that step's context
bit for bit (same kernels, same partials).
"""
import numpy as np
import pytest
import torch

import kv_cache_append_gb300 as kvc
import oracle
import workloads
from test_gpu_parity import DEV, TOL, _bits, _built  # noqa: F401
from workloads import Spec

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def make_case(B, Hq, Hk, D, Dv, M, dtype, seed, smax, num_slots=None, s_min=0, k_lo=None):
    """Random caches and packed queries: sequence b has S_b in [s_min, smax]
    queries and K_b in [max(S_b, k_lo), M] cached positions, in a permuted slot."""
    g = torch.Generator().manual_seed(seed)
    num_slots = num_slots or B + 3
    dt = DT[dtype]
    kc = torch.randn(num_slots, Hk, M, D, generator=g).to(dt)
    vc = torch.randn(num_slots, Hk, M, Dv, generator=g).to(dt)
    S = torch.randint(s_min, smax + 1, (B,), generator=g)
    lo = torch.maximum(S, torch.full((B,), k_lo if k_lo is not None else 0))
    K = lo + (torch.rand(B, generator=g) * (M - lo + 1).float()).long().clamp(max=M - lo)
    slot = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(S, 0)
    q = torch.randn(int(cu[-1]), Hq, D, generator=g).to(dt)
    return q, kc, vc, cu, K.to(torch.int32), slot


def check(q, kc, vc, cu, K, slot, k_cumulative=False, expect_flags=0, scale=None):
    kk = K
    if k_cumulative:
        kk = torch.zeros(K.numel() + 1, dtype=torch.int32)
        kk[1:] = torch.cumsum(K, 0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kcg, vcg = kc.to(DEV), vc.to(DEV)
    kb, vb = kcg.clone(), vcg.clone()
    out = kvc.attention_over_cache(q.to(DEV), kcg, vcg, cu.to(DEV), kk.to(DEV),
                                   None if slot is None else slot.to(DEV), scale=scale,
                                   status=status)
    torch.cuda.synchronize()
    want, flags = oracle.attend_cache(q, kc, vc, cu, K, slot, scale=scale)
    assert int(status.item()) == (int(np.bitwise_or.reduce(flags)) if len(flags) else 0)
    assert int(status.item()) == expect_flags
    np.testing.assert_allclose(out.double().cpu().numpy(), want, rtol=0, atol=TOL[q.dtype][1])
    assert torch.equal(_bits(kcg), _bits(kb)) and torch.equal(_bits(vcg), _bits(vb))  # read only
    return out


CASES = {
    # (B, Hq, Hk, D, Dv, M, dtype, smax): few rows per KV head (the decode
    # tensor-core kernel for 16-bit Dv = 128, the fused one otherwise)
    "decode_bf16": (12, 32, 8, 128, 128, 700, "bf16", 1),
    "specdec_bf16": (10, 32, 8, 128, 128, 900, "bf16", 4),
    "specdec32_bf16": (5, 32, 4, 128, 128, 800, "bf16", 4),  # up to 32 rows
    "fp32_gqa": (6, 8, 2, 64, 64, 300, "f32", 5),
    # tensor-core path (G * Qmax >= 64)
    "mqa_f16_D192": (4, 16, 1, 192, 128, 1500, "f16", 8),
    "chunked_bf16_r160": (3, 8, 2, 64, 64, 600, "bf16", 40),
    # generic path (rows that are not whole 16-byte words)
    "generic_D5": (5, 4, 2, 5, 7, 60, "bf16", 3),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_attend_cache_parity(name, seed):
    B, Hq, Hk, D, Dv, M, dtype, smax = CASES[name]
    check(*make_case(B, Hq, Hk, D, Dv, M, dtype, seed, smax))


def test_cumulative_seqlens_and_identity_slots():
    q, kc, vc, cu, K, _ = make_case(5, 8, 2, 64, 64, 200, "bf16", 3, 4, num_slots=5)
    check(q, kc, vc, cu, K, None, k_cumulative=True)


def test_empty_sequences_and_full_rows():
    g = torch.Generator().manual_seed(4)
    Hq, Hk, D, Dv, M = 16, 1, 128, 128, 512
    kc = torch.randn(7, Hk, M, D, generator=g).to(torch.float16)
    vc = torch.randn(7, Hk, M, Dv, generator=g).to(torch.float16)
    S = [8, 0, 5, 0, 1, 8]
    K = torch.tensor([512, 40, 5, 0, 1, 300], dtype=torch.int32)  # a full row, S == K rows
    cu = torch.tensor(np.concatenate([[0], np.cumsum(S)]), dtype=torch.int32)
    q = torch.randn(int(cu[-1]), Hq, D, generator=g).to(torch.float16)
    slot = torch.tensor([6, 0, 2, 5, 1, 3], dtype=torch.int32)
    check(q, kc, vc, cu, K, slot)


def test_sequences_outside_the_contract():
    q, kc, vc, cu, K, slot = make_case(5, 8, 2, 64, 64, 100, "bf16", 5, 3, s_min=1)
    K[1] = 0                   # S > K
    K[2] = 101                 # K > M
    slot[3] = 99               # slot out of range
    out = check(q, kc, vc, cu, K, slot, expect_flags=kvc.DEV_OVERFLOW)
    for b in (1, 2, 3):
        assert torch.count_nonzero(out[int(cu[b]):int(cu[b + 1])]) == 0


REATTEND = {
    "specdec": Spec(B=6, Hq=32, Hk=8, Q=4, D=128, Dv=128, M=640, dtype="bf16", counts=("all",)),
    "specdec24": Spec(B=4, Hq=8, Hk=1, Q=3, D=128, Dv=128, M=500, dtype="bf16", counts=("all",)),
    "mqa": Spec(B=3, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=1000, dtype="f16", counts=("all",),
                lengths=("uniform", 300, 990)),
}


@pytest.mark.parametrize("spec_name", sorted(REATTEND))
def test_reattending_the_appended_cache_reproduces_the_step(spec_name):
    spec = REATTEND[spec_name]
    x = workloads.generate(spec, 4).to(DEV)
    kc, vc = x.key_cache.clone(), x.value_cache.clone()
    ref = kvc.kv_cache_attention_step_inplace(x.query, x.new_key, x.new_value, kc, vc,
                                              x.lengths, x.append_mask, x.options)
    B, Hq, Q = spec.B, spec.Hq, spec.Q
    q = x.query.permute(0, 2, 1, 3).reshape(B * Q, Hq, spec.D).contiguous()
    cu = torch.arange(0, B * Q + 1, Q, dtype=torch.int32, device=DEV)
    out = kvc.attention_over_cache(q, kc, vc, cu, ref["lengths"], max_seqlen_q=Q,
                                   scale=x.options.get("scale"))
    want = ref["context"].permute(0, 2, 1, 3).reshape(B * Q, Hq, spec.Dv)
    assert torch.equal(_bits(out), _bits(want))


def test_decode_scale_against_the_oracle():
    """Decode-sized: 64 sequences of up to 8192 cached positions, one query each."""
    q, kc, vc, cu, K, slot = make_case(64, 32, 8, 128, 128, 8192, "bf16", 9, 1, s_min=1,
                                       k_lo=1024, num_slots=64)
    check(q, kc, vc, cu, K, slot)


@pytest.mark.parametrize("name", ["specdec_bf16", "mqa_f16_D192"])
def test_poisoned_slots_past_the_cached_length(name):
    B, Hq, Hk, D, Dv, M, dtype, smax = CASES[name]
    q, kc, vc, cu, K, slot = make_case(B, Hq, Hk, D, Dv, M, dtype, 13, smax, s_min=1)
    for b in range(B):
        kc[int(slot[b]), :, int(K[b]):] = float("inf")
        vc[int(slot[b]), :, int(K[b]):] = float("nan")
    check(q, kc, vc, cu, K, slot)
