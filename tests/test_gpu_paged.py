"""GPU parity of the paged step (kvc_step_paged) against the fp64 oracle
(oracle.step_paged): the pools after the step bit for bit, lengths exact,
attention and context within the step's tolerances, the block-id rule. The
blocks no row owns are filled with Inf/NaN, so a read outside the table would
show; and with the table laid out contiguously the results equal the
in-place step's bit for bit.
"""
import numpy as np
import pytest
import torch

import bounds
import kv_cache_append_gb300 as kvc
import oracle
import workloads
from test_gpu_parity import DEV, SMALL, TC, TOL, _bits, _built  # noqa: F401
from workloads import Spec

pytestmark = pytest.mark.gpu


def to_pool(cache, bs, seed, spare=5):
    """Logical caches [B, Hk, M, W] as a shuffled pool with `spare` extra
    blocks (Inf keys / NaN values); returns (pool, table)."""
    B, Hk, M, W = cache.shape
    mb = M // bs
    blocks = cache.reshape(B, Hk, mb, bs, W).permute(0, 2, 1, 3, 4).reshape(B * mb, Hk, bs, W)
    n = B * mb + spare
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(seed))[:B * mb]
    pool = torch.full((n, Hk, bs, W), float("nan"), dtype=cache.dtype)
    pool[perm] = blocks
    return pool.contiguous(), perm.reshape(B, mb).to(torch.int32)


def run_paged(x, bs, seed=0, table_edit=None):
    kp, table = to_pool(x.key_cache, bs, seed)
    vp, _ = to_pool(x.value_cache, bs, seed)
    kp[torch.isnan(kp)] = float("inf")  # spare key blocks: +Inf, value blocks: NaN
    if table_edit:
        table_edit(table)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kpg, vpg = kp.to(DEV), vp.to(DEV)
    out = kvc.kv_cache_attention_step_paged(x.query.to(DEV), x.new_key.to(DEV),
                                            x.new_value.to(DEV), kpg, vpg, table.to(DEV),
                                            x.lengths.to(DEV), x.append_mask.to(DEV), x.options,
                                            status=status)
    torch.cuda.synchronize()
    ref = oracle.step_paged(x.query, x.new_key, x.new_value, kp, vp, table, x.lengths,
                            x.append_mask, x.options)
    return out, int(status.item()), ref, table


def compare_paged(x, out, status, ref, expect_flags=0, table=None):
    """Pools bit for bit, lengths, flags, the absolute bars and, given the
    block table, the per-row bounds on the logical caches read back through it."""
    assert torch.equal(_bits(out["key_cache"].cpu()), _bits(ref["key_cache"]))
    assert torch.equal(_bits(out["value_cache"].cpu()), _bits(ref["value_cache"]))
    assert torch.equal(out["lengths"].cpu(), ref["lengths"])
    flags = int(np.bitwise_or.reduce(ref["flags"])) if len(ref["flags"]) else 0
    assert status == flags == expect_flags
    atol_a, atol_c = TOL[x.query.dtype]
    np.testing.assert_allclose(out["attention"].double().cpu().numpy(), ref["attention"],
                               rtol=0, atol=atol_a)
    np.testing.assert_allclose(out["context"].double().cpu().numpy(), ref["context"],
                               rtol=0, atol=atol_c)
    if table is not None:
        B, mb = table.shape
        kp, vp = ref["key_cache"], ref["value_cache"]
        _, Hk, bs, D = kp.shape
        t = table.long().clamp(0, kp.shape[0] - 1)
        lk = kp[t].permute(0, 2, 1, 3, 4).reshape(B, Hk, mb * bs, D)
        lv = vp[t].permute(0, 2, 1, 3, 4).reshape(B, Hk, mb * bs, vp.shape[-1])
        xs = workloads.StepInputs(x.query, x.new_key, x.new_value, x.key_cache, x.value_cache,
                                  x.lengths, x.append_mask.clone(), x.options)
        for b in range(B):   # rows the block check rejected append nothing
            if ref["flags"][b]:
                xs.append_mask[b] = False
        bounds.check_step(xs, lk, lv, out["attention"].double().cpu().numpy(),
                          out["context"].double().cpu().numpy(), ref["attention"],
                          ref["context"], float(x.options.get("scale", kvc.default_scale(D))),
                          "paged")


CASES = {
    # (spec, block sizes)
    "specdec_bf16": (SMALL["specdec_bf16"].replace(M=768), (16, 64, 1)),
    "decode_bf16": (SMALL["decode_bf16_ragged_M"].replace(M=1024), (32, 128)),
    "fp32_gqa": (SMALL["chunk_fp32_Q40"], (8,)),
    "tc_r128_fp16_D192": (TC["r128_fp16_D192_Dv128"].replace(M=3072), (64, 16, 128, 8)),
    "tc_r64_bf16_ragged": (TC["r64_bf16_ragged"].replace(M=704), (32, 64)),
    "tc_r160_bf16_chunk40": (TC["r160_bf16_chunk40"], (40, 8)),   # 40: not a TMA block size
    "generic_D5": (Spec(B=3, Hq=4, Hk=2, Q=3, D=5, Dv=7, M=48, dtype="bf16",
                        counts=("uniform", 0, 3)), (4,)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_paged_parity(name):
    spec, sizes = CASES[name]
    for i, bs in enumerate(sizes):
        assert spec.M % bs == 0
        x = workloads.generate(spec, 20 + i)
        out, status, ref, table = run_paged(x, bs, seed=i)
        compare_paged(x, out, status, ref, table=table)


@pytest.mark.parametrize("name,bs", [("specdec_bf16", 16), ("tc_r128_fp16_D192", 16),
                                     ("tc_r128_fp16_D192", 64)])
def test_paged_equals_inplace_bitwise(name, bs):
    spec = CASES[name][0]
    x = workloads.generate(spec, 7)
    B, Hk, M = x.key_cache.shape[:3]
    mb = M // bs
    table = torch.arange(B * mb, dtype=torch.int32).reshape(B, mb).to(DEV)
    xg = x.to(DEV)

    def pool(c):  # [B, Hk, M, W] -> [B * mb, Hk, bs, W] in table order
        W = c.shape[-1]
        return c.reshape(B, Hk, mb, bs, W).permute(0, 2, 1, 3, 4).reshape(B * mb, Hk, bs, W)
    kp, vp = pool(xg.key_cache).contiguous(), pool(xg.value_cache).contiguous()
    got = kvc.kv_cache_attention_step_paged(xg.query, xg.new_key, xg.new_value, kp, vp, table,
                                            xg.lengths, xg.append_mask, xg.options)
    kc, vc = xg.key_cache.clone(), xg.value_cache.clone()
    want = kvc.kv_cache_attention_step_inplace(xg.query, xg.new_key, xg.new_value, kc, vc,
                                               xg.lengths, xg.append_mask, xg.options)
    torch.cuda.synchronize()
    for k in ("attention", "context"):
        assert torch.equal(_bits(got[k]), _bits(want[k])), k
    assert torch.equal(got["lengths"], want["lengths"])
    assert torch.equal(_bits(kp), _bits(pool(kc))) and torch.equal(_bits(vp), _bits(pool(vc)))


@pytest.mark.parametrize("name,bs", [("specdec_bf16", 16), ("tc_r128_fp16_D192", 64)])
def test_paged_bad_block_ids(name, bs):
    spec = CASES[name][0].replace(counts=("uniform", 1, CASES[name][0].Q))
    x = workloads.generate(spec, 5)

    def edit(table):
        table[1, 0] = 10 ** 6      # row 1 always needs block 0
        table[-1, -1] = -5         # the last row needs its last block only if it reaches it
    out, status, ref, table = run_paged(x, bs, seed=3, table_edit=edit)
    compare_paged(x, out, status, ref, expect_flags=kvc.DEV_OVERFLOW, table=table)
    assert ref["flags"][1] == 1


def test_paged_decode_full_size():
    """gqa_decode shapes on a shuffled pool of 16-slot blocks; sampled rows."""
    spec = workloads.SPECS["gqa_decode"]
    bs = 16
    x = workloads.generate(spec, seed=1, device=DEV)
    B, Hk, M, D = x.key_cache.shape
    mb = M // bs
    perm = torch.randperm(B * mb, generator=torch.Generator().manual_seed(2)).to(DEV)
    table = perm.reshape(B, mb).to(torch.int32)

    def pool(c):
        W = c.shape[-1]
        blocks = c.reshape(B, Hk, mb, bs, W).permute(0, 2, 1, 3, 4).reshape(B * mb, Hk, bs, W)
        out = torch.empty_like(blocks)
        out[perm] = blocks
        return out
    kp, vp = pool(x.key_cache), pool(x.value_cache)
    out = kvc.kv_cache_attention_step_paged(x.query, x.new_key, x.new_value, kp, vp, table,
                                            x.lengths, x.append_mask, x.options)
    torch.cuda.synchronize()
    # the pool read back through the table is the updated logical cache
    logical = {"key_cache": kp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, Hk, M, D),
               "value_cache": vp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, Hk, M, D),
               "lengths": out["lengths"]}
    from test_gpu_parity import check_append_property, compare_batch_rows
    check_append_property(x, logical)
    lengths = x.lengths.cpu().numpy()
    bsel = {int(lengths.argmax()), int(lengths.argmin()), 7}
    compare_batch_rows(x, out, bsel)
