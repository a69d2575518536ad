"""Pins for the fp64 oracle: each function checks the oracle against something
other than itself -- the worked numbers a page prints, a closed form, an
invariant the contract states, or a library routine (torch's float64
scaled_dot_product_attention) on a special case. Each takes an ``Oracle``
instance so the same pins also run against deliberately mutated oracle builds
(tests/test_oracle_mutants.py) to show that a plausible mistake fails one.

Sources:
  [contract]  "Autoregressive KV-cache append and causal attention" (biotorch,
              problems/kv_cache_attention_step), Required behavior.
  [fixed]     "Fixed-capacity KV cache" (aiengineeringfromscratch,
              practice/kv-cache-append), Task and Examples.
  [incr]      "21. KV-Cache for Incremental Decoding" (cartesia-pytorch
              problems), Step-by-Step Approach, step 6.
  [lowright]  KempnerForge pull request 542, Summary and Testing: multi-token
              appends to a filled cache with a lower-right causal mask.
  [readonly]  "ClikaRT::ops::attention_over_cache" (docs.clika.io): packed
              queries re-attend an already appended cache through slot_ids
              and cu_seqlens_k, without writing it.
"""
from __future__ import annotations

import hashlib
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle as _oracle_mod
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(gen, *shape, dtype=torch.float64, std=1.0):
    return (torch.randn(*shape, generator=gen, dtype=torch.float64) * std).to(dtype)


def _updated_cache(cache, new, lengths, counts):
    """Updated cache by torch slicing (the [contract] bullet 3 write)."""
    out = cache.clone()
    for b in range(cache.shape[0]):
        L, n = int(lengths[b]), int(counts[b])
        out[b, :, L:L + n] = new[b, :, :n]
    return out


def _sdpa_reference(q, kc, vc, nk, nv, lengths, counts, scale):
    """Attention weights and context by torch's float64 SDPA with an explicit
    boolean mask j <= length + t (GQA through enable_gqa). Weights come from
    attending an identity value matrix. Rows t >= n are returned as NaN."""
    q, kc, vc, nk, nv = (x.to(torch.float64) for x in (q, kc, vc, nk, nv))
    B, Hq, Q, D = q.shape
    M = kc.shape[2]
    K = _updated_cache(kc, nk, lengths, counts)
    V = _updated_cache(vc, nv, lengths, counts)
    j = torch.arange(M)
    t = torch.arange(Q)
    allowed = j[None, None, :] <= (torch.as_tensor(lengths)[:, None, None] + t[None, :, None])
    valid = t[None, :] < torch.as_tensor(counts)[:, None]              # [B, Q]
    allowed = allowed | ~valid[:, :, None]                             # keep NaN-free
    mask = allowed[:, None, :, :]                                      # [B,1,Q,M]
    ctx = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=scale, enable_gqa=True)
    eye = torch.eye(M, dtype=torch.float64).expand(B, K.shape[1], M, M)
    att = F.scaled_dot_product_attention(q, K, eye, attn_mask=mask, scale=scale,
                                         enable_gqa=True)
    inval = ~valid[:, None, :, None]
    return (att.masked_fill(inval, float("nan")).numpy(),
            ctx.masked_fill(inval, float("nan")).numpy())


def _counts(mask):
    return mask.to(torch.int64).sum(dim=1)


# ---------------------------------------------------------------- worked example
def pin_fixed_capacity_example(o):
    """[fixed] Examples: two appends, decode_step with q=[1,0] gives weights
    [0.40111209 0.19777581 0.40111209] (8 printed decimals) and output [3 4];
    the overflowing append leaves the length at 3 and the cache unchanged."""
    ex = json.load(open(os.path.join(GOLDEN, "fixed_capacity_example.json")))
    M, dk, dv = ex["max_len"], ex["d_k"], ex["d_v"]
    kc = torch.zeros(1, 1, M, dk)
    vc = torch.zeros(1, 1, M, dv)
    lengths = torch.zeros(1, dtype=torch.int64)
    out = None
    for i, app in enumerate(ex["appends"]):
        k = torch.tensor(app["k"], dtype=torch.float32)[None, None]
        v = torch.tensor(app["v"], dtype=torch.float32)[None, None]
        Q = k.shape[2]
        q = (torch.tensor([ex["decode_query"]], dtype=torch.float32)[None, None]
             if i == len(ex["appends"]) - 1 else torch.zeros(1, 1, Q, dk))
        out = o.step(q, k, v, kc, vc, lengths, torch.ones(1, Q, dtype=torch.bool), {})
        assert int(out["lengths"][0]) == app["len_after"]
        kc, vc, lengths = out["key_cache"], out["value_cache"], out["lengths"]
    n = len(ex["values_after"])
    assert torch.equal(vc[0, 0, :n], torch.tensor(ex["values_after"], dtype=torch.float32))
    w = out["attention"][0, 0, 0]
    half_unit = 0.5 * 10.0 ** (-ex["weights_printed_decimals"])
    np.testing.assert_allclose(w[:n], ex["weights"], rtol=0, atol=half_unit + 1e-15)
    assert np.all(w[n:] == 0.0)
    np.testing.assert_allclose(out["context"][0, 0, 0], ex["output"], rtol=0, atol=1e-12)
    # the overflowing append: outside the contract, the row appends nothing
    ov = ex["overflow_append"]
    k = torch.tensor(ov["k"], dtype=torch.float32)[None, None]
    v = torch.tensor(ov["v"], dtype=torch.float32)[None, None]
    Q = k.shape[2]
    out2 = o.step(torch.zeros(1, 1, Q, dk), k, v, kc, vc, lengths,
                  torch.ones(1, Q, dtype=torch.bool), {})
    assert int(out2["lengths"][0]) == ov["len_after"]
    assert out2["flags"][0] & _oracle_mod.FLAG_OVERFLOW
    assert torch.equal(out2["key_cache"], kc) and torch.equal(out2["value_cache"], vc)
    assert np.all(out2["attention"] == 0.0) and np.all(out2["context"] == 0.0)


def pin_fixed_capacity_closed_form(o):
    """[fixed] output [3, 4] in closed form: slots 0 and 2 tie (w1 = w3 = a,
    w2 = b, 2a + b = 1), so out = (6a + 3b, 8a + 4b) = (3, 4) exactly; and
    a = e^{1/sqrt2} / (2 e^{1/sqrt2} + 1)."""
    kc = torch.zeros(1, 1, 3, 2)
    vc = torch.zeros(1, 1, 3, 2)
    kc[0, 0, 0] = torch.tensor([1.0, 0.0])
    kc[0, 0, 1] = torch.tensor([0.0, 1.0])
    vc[0, 0, 0] = torch.tensor([1.0, 2.0])
    vc[0, 0, 1] = torch.tensor([3.0, 4.0])
    out = o.step(torch.tensor([[[[1.0, 0.0]]]]), torch.tensor([[[[1.0, 1.0]]]]),
                 torch.tensor([[[[5.0, 6.0]]]]), kc, vc, torch.tensor([2]),
                 torch.ones(1, 1, dtype=torch.bool), {})
    e = math.exp(1.0 / math.sqrt(2.0))
    a = e / (2 * e + 1)
    np.testing.assert_allclose(out["attention"][0, 0, 0], [a, 1 - 2 * a, a], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["context"][0, 0, 0], [3.0, 4.0], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- stability
def pin_large_scores_finite(o):
    """[fixed] Constraints: scores above 1000 keep the output finite. One key
    scores 5000, the others at most 10: the weights are one-hot (exp(-4990)
    underflows to 0 in double) and the context equals that value row."""
    D, M = 4, 8
    kc = torch.zeros(1, 1, M, D)
    kc[0, 0, :, 0] = torch.tensor([1, 1000, 2, 3, 1, 0, 0, 0], dtype=torch.float32)
    vc = torch.arange(M * 3, dtype=torch.float32).reshape(1, 1, M, 3)
    q = torch.tensor([[[[10.0, 0, 0, 0]]]])
    out = o.step(q, torch.zeros(1, 1, 1, D), torch.zeros(1, 1, 1, 3), kc, vc,
                 torch.tensor([5]), torch.ones(1, 1, dtype=torch.bool), {"scale": 0.5})
    w = out["attention"][0, 0, 0]
    assert np.all(np.isfinite(w)) and np.all(np.isfinite(out["context"]))
    assert w[1] == 1.0 and np.all(np.delete(w, 1) == 0.0)
    np.testing.assert_array_equal(out["context"][0, 0, 0], vc[0, 0, 1].double().numpy())


# ---------------------------------------------------------------- library special cases
def pin_incremental_equals_full_causal(o):
    """[incr] step 6: decoding token by token from an empty cache gives
    exactly the rows of one-shot causal attention (torch float64 SDPA,
    is_causal=True, enable_gqa=True)."""
    gen = torch.Generator().manual_seed(11)
    B, Hq, Hk, T, D, Dv = 2, 4, 2, 9, 5, 3
    M = T + 3
    q = _rand(gen, B, Hq, T, D)
    k = _rand(gen, B, Hk, T, D)
    v = _rand(gen, B, Hk, T, Dv)
    kc = _rand(gen, B, Hk, M, D)   # garbage everywhere: nothing is valid yet
    vc = _rand(gen, B, Hk, M, Dv)
    lengths = torch.zeros(B, dtype=torch.int64)
    ctxs = []
    for t in range(T):
        out = o.step(q[:, :, t:t + 1].float(), k[:, :, t:t + 1].float(),
                     v[:, :, t:t + 1].float(), kc.float(), vc.float(), lengths,
                     torch.ones(B, 1, dtype=torch.bool), {})
        kc, vc, lengths = out["key_cache"], out["value_cache"], out["lengths"]
        ctxs.append(out["context"][:, :, 0])
    inc = np.stack(ctxs, axis=2)
    full = F.scaled_dot_product_attention(q.float().double(), k.float().double(),
                                          v.float().double(), is_causal=True,
                                          enable_gqa=True).numpy()
    np.testing.assert_allclose(inc, full, rtol=0, atol=1e-12)
    assert torch.equal(lengths, torch.full((B,), T))


def _chunk_chain_vs_full(o, prefix, chunks, B, Hq, Hk, D, Dv, seed, dtype=torch.float32):
    gen = torch.Generator().manual_seed(seed)
    T = prefix + sum(chunks)
    M = T + 5
    q = _rand(gen, B, Hq, T, D).to(dtype)
    k = _rand(gen, B, Hk, T, D).to(dtype)
    v = _rand(gen, B, Hk, T, Dv).to(dtype)
    kc = _rand(gen, B, Hk, M, D).to(dtype)
    vc = _rand(gen, B, Hk, M, Dv).to(dtype)
    kc[:, :, :prefix] = k[:, :, :prefix]
    vc[:, :, :prefix] = v[:, :, :prefix]
    lengths = torch.full((B,), prefix, dtype=torch.int64)
    full_ctx = F.scaled_dot_product_attention(q.double(), k.double(), v.double(),
                                              is_causal=True, enable_gqa=True).numpy()
    eye = torch.eye(T, dtype=torch.float64).expand(B, Hk, T, T)
    full_att = F.scaled_dot_product_attention(q.double(), k.double(), eye, is_causal=True,
                                              enable_gqa=True).numpy()
    pos = prefix
    for c in chunks:
        out = o.step(q[:, :, pos:pos + c], k[:, :, pos:pos + c], v[:, :, pos:pos + c], kc, vc,
                     lengths, torch.ones(B, c, dtype=torch.bool), {})
        np.testing.assert_allclose(out["context"], full_ctx[:, :, pos:pos + c], rtol=0,
                                   atol=1e-12)
        np.testing.assert_allclose(out["attention"][..., :T], full_att[:, :, pos:pos + c],
                                   rtol=0, atol=1e-12)
        assert np.all(out["attention"][..., T:] == 0.0)
        kc, vc, lengths = out["key_cache"], out["value_cache"], out["lengths"]
        pos += c
    assert torch.equal(kc[:, :, :T], k) and torch.equal(vc[:, :, :T], v)


def pin_chunked_appends_equal_full_rows(o):
    """[lowright] Testing: chunks 3+2+3, 1+7 and 5+1+2 appended to a filled
    cache (GQA, batch 2) reproduce the full forward's rows, weights included;
    and 40/32/24 on a longer prefix as in the pull request's model test."""
    for chunks in ((3, 2, 3), (1, 7), (5, 1, 2)):
        _chunk_chain_vs_full(o, prefix=6, chunks=chunks, B=2, Hq=8, Hk=2, D=4, Dv=3, seed=5)
    _chunk_chain_vs_full(o, prefix=37, chunks=(40, 32, 24), B=2, Hq=8, Hk=2, D=8, Dv=8, seed=6)


def pin_bruteforce_vs_sdpa(o):
    """[contract] bullets 2-5 on small random cases (ragged lengths and
    counts, GQA and MHA, D != Dv, random tails), against torch float64 SDPA
    with the explicit mask j <= length + t; rows t >= n must be all zero."""
    cases = [
        dict(B=3, Hq=4, Hk=2, Q=4, D=5, Dv=3, M=13, seed=1),
        dict(B=2, Hq=3, Hk=3, Q=2, D=2, Dv=6, M=7, seed=2),
        dict(B=4, Hq=8, Hk=1, Q=3, D=7, Dv=4, M=11, seed=3),
        dict(B=1, Hq=2, Hk=1, Q=5, D=1, Dv=1, M=5, seed=4),
    ]
    for c in cases:
        gen = torch.Generator().manual_seed(c["seed"])
        rng = np.random.default_rng(c["seed"])
        B, Hq, Hk, Q, D, Dv, M = (c[x] for x in ("B", "Hq", "Hk", "Q", "D", "Dv", "M"))
        q = _rand(gen, B, Hq, Q, D).float()
        nk = _rand(gen, B, Hk, Q, D).float()
        nv = _rand(gen, B, Hk, Q, Dv).float()
        kc = _rand(gen, B, Hk, M, D).float()
        vc = _rand(gen, B, Hk, M, Dv).float()
        lengths = torch.as_tensor(rng.integers(0, M - Q + 1, size=B))
        counts = rng.integers(0, Q + 1, size=B)
        mask = workloads.prefix_mask(counts, Q)
        scale = float(rng.uniform(0.2, 1.5))
        out = o.step(q, nk, nv, kc, vc, lengths, mask, {"scale": scale})
        ref_att, ref_ctx = _sdpa_reference(q, kc, vc, nk, nv, lengths, counts, scale)
        valid = ~np.isnan(ref_ctx[..., 0])
        np.testing.assert_allclose(out["attention"][valid], ref_att[valid], rtol=0, atol=1e-12)
        np.testing.assert_allclose(out["context"][valid], ref_ctx[valid], rtol=0, atol=1e-12)
        assert np.all(out["attention"][~valid] == 0.0) and np.all(out["context"][~valid] == 0.0)
        assert torch.equal(out["lengths"], lengths + torch.as_tensor(counts))
        assert torch.equal(out["key_cache"], _updated_cache(kc, nk, lengths, counts))
        assert torch.equal(out["value_cache"], _updated_cache(vc, nv, lengths, counts))
        # sampled-row entry point: same rows, read through the definition
        bht = [(b, h, t) for b in range(B) for h in range(Hq) for t in range(Q)]
        att_r, ctx_r = o.rows(q, nk, nv, kc, vc, lengths, mask, bht, {"scale": scale})
        np.testing.assert_array_equal(att_r, out["attention"].reshape(-1, M))
        np.testing.assert_array_equal(ctx_r, out["context"].reshape(-1, Dv))


# ---------------------------------------------------------------- contract invariants
def pin_q0_and_n0_are_noops(o):
    """[contract] bullet 6: Q = 0, or rows with n = 0, preserve cache and
    lengths and return empty / zero query outputs."""
    gen = torch.Generator().manual_seed(7)
    B, Hq, Hk, D, Dv, M = 2, 4, 2, 3, 2, 6
    kc = _rand(gen, B, Hk, M, D).to(torch.bfloat16)
    vc = _rand(gen, B, Hk, M, Dv).to(torch.bfloat16)
    lengths = torch.tensor([2, 6])
    out = o.step(torch.zeros(B, Hq, 0, D, dtype=torch.bfloat16),
                 torch.zeros(B, Hk, 0, D, dtype=torch.bfloat16),
                 torch.zeros(B, Hk, 0, Dv, dtype=torch.bfloat16), kc, vc, lengths,
                 torch.zeros(B, 0, dtype=torch.bool), {})
    assert out["attention"].shape == (B, Hq, 0, M) and out["context"].shape == (B, Hq, 0, Dv)
    assert torch.equal(out["key_cache"].view(torch.int16), kc.view(torch.int16))
    assert torch.equal(out["value_cache"].view(torch.int16), vc.view(torch.int16))
    assert torch.equal(out["lengths"], lengths)
    Q = 3
    q = _rand(gen, B, Hq, Q, D).to(torch.bfloat16)
    nk = _rand(gen, B, Hk, Q, D).to(torch.bfloat16)
    nv = _rand(gen, B, Hk, Q, Dv).to(torch.bfloat16)
    out = o.step(q, nk, nv, kc, vc, lengths, torch.zeros(B, Q, dtype=torch.bool), {})
    assert torch.equal(out["key_cache"].view(torch.int16), kc.view(torch.int16))
    assert torch.equal(out["value_cache"].view(torch.int16), vc.view(torch.int16))
    assert torch.equal(out["lengths"], lengths)
    assert np.all(out["attention"] == 0.0) and np.all(out["context"] == 0.0)


def pin_first_token_one_hot(o):
    """[contract] with length 0 and n = 1 the only allowed slot is 0: the
    weights are exactly one-hot and the context is the new value row, exactly."""
    gen = torch.Generator().manual_seed(8)
    B, Hq, Hk, D, Dv, M = 2, 6, 3, 4, 5, 7
    nv = _rand(gen, B, Hk, 1, Dv).float()
    out = o.step(_rand(gen, B, Hq, 1, D).float(), _rand(gen, B, Hk, 1, D).float(), nv,
                 _rand(gen, B, Hk, M, D).float(), _rand(gen, B, Hk, M, Dv).float(),
                 torch.zeros(B, dtype=torch.int64), torch.ones(B, 1, dtype=torch.bool), {})
    att = out["attention"][:, :, 0]
    assert np.all(att[..., 0] == 1.0) and np.all(att[..., 1:] == 0.0)
    want = nv[:, :, 0].double().repeat_interleave(Hq // Hk, dim=1).numpy()
    np.testing.assert_array_equal(out["context"][:, :, 0], want)


def pin_gqa_equals_replicated_mha(o):
    """[contract] bullet 2: query head h uses KV head floor(h / (Hq / Hk)).
    GQA must equal MHA on KV heads replicated by repeat_interleave."""
    gen = torch.Generator().manual_seed(9)
    rng = np.random.default_rng(9)
    B, Hq, Hk, Q, D, Dv, M = 2, 6, 2, 3, 4, 3, 10
    q = _rand(gen, B, Hq, Q, D).float()
    nk = _rand(gen, B, Hk, Q, D).float()
    nv = _rand(gen, B, Hk, Q, Dv).float()
    kc = _rand(gen, B, Hk, M, D).float()
    vc = _rand(gen, B, Hk, M, Dv).float()
    lengths = torch.as_tensor(rng.integers(0, M - Q + 1, size=B))
    mask = workloads.prefix_mask([3, 2], Q)
    g = o.step(q, nk, nv, kc, vc, lengths, mask, {})
    G = Hq // Hk
    rep = [x.repeat_interleave(G, dim=1) for x in (nk, nv, kc, vc)]
    m = o.step(q, *rep[:2], *rep[2:], lengths, mask, {})
    np.testing.assert_array_equal(g["attention"], m["attention"])
    np.testing.assert_array_equal(g["context"], m["context"])


def pin_tail_and_future_isolation(o):
    """[contract] bullet 6: cache-tail values and future tokens cannot
    influence an earlier query's context. Poison every slot >= new_length
    with huge values, and the last appended token: earlier rows are unchanged."""
    gen = torch.Generator().manual_seed(10)
    B, Hq, Hk, Q, D, Dv, M = 2, 4, 2, 4, 3, 3, 12
    q = _rand(gen, B, Hq, Q, D).float()
    nk = _rand(gen, B, Hk, Q, D).float()
    nv = _rand(gen, B, Hk, Q, Dv).float()
    kc = _rand(gen, B, Hk, M, D).float()
    vc = _rand(gen, B, Hk, M, Dv).float()
    lengths = torch.tensor([3, 5])
    mask = torch.ones(B, Q, dtype=torch.bool)
    base = o.step(q, nk, nv, kc, vc, lengths, mask, {})
    kc2, vc2 = kc.clone(), vc.clone()
    for b in range(B):
        N = int(lengths[b]) + Q
        kc2[b, :, N:] = 1e4
        vc2[b, :, N:] = -1e6
    tail = o.step(q, nk, nv, kc2, vc2, lengths, mask, {})
    np.testing.assert_array_equal(base["attention"], tail["attention"])
    np.testing.assert_array_equal(base["context"], tail["context"])
    nk3, nv3 = nk.clone(), nv.clone()
    nk3[:, :, Q - 1] = 1e4
    nv3[:, :, Q - 1] = -1e6
    fut = o.step(q, nk3, nv3, kc, vc, lengths, mask, {})
    np.testing.assert_array_equal(base["attention"][:, :, :Q - 1], fut["attention"][:, :, :Q - 1])
    np.testing.assert_array_equal(base["context"][:, :, :Q - 1], fut["context"][:, :, :Q - 1])
    assert not np.array_equal(base["context"][:, :, Q - 1], fut["context"][:, :, Q - 1])


def pin_rows_sum_to_one_zero_is_positive(o):
    """[contract] softmax over the allowed keys: every valid row sums to 1;
    every masked entry is +0.0 (never -0.0 or NaN)."""
    spec = workloads.SPECS["tiny_fp32"]
    for seed in range(3):
        x = workloads.generate(spec, seed)
        out = o.step(*x.args(), x.options)
        att = out["attention"]
        counts = _counts(x.append_mask).numpy()
        for b in range(spec.B):
            L = int(x.lengths[b])
            for t in range(spec.Q):
                rowset = att[b, :, t]
                if t < counts[b]:
                    np.testing.assert_allclose(rowset.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
                    tail = rowset[:, L + t + 1:]
                else:
                    tail = rowset
                assert np.all(tail == 0.0) and not np.any(np.signbit(tail))


def pin_inputs_unchanged(o):
    """[contract] bullet 4 and [fixed] Constraints: the inputs are never
    modified (the returned cache is a copy)."""
    x = workloads.generate(workloads.SPECS["tiny_fp32"], 3)
    digest = [hashlib.sha256(t.numpy().tobytes()).hexdigest() for t in x.args()]
    out = o.step(*x.args(), x.options)
    assert [hashlib.sha256(t.numpy().tobytes()).hexdigest() for t in x.args()] == digest
    out["key_cache"].zero_()
    assert hashlib.sha256(x.key_cache.numpy().tobytes()).hexdigest() == digest[3]


def pin_contract_violations_append_nothing(o):
    """Outside the contract ([contract] bullet 7): a non-prefix mask, length
    > M or length + n > M. The row appends nothing, keeps its length and
    returns zero query outputs, with a flag ([fixed] Task: when append raises,
    the cache does not change)."""
    gen = torch.Generator().manual_seed(12)
    B, Hq, Hk, Q, D, Dv, M = 4, 2, 1, 3, 2, 2, 6
    x = [_rand(gen, B, Hq, Q, D).float(), _rand(gen, B, Hk, Q, D).float(),
         _rand(gen, B, Hk, Q, Dv).float(), _rand(gen, B, Hk, M, D).float(),
         _rand(gen, B, Hk, M, Dv).float()]
    lengths = torch.tensor([1, 5, 7, 2])
    mask = torch.tensor([[1, 0, 1], [1, 1, 0], [1, 0, 0], [1, 1, 0]], dtype=torch.bool)
    out = o.step(*x, lengths, mask, {})
    assert list(out["flags"]) == [_oracle_mod.FLAG_MASK, _oracle_mod.FLAG_OVERFLOW,
                                  _oracle_mod.FLAG_OVERFLOW, 0]
    assert torch.equal(out["lengths"], torch.tensor([1, 5, 7, 4]))
    for b in range(3):
        assert torch.equal(out["key_cache"][b], x[3][b])
        assert torch.equal(out["value_cache"][b], x[4][b])
        assert np.all(out["attention"][b] == 0.0) and np.all(out["context"][b] == 0.0)
    assert np.all(out["context"][3, :, :2] != 0.0)


# ---------------------------------------------------------------- storage decoding
def pin_widen_fp16_all_patterns(o):
    """Every binary16 bit pattern widens to numpy's float16 -> float64 value."""
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    h = bits.view(torch.float16)
    got = o.widen(h)
    want = h.numpy().astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def pin_widen_bf16_all_patterns(o):
    """Every bfloat16 bit pattern widens to torch's bfloat16 -> float64 value."""
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    h = bits.view(torch.bfloat16)
    got = o.widen(h)
    want = h.to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def pin_low_precision_inputs_vs_sdpa(o):
    """bf16 and fp16 storage: the oracle widens exactly, so it must equal the
    float64 SDPA on the widened values."""
    for dt in (torch.bfloat16, torch.float16):
        spec = workloads.Spec(B=2, Hq=4, Hk=2, Q=3, D=6, Dv=5, M=14, dtype="f32",
                              lengths=("uniform", 0, 11), counts=("uniform", 0, 3))
        x = workloads.generate(spec, 21)
        q, nk, nv, kc, vc = (t.to(dt) for t in (x.query, x.new_key, x.new_value, x.key_cache,
                                                x.value_cache))
        counts = _counts(x.append_mask)
        out = o.step(q, nk, nv, kc, vc, x.lengths, x.append_mask, {"scale": 0.3})
        ref_att, ref_ctx = _sdpa_reference(q, kc, vc, nk, nv, x.lengths, counts, 0.3)
        valid = ~np.isnan(ref_ctx[..., 0])
        np.testing.assert_allclose(out["attention"][valid], ref_att[valid], rtol=0, atol=1e-12)
        np.testing.assert_allclose(out["context"][valid], ref_ctx[valid], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- [readonly]
def _pack_step_queries(x, counts):
    """The step's valid query rows (t < n_b) as packed [total_q, Hq, D] rows."""
    rows, cu = [], [0]
    for b in range(x.query.shape[0]):
        n = int(counts[b])
        rows.append(x.query[b, :, :n].permute(1, 0, 2))  # [n, Hq, D]
        cu.append(cu[-1] + n)
    return torch.cat(rows, 0).contiguous(), torch.tensor(cu, dtype=torch.int32)


def pin_attend_cache_equals_step_context(o):
    """[readonly] + [contract]: appending n rows and attending with the step
    gives the context that re-attending the updated cache with those n
    queries (total length L + n) gives."""
    from workloads import Spec
    for dtype, seed in (("f32", 0), ("bf16", 1), ("f16", 2)):
        spec = Spec(B=3, Hq=4, Hk=2, Q=4, D=16, Dv=8, M=40, dtype=dtype,
                    counts=("uniform", 0, 4))
        x = workloads.generate(spec, seed)
        ref = o.step(*x.args(), x.options)
        counts = x.append_mask.to(torch.int64).sum(1)
        q, cu = _pack_step_queries(x, counts)
        kl = (x.lengths + counts).to(torch.int32)
        out, flags = o.attend_cache(q, ref["key_cache"], ref["value_cache"], cu, kl)
        assert not flags.any()
        for b in range(spec.B):
            for t in range(int(counts[b])):
                np.testing.assert_allclose(out[int(cu[b]) + t], ref["context"][b, :, t],
                                           rtol=0, atol=1e-12)


def pin_attend_cache_vs_sdpa(o):
    """[readonly]: torch's fp64 scaled_dot_product_attention with an explicit
    lower-right boolean mask, per sequence, through the slot map."""
    g = torch.Generator().manual_seed(5)
    Hq, Hk, D, Dv, M, slots = 6, 2, 8, 5, 24, 4
    kc = torch.randn(slots, Hk, M, D, generator=g, dtype=torch.float64).float()
    vc = torch.randn(slots, Hk, M, Dv, generator=g, dtype=torch.float64).float()
    S, K = [3, 1, 0, 5], [10, 1, 7, 24]
    slot = torch.tensor([2, 0, 3, 1], dtype=torch.int32)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(S)]), dtype=torch.int32)
    q = torch.randn(int(cu[-1]), Hq, D, generator=g, dtype=torch.float64).float()
    scale = 0.3
    out, flags = o.attend_cache(q, kc, vc, cu, torch.tensor(K, dtype=torch.int32), slot,
                                scale=scale)
    assert not flags.any()
    q, kc, vc = q.double(), kc.double(), vc.double()
    for b in range(len(S)):
        if S[b] == 0:
            continue
        s = int(slot[b])
        keys = kc[s, :, :K[b]].repeat_interleave(Hq // Hk, 0)      # [Hq, K, D]
        vals = vc[s, :, :K[b]].repeat_interleave(Hq // Hk, 0)
        qb = q[int(cu[b]):int(cu[b + 1])].permute(1, 0, 2)          # [Hq, S, D]
        pos = torch.arange(S[b])[:, None] + (K[b] - S[b])
        allowed = torch.arange(K[b])[None, :] <= pos                # lower-right causal
        want = F.scaled_dot_product_attention(qb, keys, vals, attn_mask=allowed, scale=scale)
        np.testing.assert_allclose(out[int(cu[b]):int(cu[b + 1])],
                                   want.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_attend_cache_slot_permutation(o):
    """[readonly]: permuting the cache rows together with slot_ids changes nothing."""
    g = torch.Generator().manual_seed(8)
    kc = torch.randn(5, 1, 12, 4, generator=g).to(torch.bfloat16)
    vc = torch.randn(5, 1, 12, 3, generator=g).to(torch.bfloat16)
    q = torch.randn(6, 2, 4, generator=g).to(torch.bfloat16)
    cu = torch.tensor([0, 2, 3, 6], dtype=torch.int32)
    kl = torch.tensor([5, 12, 3], dtype=torch.int32)
    slot = torch.tensor([4, 0, 2], dtype=torch.int32)
    a, _ = o.attend_cache(q, kc, vc, cu, kl, slot)
    perm = torch.tensor([3, 1, 4, 0, 2])  # new row i holds old row perm[i]
    inv = torch.argsort(perm)
    b, _ = o.attend_cache(q, kc[perm], vc[perm], cu, kl, inv[slot.long()].to(torch.int32))
    np.testing.assert_array_equal(a, b)


def pin_attend_cache_outside_contract(o):
    """[readonly]: a sequence with S > K, K > M or its slot out of range gets
    zero rows and a flag; the others are untouched by it."""
    kc = torch.ones(2, 1, 8, 4)
    vc = torch.ones(2, 1, 8, 4)
    q = torch.ones(7, 1, 4)
    cu = torch.tensor([0, 3, 4, 5, 7], dtype=torch.int32)
    kl = torch.tensor([2, 9, 4, 5], dtype=torch.int32)
    slot = torch.tensor([0, 1, 5, 1], dtype=torch.int32)
    out, flags = o.attend_cache(q, kc, vc, cu, kl, slot)
    assert flags.tolist() == [1, 1, 1, 0]
    assert np.all(out[:5] == 0.0)
    np.testing.assert_allclose(out[5:], 1.0, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- [paged]
def _to_pool(cache, perm, max_blocks, bs):
    """[B, Hk, M, W] logical caches as a pool whose block perm[b*max_blocks + i]
    holds block i of row b; returns (pool, table)."""
    B, Hk, M, W = cache.shape
    blocks = cache.reshape(B, Hk, max_blocks, bs, W).permute(0, 2, 1, 3, 4).reshape(
        B * max_blocks, Hk, bs, W)
    pool = torch.empty_like(blocks)
    pool[perm] = blocks
    table = perm.reshape(B, max_blocks).to(torch.int32)
    return pool, table


def _from_pool(pool, table):
    B, max_blocks = table.shape
    nb, Hk, bs, W = pool.shape
    return pool[table.long()].permute(0, 2, 1, 3, 4).reshape(B, Hk, max_blocks * bs, W)


def pin_paged_equals_contiguous_step(o):
    """[paged] + [contract]: on any block placement, the paged step gives the
    contiguous step's attention, context and lengths, and the pool read back
    through the table is the contiguous step's updated cache."""
    from workloads import Spec
    for dtype, seed, bs in (("f32", 0, 4), ("bf16", 1, 8), ("f16", 2, 16)):
        spec = Spec(B=3, Hq=4, Hk=2, Q=3, D=8, Dv=4, M=48, dtype=dtype,
                    counts=("uniform", 0, 3))
        x = workloads.generate(spec, seed)
        ref = o.step(*x.args(), x.options)
        mb = spec.M // bs
        perm = torch.randperm(spec.B * mb, generator=torch.Generator().manual_seed(seed))
        kp, table = _to_pool(x.key_cache, perm, mb, bs)
        vp, _ = _to_pool(x.value_cache, perm, mb, bs)
        got = o.step_paged(x.query, x.new_key, x.new_value, kp, vp, table,
                                     x.lengths, x.append_mask, x.options)
        np.testing.assert_array_equal(got["attention"], ref["attention"])
        np.testing.assert_array_equal(got["context"], ref["context"])
        assert torch.equal(got["lengths"], ref["lengths"])
        assert torch.equal(_from_pool(got["key_cache"], table), ref["key_cache"])
        assert torch.equal(_from_pool(got["value_cache"], table), ref["value_cache"])


def pin_paged_bad_block_ids_append_nothing(o):
    """[paged]: a row whose needed table entries fall outside the pool appends
    nothing, has zero query rows and is flagged; blocks outside every row's
    table keep their bytes; the other rows are unaffected."""
    from workloads import Spec
    spec = Spec(B=3, Hq=2, Hk=1, Q=2, D=4, Dv=4, M=16, dtype="f32", counts=("fixed", 2),
                lengths=("fixed", 5))
    x = workloads.generate(spec, 3)
    bs, mb = 4, 4
    perm = torch.arange(spec.B * mb) + 2            # blocks 0 and 1 belong to nobody
    kp, table = _to_pool(x.key_cache, perm - 2, mb, bs)
    kp = torch.cat([torch.full((2, 1, bs, 4), 7.0), kp]).contiguous()
    vp, _ = _to_pool(x.value_cache, perm - 2, mb, bs)
    vp = torch.cat([torch.full((2, 1, bs, 4), 7.0), vp]).contiguous()
    table = perm.reshape(spec.B, mb).to(torch.int32)
    table[1, 1] = 99                               # row 1 needs blocks 0, 1 (slots 0..6)
    got = o.step_paged(x.query, x.new_key, x.new_value, kp, vp, table, x.lengths,
                                 x.append_mask, x.options)
    assert got["flags"].tolist() == [0, 1, 0]
    assert int(got["lengths"][1]) == 5 and np.all(got["attention"][1] == 0)
    assert torch.equal(got["key_cache"][:2], kp[:2])
    ok = table.clone()
    ok[1, 1] = 0
    ref = o.step(x.query, x.new_key, x.new_value, _from_pool(kp, ok), _from_pool(vp, ok),
                 x.lengths, x.append_mask, x.options)
    for b in (0, 2):
        np.testing.assert_array_equal(got["context"][b], ref["context"][b])


# ------------------------------------------------------------------ gradients
def _grad_case(dtype, seed):
    """A small ragged case (rows appending 3, 2, 0 and 1 tokens, one full
    cache, one empty prefix) with random upstream gradients for all four
    outputs, all stored in `dtype`."""
    g = torch.Generator().manual_seed(seed)
    B, Hq, Hk, Q, D, Dv, M = 4, 4, 2, 3, 5, 6, 10
    q = _rand(g, B, Hq, Q, D, dtype=dtype)
    nk = _rand(g, B, Hk, Q, D, dtype=dtype)
    nv = _rand(g, B, Hk, Q, Dv, dtype=dtype)
    kc = _rand(g, B, Hk, M, D, dtype=dtype)
    vc = _rand(g, B, Hk, M, Dv, dtype=dtype)
    lengths = torch.tensor([0, 4, 7, 9])
    counts = torch.tensor([3, 2, 0, 1])
    mask = torch.arange(Q)[None, :] < counts[:, None]
    grads = dict(d_key_cache=_rand(g, B, Hk, M, D, dtype=dtype),
                 d_value_cache=_rand(g, B, Hk, M, Dv, dtype=dtype),
                 d_attention=_rand(g, B, Hq, Q, M, dtype=dtype),
                 d_context=_rand(g, B, Hq, Q, Dv, dtype=dtype))
    return (q, nk, nv, kc, vc, lengths, mask), counts, grads


def _torch_step_fp64(q, nk, nv, kc, vc, lengths, counts, scale):
    """The step's four outputs as differentiable float64 torch ops, written
    independently of the oracle: the updated caches by slice assignment into
    a copy ([contract] bullet 3), query head h on KV head h // G by
    repeat_interleave (bullet 2), softmax over the allowed slots j <= L + t of
    the valid rows t < n (bullets 4-5), attention times updated values."""
    B, Hq, Q, D = q.shape
    Hk, M = kc.shape[1], kc.shape[2]
    G = Hq // Hk
    Kp, Vp = kc.clone(), vc.clone()
    for b in range(B):
        L, n = int(lengths[b]), int(counts[b])
        Kp[b, :, L:L + n] = nk[b, :, :n]
        Vp[b, :, L:L + n] = nv[b, :, :n]
    s = scale * q @ Kp.repeat_interleave(G, dim=1).transpose(-1, -2)  # [B,Hq,Q,M]
    t = torch.arange(Q)[None, :, None]
    j = torch.arange(M)[None, None, :]
    allowed = (t < counts[:, None, None]) & (j <= lengths[:, None, None] + t)  # [B,Q,M]
    allowed = allowed[:, None]
    a = torch.softmax(torch.where(allowed, s, torch.full_like(s, -1e30)), dim=-1)
    a = a * allowed.to(a.dtype)
    c = a @ Vp.repeat_interleave(G, dim=1)
    return Kp, Vp, a, c


def pin_backward_vs_autograd(o):
    """[contract] Starter code: the suite grades gradients. torch autograd of
    an independent float64 statement of the step (differentiable slicing,
    repeat_interleave, masked softmax) gives the same gradients as the
    oracle's chain rule, for every input, in fp32 and bf16 storage."""
    for dtype, seed in ((torch.float32, 31), (torch.bfloat16, 32)):
        args, counts, grads = _grad_case(dtype, seed)
        q, nk, nv, kc, vc, lengths, mask = args
        scale = 0.37
        got = o.step_backward(*args, options={"scale": scale}, **grads)
        leaves = [o.widen(t) for t in (q, nk, nv, kc, vc)]
        leaves = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in leaves]
        outs = _torch_step_fp64(*leaves, lengths, counts, scale)
        gw = [torch.tensor(o.widen(grads[k]), dtype=torch.float64)
              for k in ("d_key_cache", "d_value_cache", "d_attention", "d_context")]
        loss = sum((x * w).sum() for x, w in zip(outs, gw))
        ref = torch.autograd.grad(loss, leaves)
        for name, r in zip(("d_query", "d_new_key", "d_new_value", "d_key_cache",
                            "d_value_cache"), ref):
            np.testing.assert_allclose(got[name], r.numpy(), rtol=1e-9, atol=1e-12, err_msg=name)


def pin_backward_finite_differences(o):
    """The gradient of a scalar of the step's outputs, by central differences
    of the oracle's own forward (kvo_step) at stored fp32 values, equals the
    backward's gradient element for elements of every input (query rows of
    valid and invalid rows, appended and ignored new rows, cache slots below
    the old length, overwritten and past the new length)."""
    args, counts, grads = _grad_case(torch.float32, 33)
    q, nk, nv, kc, vc, lengths, mask = args
    opts = {"scale": 0.41}
    back = o.step_backward(*args, options=opts, **grads)
    gw = {k: o.widen(v) for k, v in grads.items()}

    def loss(xs):
        r = o.step(*xs, lengths, mask, opts)
        return float((o.widen(r["key_cache"]) * gw["d_key_cache"]).sum()
                     + (o.widen(r["value_cache"]) * gw["d_value_cache"]).sum()
                     + (r["attention"] * gw["d_attention"]).sum()
                     + (r["context"] * gw["d_context"]).sum())

    base = [q, nk, nv, kc, vc]
    picks = {0: [(1, 2, 0, 3), (2, 1, 1, 0), (0, 0, 2, 4), (3, 3, 0, 1), (1, 0, 2, 2)],
             1: [(1, 0, 1, 2), (0, 1, 2, 4), (2, 0, 0, 1)],
             2: [(1, 1, 0, 5), (0, 0, 2, 0), (3, 1, 1, 3)],
             3: [(1, 0, 2, 1), (1, 1, 4, 3), (1, 0, 5, 0), (2, 1, 6, 2), (0, 0, 9, 4)],
             4: [(1, 1, 3, 5), (1, 0, 4, 2), (2, 0, 8, 1), (3, 1, 2, 0)]}
    names = ("d_query", "d_new_key", "d_new_value", "d_key_cache", "d_value_cache")
    for which, idxs in picks.items():
        for idx in idxs:
            x0 = float(base[which][idx])
            h = 2.0 ** -9 * max(1.0, abs(x0))
            vals = []
            for sgn in (1.0, -1.0):
                xs = [t.clone() for t in base]
                xs[which][idx] = x0 + sgn * h
                vals.append((loss(xs), float(xs[which][idx])))
            fd = (vals[0][0] - vals[1][0]) / (vals[0][1] - vals[1][1])
            an = back[names[which]][idx]
            assert abs(fd - an) <= 2e-4 * max(1.0, abs(an)), (names[which], idx, fd, an)


def pin_backward_cache_routing(o):
    """[contract] bullets 3-4: each entry of a returned cache is either the old
    cache entry or a new row, so with gradients on the returned caches only,
    they go back exactly where the entries came from: slots outside
    [L, L + n) to the input cache, slots L + t to new row t (rows t >= n get
    none, overwritten cache slots get none), and the query gets none."""
    args, counts, grads = _grad_case(torch.float32, 34)
    q, nk, nv, kc, vc, lengths, mask = args
    got = o.step_backward(*args, d_key_cache=grads["d_key_cache"],
                          d_value_cache=grads["d_value_cache"])
    assert np.all(got["d_query"] == 0.0)
    for dname, nname, src in (("d_key_cache", "d_new_key", grads["d_key_cache"]),
                              ("d_value_cache", "d_new_value", grads["d_value_cache"])):
        gsrc = o.widen(src)
        want_c, want_n = gsrc.copy(), np.zeros(got[nname].shape)
        for b in range(gsrc.shape[0]):
            L, n = int(lengths[b]), int(counts[b])
            want_c[b, :, L:L + n] = 0.0
            want_n[b, :, :n] = gsrc[b, :, L:L + n]
        assert np.array_equal(got[dname], want_c), dname
        assert np.array_equal(got[nname], want_n), nname


ALL_PINS = [
    pin_fixed_capacity_example,
    pin_fixed_capacity_closed_form,
    pin_large_scores_finite,
    pin_incremental_equals_full_causal,
    pin_chunked_appends_equal_full_rows,
    pin_bruteforce_vs_sdpa,
    pin_q0_and_n0_are_noops,
    pin_first_token_one_hot,
    pin_gqa_equals_replicated_mha,
    pin_tail_and_future_isolation,
    pin_rows_sum_to_one_zero_is_positive,
    pin_inputs_unchanged,
    pin_contract_violations_append_nothing,
    pin_widen_fp16_all_patterns,
    pin_widen_bf16_all_patterns,
    pin_low_precision_inputs_vs_sdpa,
    pin_attend_cache_equals_step_context,
    pin_attend_cache_vs_sdpa,
    pin_attend_cache_slot_permutation,
    pin_attend_cache_outside_contract,
    pin_paged_equals_contiguous_step,
    pin_paged_bad_block_ids_append_nothing,
    pin_backward_vs_autograd,
    pin_backward_finite_differences,
    pin_backward_cache_routing,
]
