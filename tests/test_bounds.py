"""The per-row error bounds of bounds.py, pinned on the CPU.

They must admit what a correct kernel can return (the oracle's exact result
rounded to the output dtype, which the bounds' model covers with room for the
kernels' fp32 arithmetic) and reject plausible mistakes at every row length,
including long rows where the contract's absolute tolerances cannot fail:
a dropped scale, a causal limit one slot short, the last allowed slot dropped
and the row renormalised, rows scaled by 0.9, all-zero outputs, and backward
cache gradients with the attention-derived part missing.
"""
import numpy as np
import pytest
import torch

import bounds
import oracle
import workloads
from workloads import Spec

CASES = {
    "tiny_fp32": workloads.SPECS["tiny_fp32"],
    "gqa_bf16": Spec(B=3, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=700, dtype="bf16",
                     lengths=("uniform", 0, 699)),
    "specdec_bf16_hot": Spec(B=4, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=300, dtype="bf16",
                             lengths=("zipf", 1.2), counts=("uniform", 0, 4), hot_frac=0.1,
                             hot_scale=50.0),
    # long rows: attention entries ~1/6000, far below the 4e-3 absolute bar
    "long_fp16": Spec(B=1, Hq=4, Hk=1, Q=2, D=192, Dv=128, M=6200, dtype="f16",
                      lengths=("uniform", 6000, 6198), std=0.5, scale=0.05),
    "long_bf16": Spec(B=1, Hq=2, Hk=1, Q=2, D=128, Dv=128, M=9000, dtype="bf16",
                      lengths=("uniform", 8500, 8998)),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _scale(x):
    return float(x.options.get("scale", 1.0 / np.sqrt(x.query.shape[-1])))


def _rounded(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).double().numpy()


def _bounds_for(x, ref):
    q = x.query.double().numpy()
    K = ref["key_cache"].double().numpy()
    V = ref["value_cache"].double().numpy()
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1).numpy()
    out = []
    for b in range(q.shape[0]):
        out.append(bounds.row_bounds(q[b], K[b], V[b], int(x.lengths[b]), int(counts[b]),
                                     _scale(x), x.query.dtype, ref["attention"][b]))
    return out


@pytest.mark.parametrize("name", sorted(CASES))
def test_rounded_oracle_passes_and_mistakes_fail(name):
    x = workloads.generate(CASES[name], 4)
    assert int(x.append_mask.sum()) > 0
    ref = oracle.step(*x.args(), x.options)
    dt = x.query.dtype
    att = _rounded(ref["attention"], dt)
    ctx = _rounded(ref["context"], dt)
    # a correct result rounded to the dtype passes (check_rows also asserts that
    # scaled and zero outputs fail)
    bounds.check_step(x, ref["key_cache"], ref["value_cache"], att, ctx, ref["attention"],
                      ref["context"], _scale(x), name)
    bnds = _bounds_for(x, ref)
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1).numpy()

    def fails(att_w, ctx_w):
        for b, bnd in enumerate(bnds):
            if counts[b] == 0:
                continue
            if (bounds.attention_ratio(att_w[b], ref["attention"][b], bnd) > 1.0 or
                    bounds.context_ratio(ctx_w[b], ref["context"][b], bnd) > 1.0):
                return True
        return False

    # a dropped scale (scores unscaled)
    wrong = oracle.step(*x.args(), {"scale": 1.0})
    assert fails(_rounded(wrong["attention"], dt), _rounded(wrong["context"], dt))
    # the last allowed slot of every valid row dropped and the row renormalised
    a2 = ref["attention"].copy()
    c2 = ref["context"].copy()
    V = ref["value_cache"].double().numpy()
    G = x.query.shape[1] // x.key_cache.shape[1]
    for b in range(a2.shape[0]):
        L = int(x.lengths[b])
        for h in range(a2.shape[1]):
            for t in range(int(counts[b])):
                j = L + t
                keep = 1.0 - a2[b, h, t, j]
                if keep <= 0.0:
                    continue
                a2[b, h, t, j] = 0.0
                a2[b, h, t] /= keep
                c2[b, h, t] = a2[b, h, t, :j + 1] @ V[b, h // G, :j + 1]
    assert fails(_rounded(a2, dt), _rounded(c2, dt))
    # attention shifted by one slot (an off-by-one in the slot index)
    a3 = np.roll(ref["attention"], 1, axis=-1)
    assert fails(_rounded(a3, dt), ctx)


def test_long_rows_are_below_the_absolute_bar():
    """On long rows the absolute tolerances pass an all-zero attention and a
    context that is 10% off, which is why the per-row bounds exist."""
    x = workloads.generate(CASES["long_fp16"], 3)
    ref = oracle.step(*x.args(), x.options)
    assert np.abs(ref["attention"]).max() < 4e-3
    assert np.abs(0.1 * ref["context"]).max() < 2e-2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_gradient_bound(dtype):
    """The gradient bound admits the reference rounded to the dtype and rejects
    it scaled by 0.9, zeroed, or with a slice of its entries zeroed."""
    rng = np.random.default_rng(5)
    ref = rng.standard_normal((3, 2, 400, 64)) * 1e-3
    ref[:, :, 300:] = 0.0
    got = torch.from_numpy(ref).to(dtype).double().numpy()
    assert bounds.grad_ratio(got, ref, dtype) <= 1.0
    assert bounds.grad_ratio(0.9 * ref, ref, dtype) > 1.0
    assert bounds.grad_ratio(np.zeros_like(ref), ref, dtype) > 1.0
    cut = ref.copy()
    cut[:, :, :100] = 0.0
    assert bounds.grad_ratio(cut, ref, dtype) > 1.0
    # an entry the structure makes zero must come back exactly zero; one that
    # is zero by cancellation keeps the absolute term
    bad = got.copy()
    bad[0, 0, 350, 0] = 1e-30
    structural = np.zeros(ref.shape, dtype=bool)
    structural[:, :, 300:] = True
    assert bounds.grad_ratio(bad, ref, dtype, exact_zero=structural) > 1.0
    assert bounds.grad_ratio(bad, ref, dtype) <= 1.0


def test_grad_terms_sum_to_the_oracle_gradients():
    """grad_terms' per-term decomposition (a, g, D, ds from the oracle's
    forward pass) sums to the oracle's own backward (an independent C
    statement of the chain rule): with gradients reaching only attention and
    context, the cache gradients below the old length, the new rows' and the
    query's are exactly those sums. T bounds each sum: |sum| <= sqrt(terms) T."""
    spec = Spec(B=4, Hq=6, Hk=2, Q=3, D=16, Dv=8, M=40, dtype="f32",
                lengths=("uniform", 0, 36), counts=("uniform", 0, 3))
    x = workloads.generate(spec, 21)
    x.lengths[2] = 39   # 39 + n > M for n >= 2: a flagged row
    x.append_mask[2] = True
    g = torch.Generator().manual_seed(22)
    da = torch.randn(4, 6, 3, 40, generator=g)
    dc = torch.randn(4, 6, 3, 8, generator=g)
    ref = oracle.step_backward(*x.args(), d_attention=da, d_context=dc, options=x.options)
    assert ref["flags"][2] != 0
    fwd = oracle.step(*x.args(), options=x.options)
    scale = oracle.default_scale(16)
    t = bounds.grad_terms(x.query, x.lengths, x.append_mask, fwd, da, dc, scale, sums=True)
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1)
    for b in range(4):
        L, n = int(x.lengths[b]), (0 if ref["flags"][b] else int(counts[b]))
        np.testing.assert_allclose(t["sum_key_cache"][b, :, :L], ref["d_key_cache"][b, :, :L],
                                   rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(t["sum_value_cache"][b, :, :L],
                                   ref["d_value_cache"][b, :, :L], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(t["sum_new_key"][b, :, :n], ref["d_new_key"][b, :, :n],
                                   rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(t["sum_new_value"][b, :, :n], ref["d_new_value"][b, :, :n],
                                   rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(t["sum_query"], ref["d_query"], rtol=1e-9, atol=1e-12)
    # the root of the sum of squares bounds the sum over at most M (slots) or
    # Hq / Hk * Q (rows) terms
    assert np.all(np.abs(t["sum_query"]) <= np.sqrt(40) * t["query"] + 1e-12)
    assert np.all(np.abs(t["sum_key_cache"]) <= np.sqrt(9) * t["key_cache"] + 1e-12)
    assert np.any(t["key_cache"] > 0) and np.any(t["query"] > 0)
