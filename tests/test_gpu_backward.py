"""GPU parity of the step's gradients (kvc_step_backward) against the fp64
oracle (oracle.step_backward), and of the autograd face of
kv_cache_attention_step.

Tolerances (bounds.grad_ratio): the kernels sum in fp32 and round each
gradient to the dtype once (the tensor-core slot kernel also rounds a and ds
to the dtype as its operands), so the error is that rounding plus sums of
independently rounded terms: |got - ref| <= rtol |ref| + atol RMS(ref) per
tensor (RMS over its nonzero reference entries) plus one fp16 subnormal
spacing, with (rtol, atol) = (2^-7, 2^-5) bf16, (2^-9, 2^-8) fp16,
(1e-4, 1e-4) fp32 (atol = 8u: the Hoeffding bound on sums of independently
rounded 16-bit operands, lambda = 8). Every case runs twice: with all four upstream gradients,
and with gradients reaching only attention and context, so that the
attention-derived part of the cache gradients (about a_j * dcontext, 1e-4 on
long rows) is bounded by its own RMS rather than hidden under the routed part
(~1). On those runs, wrong variants made from the oracle's own output (the
cache gradients zeroed below the old length, the query gradient scaled by
0.9) must exceed the bound. The pure routing parts are exact: cache slots
from the new length on carry the returned caches' gradient bit for bit, and
slots a new row overwrote get exactly zero.
"""
import numpy as np
import pytest
import torch

import bounds
import kv_cache_append_gb300 as kvc
import oracle
import workloads
from test_gpu_parity import DEV, SMALL, _bits, _built  # noqa: F401
from workloads import Spec

pytestmark = pytest.mark.gpu

NAMES = ("query", "new_key", "new_value", "key_cache", "value_cache")


def upstream(x, seed, which=("key_cache", "value_cache", "attention", "context")):
    g = torch.Generator().manual_seed(seed)
    B, Hq, Q, _ = x.query.shape
    M, Dv = x.key_cache.shape[2], x.value_cache.shape[-1]
    shapes = {"key_cache": tuple(x.key_cache.shape), "value_cache": tuple(x.value_cache.shape),
              "attention": (B, Hq, Q, M), "context": (B, Hq, Q, Dv)}
    return {k: (torch.randn(*shapes[k], generator=g).to(x.query.dtype) if k in which else None)
            for k in shapes}


def structural_zeros(x, ref):
    """The row gradients the step's structure makes zero: query rows t >= n_b
    (invalid rows) and new rows t >= n_b (nothing appended), n_b = 0 for a
    row outside the contract."""
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1).numpy()
    n = np.where(np.asarray(ref["flags"]) != 0, 0, counts)
    Q = x.query.shape[2]
    invalid = np.arange(Q)[None, :] >= n[:, None]          # [B, Q]
    return {"query": invalid[:, None, :, None], "new_key": invalid[:, None, :, None],
            "new_value": invalid[:, None, :, None]}


def terms_of(x, grads):
    """bounds.grad_terms for the inputs x and the incoming gradients."""
    fwd = oracle.step(*x.args(), options=x.options)
    scale = x.options.get("scale", oracle.default_scale(x.query.shape[-1]))
    cpu = {k: (None if v is None else v.cpu()) for k, v in grads.items()}
    return bounds.grad_terms(x.query, x.lengths, x.append_mask, fwd, cpu["attention"],
                             cpu["context"], scale)


def check_grads(got, ref, x, grads, where=""):
    """Every gradient within bounds.grad_ratio (with each entry's own terms),
    the structurally zero row gradients exactly zero."""
    dt = x.query.dtype
    zeros = structural_zeros(x, ref)
    terms = terms_of(x, grads)
    for name in NAMES:
        r = ref["d_" + name]
        gw = got[name]
        gw = gw.double().cpu().numpy() if torch.is_tensor(gw) else gw
        ez = np.broadcast_to(zeros[name], r.shape) if name in zeros else None
        ratio = bounds.grad_ratio(gw, r, dt, exact_zero=ez, terms=terms[name])
        assert ratio <= 1.0, (where, name, ratio)
    return terms


def check_mutants(ref, x, lengths, terms, where=""):
    """With no gradient reaching the returned caches (grads of attention and
    context only), the cache gradients below the old length are the
    attention-derived dK', dV' alone: zeroing them, or scaling the query
    gradient by 0.9, made from the oracle's own output, must exceed the bound."""
    dt = x.query.dtype
    for name in ("key_cache", "value_cache"):
        r = ref["d_" + name]
        cut = r.copy()
        for b in range(r.shape[0]):
            cut[b, :, :max(0, int(lengths[b]))] = 0.0
        if np.any(cut != r):
            assert bounds.grad_ratio(cut, r, dt, terms=terms[name]) > 1.0, (where, name, "zeroed dK'")
    r = ref["d_query"]
    if np.any(r != 0.0):
        assert bounds.grad_ratio(0.9 * r, r, dt, terms=terms["query"]) > 1.0, (where, "0.9 dq")


def check(x, grads, status_expect=0):
    xg = x.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = kvc.kv_cache_attention_step_backward(
        *xg.args(), xg.options, status=status,
        **{f"d_{k}": (None if v is None else v.to(DEV)) for k, v in grads.items()})
    torch.cuda.synchronize()
    ref = oracle.step_backward(*x.args(), options=x.options,
                               **{f"d_{k}": v for k, v in grads.items()})
    flags = int(np.bitwise_or.reduce(ref["flags"])) if len(ref["flags"]) else 0
    assert int(status.item()) == flags == status_expect
    terms = check_grads(got, ref, x, grads)
    if grads["key_cache"] is None and grads["value_cache"] is None:
        check_mutants(ref, x, x.lengths, terms)
    # exact routing: slots from the new length on, and overwritten slots
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1)
    for name, gk in (("key_cache", grads["key_cache"]), ("value_cache", grads["value_cache"])):
        out = got[name].cpu()
        for b in range(x.query.shape[0]):
            if ref["flags"][b]:
                continue
            L, n = int(x.lengths[b]), int(counts[b])
            tail = out[b, :, L + n:]
            want = gk[b, :, L + n:] if gk is not None else torch.zeros_like(tail)
            assert torch.equal(_bits(tail), _bits(want.contiguous())), (name, b)
            assert torch.count_nonzero(out[b, :, L:L + n]) == 0, (name, b)
    return got, ref


CASES = {
    "tiny_fp32": SMALL["tiny_fp32"],
    "decode_bf16_ragged_M": SMALL["decode_bf16_ragged_M"],
    "specdec_bf16_hot": SMALL["specdec_bf16"],
    "chunk_fp32_Q40": SMALL["chunk_fp32_Q40"],
    "mqa_fp16_D192": SMALL["mqa_fp16_D192"].replace(M=700, lengths=("uniform", 100, 690)),
    "gqa_fp32_small_rows": SMALL["gqa_fp32_small_rows"],   # generic statistics path
    "generic_bf16_D5_Dv7": Spec(B=3, Hq=4, Hk=2, Q=3, D=5, Dv=7, M=50, dtype="bf16",
                                counts=("uniform", 0, 3)),
    "mha_fp16_Dv256": SMALL["mha_fp16_Dv256"],
    # the few-rows kernel at each width it takes (D = Dv = 64, 128, 256)
    "rows_f16_D64_R8": Spec(B=3, Hq=8, Hk=2, Q=2, D=64, Dv=64, M=300, dtype="f16",
                            counts=("uniform", 0, 2)),
    "rows_f32_D256_R16": Spec(B=2, Hq=8, Hk=2, Q=4, D=256, Dv=256, M=200, dtype="f32",
                              counts=("uniform", 1, 4)),
    "rows_bf16_D256_R4_ragged": Spec(B=4, Hq=4, Hk=1, Q=1, D=256, Dv=256, M=700, dtype="bf16",
                                     lengths=("uniform", 0, 699)),
    # units of more than 4 rows with D and Dv multiples of 64 that the
    # few-rows kernel does not take: the tensor-core kernel for the 16-bit ones
    # of 9-128 rows whose widths fit it (R40, R18 here), the tiled kernel for
    # the rest (each of its instances, a last row chunk of 8 rows, D != Dv,
    # tiles cut by M and N)
    "tiled_bf16_D128_R40_ragged": Spec(B=3, Hq=10, Hk=1, Q=4, D=128, Dv=128, M=500,
                                       dtype="bf16", lengths=("uniform", 0, 495),
                                       counts=("uniform", 0, 4)),
    "tiled_f16_D256_R32": Spec(B=2, Hq=8, Hk=2, Q=8, D=256, Dv=256, M=300, dtype="f16",
                               counts=("uniform", 1, 8)),
    "tiled_f32_D128_Dv64_R24": Spec(B=3, Hq=6, Hk=1, Q=4, D=128, Dv=64, M=130, dtype="f32",
                                    lengths=("uniform", 60, 126)),
    "tiled_bf16_D64_Dv192_R18": Spec(B=2, Hq=12, Hk=2, Q=3, D=64, Dv=192, M=260, dtype="bf16",
                                     hot_frac=0.05, hot_scale=20.0),
    "tiled_f16_D64_Dv128_R8": Spec(B=3, Hq=8, Hk=2, Q=2, D=64, Dv=128, M=400, dtype="f16",
                                   counts=("uniform", 0, 2)),
    # the tensor-core kernel (16-bit, 9-128 rows): 128 rows exactly with tiles
    # cut by M and N, 17 rows (111 padding rows), hot rows
    "tc_bf16_D64_R128_ragged": Spec(B=3, Hq=32, Hk=1, Q=4, D=64, Dv=64, M=700, dtype="bf16",
                                    lengths=("uniform", 0, 690), counts=("uniform", 0, 4)),
    "tc_f16_D128_R17": Spec(B=2, Hq=17, Hk=1, Q=1, D=128, Dv=128, M=300, dtype="f16",
                            lengths=("uniform", 100, 299)),
    "tc_bf16_D128_R32_hot": Spec(B=2, Hq=16, Hk=2, Q=4, D=128, Dv=128, M=500, dtype="bf16",
                                 hot_frac=0.05, hot_scale=30.0),
    # M a multiple of 8: the attention gradients staged through shared memory
    "tc_bf16_D64_R64_staged": Spec(B=3, Hq=16, Hk=1, Q=4, D=64, Dv=64, M=520, dtype="bf16",
                                   lengths=("uniform", 0, 515), counts=("uniform", 0, 4)),
    "tc_f16_D128_R32_staged": Spec(B=2, Hq=8, Hk=1, Q=4, D=128, Dv=128, M=384, dtype="f16",
                                   lengths=("uniform", 120, 379)),
    # more tiles than the tensor-core kernel has CTAs (one per SM), so that a
    # CTA's range of tiles starts, ends and crosses units mid-way
    "tc_walk_bf16_R32_units": Spec(B=40, Hq=16, Hk=2, Q=4, D=64, Dv=64, M=700, dtype="bf16",
                                   lengths=("uniform", 0, 690), counts=("uniform", 0, 4)),
    "tc_walk_f16_R64_D128": Spec(B=40, Hq=16, Hk=1, Q=4, D=128, Dv=128, M=1100, dtype="f16",
                                 lengths=("uniform", 300, 1090)),
    # new rows at slots 126-129: two in the first, whole tile (whose cache
    # gradient goes out through shared memory), two in the second, partial one
    "tc_bf16_R32_new_rows_in_whole_tile": Spec(B=2, Hq=16, Hk=2, Q=4, D=128, Dv=128, M=300,
                                               dtype="bf16", lengths=("uniform", 126, 126)),
    # statistics on the decode tensor-core kernel (16-bit, Dv = 128, at most 32
    # rows), which takes the appended rows from new_key / new_value: 16 rows
    # whose new rows straddle the first 128-slot tile's end, D = 256 (8 rows)
    # (the tiled slot kernel) and D = 64 (4 rows, the generic slot kernel)
    "dec_bf16_R16_tile_edge": Spec(B=6, Hq=16, Hk=4, Q=4, D=128, Dv=128, M=400, dtype="bf16",
                                   lengths=("uniform", 123, 129), counts=("uniform", 0, 4)),
    "dec_f16_D256_R8": Spec(B=3, Hq=8, Hk=2, Q=2, D=256, Dv=128, M=300, dtype="f16",
                            lengths=("uniform", 0, 297), counts=("uniform", 0, 2)),
    "dec_bf16_D64_R4": Spec(B=4, Hq=4, Hk=1, Q=1, D=64, Dv=128, M=260, dtype="bf16",
                            lengths=("uniform", 0, 259)),
}


# the slot kernel each case runs (kvc_backward_plan_info), so that every
# kernel stays covered
SLOT = {"tiny_fp32": "bwd_kv_kernel", "decode_bf16_ragged_M": "bwd_kv_rows_kernel",
        "specdec_bf16_hot": "bwd_kv_tc_kernel", "chunk_fp32_Q40": "bwd_kv_tiled_kernel",
        "mqa_fp16_D192": "bwd_kv_tc_kernel", "gqa_fp32_small_rows": "bwd_kv_kernel",
        "generic_bf16_D5_Dv7": "bwd_kv_kernel", "mha_fp16_Dv256": "bwd_kv_kernel",
        "rows_f16_D64_R8": "bwd_kv_rows_kernel", "rows_f32_D256_R16": "bwd_kv_rows_kernel",
        "rows_bf16_D256_R4_ragged": "bwd_kv_rows_kernel",
        "tiled_bf16_D128_R40_ragged": "bwd_kv_tc_kernel",
        "tiled_f16_D256_R32": "bwd_kv_tiled_kernel",
        "tiled_f32_D128_Dv64_R24": "bwd_kv_tiled_kernel",
        "tiled_bf16_D64_Dv192_R18": "bwd_kv_tc_kernel",
        "tiled_f16_D64_Dv128_R8": "bwd_kv_tiled_kernel",
        "tc_bf16_D64_R128_ragged": "bwd_kv_tc_kernel", "tc_f16_D128_R17": "bwd_kv_tc_kernel",
        "tc_bf16_D128_R32_hot": "bwd_kv_tc_kernel", "tc_bf16_D64_R64_staged": "bwd_kv_tc_kernel",
        "tc_f16_D128_R32_staged": "bwd_kv_tc_kernel",
        "dec_bf16_R16_tile_edge": "bwd_kv_tc_kernel", "dec_f16_D256_R8": "bwd_kv_tiled_kernel",
        "dec_bf16_D64_R4": "bwd_kv_kernel", "tc_walk_bf16_R32_units": "bwd_kv_tc_kernel",
        "tc_walk_f16_R64_D128": "bwd_kv_tc_kernel",
        "tc_bf16_R32_new_rows_in_whole_tile": "bwd_kv_tc_kernel"}

# the cases whose statistics pass runs the decode tensor-core kernel
DECODE_STATS = ("decode_bf16_ragged_M", "specdec_bf16_hot", "tiled_f16_D64_Dv128_R8",
                "dec_bf16_R16_tile_edge", "dec_f16_D256_R8", "dec_bf16_D64_R4",
                "tc_f16_D128_R17", "tc_bf16_D128_R32_hot", "tc_f16_D128_R32_staged",
                "tc_bf16_R32_new_rows_in_whole_tile")


def plan_of(spec):
    dims = kvc.make_dims(spec.B, spec.Hq, spec.Hk, spec.Q, spec.D, spec.Dv, spec.M,
                         workloads.DTYPES[spec.dtype])
    return kvc.backward_plan_info(dims)


def test_backward_plan():
    assert sorted(SLOT) == sorted(CASES)
    for name, spec in CASES.items():
        assert plan_of(spec)[2] == SLOT[name], name
    # the statistics pass: the tensor-core step where the tensor-core slot
    # kernel and the tensor-core step both take the shape (64-128 rows)
    assert plan_of(workloads.SPECS["long_mqa"]) == (7, "tensor", "bwd_kv_tc_kernel")
    assert plan_of(CASES["tc_bf16_D64_R128_ragged"])[:2] == (7, "tensor")
    assert plan_of(CASES["tiled_bf16_D128_R40_ragged"])[:2] == (6, "fused")
    assert plan_of(workloads.SPECS["chunked_append"]) == (6, "fused", "bwd_kv_tiled_kernel")
    # 16-bit, Dv = 128, at most 32 rows: the decode tensor-core kernel
    assert plan_of(workloads.SPECS["gqa_decode"]) == (6, "decode", "bwd_kv_rows_kernel")
    assert plan_of(workloads.SPECS["ragged_specdec"]) == (6, "decode", "bwd_kv_tc_kernel")
    for name in DECODE_STATS:
        assert plan_of(CASES[name])[1] == "decode", name
    assert plan_of(CASES["rows_f32_D256_R16"])[1] != "decode"   # fp32
    assert plan_of(CASES["rows_f16_D64_R8"])[1] != "decode"     # Dv = 64
    assert plan_of(workloads.SPECS["gqa_decode"].replace(Q=0))[0] == 2


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_backward_parity(name, seed):
    x = workloads.generate(CASES[name], seed)
    check(x, upstream(x, 100 + seed))
    check(x, upstream(x, 200 + seed, which=("attention", "context")))


@pytest.mark.parametrize("name", ["tc_f16_D128_R17", "tc_bf16_D64_R128_ragged", "rows_f16_D64_R8",
                                  "tiled_f16_D256_R32", "mha_fp16_Dv256", "tc_f16_D128_R32_staged"])
def test_backward_poisoned_tail(name):
    """Inf keys and NaN values from each row's new length on reach no gradient
    (every slot kernel reads only the slots below the new length)."""
    x = workloads.generate(CASES[name], 6)
    counts = x.append_mask.to(torch.int64).cumprod(1).sum(1)
    for b in range(x.key_cache.shape[0]):
        n_b = int(x.lengths[b]) + int(counts[b])
        x.key_cache[b, :, n_b:] = float("inf")
        x.value_cache[b, :, n_b:] = float("nan")
    check(x, upstream(x, 8))


@pytest.mark.parametrize("name", DECODE_STATS)
def test_backward_overwritten_slots_poisoned(name):
    """The statistics pass reads the inputs, whose caches still hold the old
    contents at the slots the new rows overwrite: Inf keys and NaN values
    there, and from the new length on, reach no gradient (the decode kernel
    replaces those slots' scores and value rows by the new rows')."""
    x = workloads.generate(CASES[name], 9)
    for b in range(x.key_cache.shape[0]):
        L = max(0, int(x.lengths[b]))
        x.key_cache[b, :, L:] = float("inf")
        x.value_cache[b, :, L:] = float("nan")
    check(x, upstream(x, 10))
    check(x, upstream(x, 11, which=("attention", "context")))


@pytest.mark.parametrize("which", [("context",), ("attention",), ("key_cache", "value_cache"),
                                   ()])
@pytest.mark.parametrize("name", ["specdec_bf16_hot", "tiled_bf16_D128_R40_ragged",
                                  "tiled_f16_D256_R32"])
def test_backward_partial_gradients(which, name):
    x = workloads.generate(CASES[name], 3)
    check(x, upstream(x, 7, which))


def test_backward_q0_and_nothing_appended():
    for spec in (Spec(B=3, Hq=4, Hk=2, Q=0, D=64, Dv=64, M=100, dtype="bf16"),
                 Spec(B=4, Hq=8, Hk=2, Q=3, D=128, Dv=128, M=300, dtype="bf16",
                      counts=("fixed", 0))):
        x = workloads.generate(spec, 1)
        check(x, upstream(x, 2))


def test_backward_contract_violations():
    spec = Spec(B=5, Hq=4, Hk=2, Q=3, D=64, Dv=64, M=200, dtype="bf16")
    x = workloads.generate(spec, 11)
    x.lengths = torch.tensor([10, 199, 250, -3, 40])
    m = workloads.prefix_mask([3, 3, 1, 1, 3], spec.Q)
    m[-1, 1] = False  # not a prefix
    x.append_mask = m
    check(x, upstream(x, 5), status_expect=kvc.DEV_MASK | kvc.DEV_OVERFLOW)


def test_backward_tc_walk_skips_flagged_rows():
    """Rows outside the contract (a non-prefix mask, a length past the
    capacity) hold no tile: the tensor-core kernel's walk over all units'
    tiles steps over them, and their caches pass the gradient straight through."""
    spec = CASES["tc_walk_bf16_R32_units"]
    x = workloads.generate(spec, 12)
    lengths = x.lengths.clone()
    lengths[3], lengths[17], lengths[18] = 699, -1, 0
    x.lengths = lengths
    m = x.append_mask.clone()
    m[3] = True                                        # 699 + 4 > M = 700
    m[5] = torch.tensor([True, False, True, False])   # not a prefix
    m[18] = False                                      # L = 0, nothing appended: no tile
    x.append_mask = m
    check(x, upstream(x, 13), status_expect=kvc.DEV_MASK | kvc.DEV_OVERFLOW)
    check(x, upstream(x, 14, which=("attention", "context")),
          status_expect=kvc.DEV_MASK | kvc.DEV_OVERFLOW)


def test_autograd_matches_oracle():
    """loss.backward() through kv_cache_attention_step gives the oracle's gradients."""
    x = workloads.generate(SMALL["decode_bf16_ragged_M"].replace(B=3, M=300), 4)
    grads = upstream(x, 9)
    xg = x.to(DEV)
    leaves = [t.clone().requires_grad_(True) for t in (xg.query, xg.new_key, xg.new_value,
                                                        xg.key_cache, xg.value_cache)]
    out = kvc.kv_cache_attention_step(*leaves, xg.lengths, xg.append_mask, xg.options)
    assert out["context"].requires_grad and not out["lengths"].requires_grad
    loss = sum((out[k].float() * grads[k].to(DEV).float()).sum()
               for k in ("key_cache", "value_cache", "attention", "context"))
    loss.backward()
    ref = oracle.step_backward(*x.args(), options=x.options,
                               **{f"d_{k}": v for k, v in grads.items()})
    check_grads({name: leaf.grad for name, leaf in zip(NAMES, leaves)}, ref, x, grads, "autograd")


def test_backward_decode_full_size_sampled():
    """gqa_decode sizes; the gradients of sampled batch rows against the oracle
    on the sub-batch they form (batch rows are independent)."""
    spec = workloads.SPECS["gqa_decode"]
    x = workloads.generate(spec, seed=1, device=DEV)
    grads = upstream(x, 12, which=("attention", "context"))
    grads = {k: (None if v is None else v.to(DEV)) for k, v in grads.items()}
    got = kvc.kv_cache_attention_step_backward(*x.args(), x.options,
                                               **{f"d_{k}": v for k, v in grads.items()})
    torch.cuda.synchronize()
    lengths = x.lengths.cpu().numpy()
    bsel = sorted({int(lengths.argmax()), int(lengths.argmin()), 7})
    idx = torch.tensor(bsel, device=DEV)
    sub = [t.index_select(0, idx).cpu() for t in x.args()]
    ref = oracle.step_backward(*sub, options=x.options,
                               **{f"d_{k}": (None if v is None else v.index_select(0, idx).cpu())
                                  for k, v in grads.items()})
    xs = workloads.StepInputs(*sub, x.options)
    gs = {k: (None if v is None else v.index_select(0, idx).cpu()) for k, v in grads.items()}
    terms = check_grads({k: v.index_select(0, idx) for k, v in got.items()}, ref, xs, gs, "sampled")
    check_mutants(ref, xs, xs.lengths, terms, "sampled")
    del got, x
    torch.cuda.empty_cache()


def test_backward_long_mqa_heads_sampled():
    """long_mqa's heads (128 query rows per KV head, D=192, Dv=128, fp16) over
    8192 slots, B=8: the tensor-core kernel over 64 tiles per unit, two per
    CTA (the query-gradient sums kept across a CTA's tiles); the longest
    batch row against the oracle (the oracle takes about a minute per batch
    row at long_mqa's full 65536 slots)."""
    spec = workloads.SPECS["long_mqa"].replace(M=8192, lengths=("uniform", 7000, 8184))
    x = workloads.generate(spec, seed=2, device=DEV)
    grads = upstream(x, 13, which=("attention", "context"))
    grads = {k: (None if v is None else v.to(DEV)) for k, v in grads.items()}
    got = kvc.kv_cache_attention_step_backward(*x.args(), x.options,
                                               **{f"d_{k}": v for k, v in grads.items()})
    torch.cuda.synchronize()
    idx = torch.tensor([int(x.lengths.cpu().argmax())], device=DEV)
    sub = [t.index_select(0, idx).cpu() for t in x.args()]
    ref = oracle.step_backward(*sub, options=x.options,
                               **{f"d_{k}": (None if v is None else v.index_select(0, idx).cpu())
                                  for k, v in grads.items()})
    xs = workloads.StepInputs(*sub, x.options)
    gs = {k: (None if v is None else v.index_select(0, idx).cpu()) for k, v in grads.items()}
    terms = check_grads({k: v.index_select(0, idx) for k, v in got.items()}, ref, xs, gs, "sampled")
    check_mutants(ref, xs, xs.lengths, terms, "sampled")
    del got, x
    torch.cuda.empty_cache()
