"""GPU parity of the decode tensor-core kernel (kvc_decode_tc.cu) against the
fp64 oracle: steps that copy no cache (in place, paged, read-only) with 16-bit
caches, D a multiple of 64 up to 256, Dv = 128 and at most 32 query rows per
KV head. The caches after the step bit for bit, lengths exact, attention and
context within the step's tolerances. Shapes cover every row count the kernel
is instantiated for, tiles cut by M and by the new length, many chunks per
unit, hot scores that raise a row's reference maximum in the middle of a
chunk, and Inf/NaN past the new length.
"""
import pytest
import torch

import kv_cache_append_gb300 as kvc
import workloads
from test_gpu_inplace import run_inplace
from test_gpu_paged import compare_paged, run_paged
from test_gpu_parity import (DEV, _built, check_append_property, compare_batch_rows,  # noqa: F401
                             compare_full)
from workloads import Spec

pytestmark = pytest.mark.gpu


def path_of(spec):
    x = workloads.generate(spec, 0).to(DEV)
    dims = kvc.dims_of(x.query, x.key_cache, x.value_cache)
    return kvc.plan_info_inplace(dims, x.key_cache, x.value_cache, x.new_key, x.new_value)[1]


CASES = {
    # rows per unit R = (Hq / Hk) * Q
    "r1_mha_bf16": Spec(B=3, Hq=4, Hk=4, Q=1, D=128, Dv=128, M=300, dtype="bf16"),
    "r2_f16_M129": Spec(B=4, Hq=4, Hk=2, Q=1, D=64, Dv=128, M=129, dtype="f16",
                        lengths=("uniform", 0, 128)),
    "r3_bf16_D192": Spec(B=2, Hq=6, Hk=2, Q=1, D=192, Dv=128, M=500, dtype="bf16"),
    "r4_bf16_D256": Spec(B=3, Hq=8, Hk=2, Q=1, D=256, Dv=128, M=640, dtype="bf16",
                         lengths=("uniform", 100, 639)),
    "r5_f16_ragged": Spec(B=3, Hq=10, Hk=2, Q=1, D=128, Dv=128, M=1000, dtype="f16",
                          lengths=("uniform", 0, 999)),
    "r8_bf16_Q2": Spec(B=4, Hq=8, Hk=2, Q=2, D=128, Dv=128, M=777, dtype="bf16",
                       counts=("uniform", 0, 2)),
    "r12_f16_Q3_D64": Spec(B=3, Hq=8, Hk=2, Q=3, D=64, Dv=128, M=400, dtype="f16",
                           counts=("uniform", 0, 3)),
    "r16_bf16_Q4_hot": Spec(B=4, Hq=8, Hk=2, Q=4, D=128, Dv=128, M=1500, dtype="bf16",
                            lengths=("uniform", 200, 1490), hot_frac=0.05, hot_scale=50.0),
    "r16_f16_Q16_mqa": Spec(B=2, Hq=1, Hk=1, Q=16, D=128, Dv=128, M=600, dtype="f16",
                            counts=("uniform", 1, 16)),
    # 17 to 32 rows: two groups of 16 padded rows, the second one partly empty
    "r24_bf16_Q3": Spec(B=3, Hq=8, Hk=1, Q=3, D=128, Dv=128, M=700, dtype="bf16",
                        counts=("uniform", 0, 3)),
    "r20_f16_Q5_D64": Spec(B=2, Hq=4, Hk=1, Q=5, D=64, Dv=128, M=333, dtype="f16",
                           lengths=("uniform", 0, 300)),
    "r32_bf16_Q4_hot": Spec(B=3, Hq=32, Hk=4, Q=4, D=128, Dv=128, M=1300, dtype="bf16",
                            lengths=("uniform", 100, 1290), hot_frac=0.05, hot_scale=50.0),
    "r32_f16_Q8_D192": Spec(B=2, Hq=4, Hk=1, Q=8, D=192, Dv=128, M=500, dtype="f16",
                            counts=("uniform", 1, 8)),
    # one unit, many chunks (one tile each at 152 CTAs), a hot slot late in the row
    "r4_bf16_long_row": Spec(B=1, Hq=4, Hk=1, Q=1, D=128, Dv=128, M=20000, dtype="bf16",
                             lengths=("uniform", 19000, 19990), hot_frac=0.5, hot_scale=40.0),
    # lengths at tile edges: the new length lands on 127, 128, 129 ... in turn
    "r4_bf16_edges": Spec(B=8, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=384, dtype="bf16",
                          lengths=("uniform", 126, 130)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_tc_path_taken(name):
    assert path_of(CASES[name]) == "decode_tc"


def test_decode_tc_not_taken_outside_its_shapes():
    assert path_of(Spec(B=2, Hq=8, Hk=2, Q=1, D=128, Dv=128, M=100, dtype="f32")) == "fused"
    assert path_of(Spec(B=2, Hq=8, Hk=2, Q=1, D=128, Dv=64, M=100, dtype="bf16")) == "fused"
    # 40 rows: the tensor-core step (from 9 rows), 16-bit with widths it takes
    assert path_of(Spec(B=2, Hq=8, Hk=1, Q=5, D=128, Dv=128, M=100, dtype="bf16")) == "tensor"
    assert path_of(Spec(B=2, Hq=8, Hk=2, Q=1, D=96, Dv=128, M=100, dtype="bf16")) == "fused"
    # 17 to 32 rows with D = 256: two stages of 32 padded rows overflow shared memory
    assert path_of(Spec(B=2, Hq=4, Hk=1, Q=8, D=256, Dv=128, M=100, dtype="f16")) == "tensor"


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_decode_tc_inplace_parity(name, seed):
    x = workloads.generate(CASES[name], seed)
    out, status = run_inplace(x.to(DEV))
    compare_full(x, out, status)


@pytest.mark.parametrize("name", ["r4_bf16_D256", "r16_bf16_Q4_hot", "r5_f16_ragged",
                                  "r32_bf16_Q4_hot"])
def test_decode_tc_poisoned_tail(name):
    """Inf keys and NaN values from each row's new length on reach nothing."""
    x = workloads.generate(CASES[name], 3)
    counts = x.append_mask.to(torch.int64).sum(1)
    for b in range(x.key_cache.shape[0]):
        n_b = int(x.lengths[b]) + int(counts[b])
        x.key_cache[b, :, n_b:] = float("inf")
        x.value_cache[b, :, n_b:] = float("nan")
    out, status = run_inplace(x.to(DEV))
    compare_full(x, out, status)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("name", ["r4_bf16_D256", "r16_bf16_Q4_hot", "r24_bf16_Q3"])
def test_decode_tc_paged(name, bs):
    spec = CASES[name]
    M = (spec.M + bs - 1) // bs * bs
    spec = spec.replace(M=M)
    assert path_of(spec) == "decode_tc"
    x = workloads.generate(spec, 9)
    out, status, ref, table = run_paged(x, bs, seed=bs)
    compare_paged(x, out, status, ref, table=table)


def test_decode_tc_multi_tile_chunks_hot_rows():
    """gqa_decode sizes (several tiles per chunk) with hot query rows, whose
    reference maximum is raised, and O^T rescaled, in the middle of chunks;
    sampled batch rows against the oracle."""
    spec = workloads.SPECS["gqa_decode"].replace(hot_frac=0.1, hot_scale=50.0)
    x = workloads.generate(spec, seed=4, device=DEV)
    out, status = run_inplace(x)
    assert status == 0
    check_append_property(x, out)
    lengths = x.lengths.cpu().numpy()
    compare_batch_rows(x, out, {int(lengths.argmax()), int(lengths.argmin()), 5, 17})
    del out, x
    torch.cuda.empty_cache()
