"""bench.py's byte and flop model (the numerator of every reported GB/s and
roofline fraction) against independent counts on small seeded inputs.

The out-of-place step's algorithmic bytes are, by their definition, every
input read once and every output written once: the sum of the tensors'
sizes. The steps that copy no cache move the valid prefix of each KV head
(the new length N_b = L_b + n_b slots, "Required behavior": query t sees
slots j <= L_b + t) instead of the whole cache; the backward's arithmetic is
4 (D + Dv) flops for every allowed (query row, slot) pair. Here the prefixes
and pairs are enumerated slot by slot from the mask's leading True entries.
"""
import pytest
import torch

import bench
import workloads
from workloads import Spec

SPECS = [
    workloads.SPECS["tiny_fp32"],
    Spec(B=3, Hq=8, Hk=2, Q=4, D=64, Dv=32, M=50, dtype="bf16", counts=("uniform", 0, 4)),
    Spec(B=2, Hq=6, Hk=3, Q=2, D=16, Dv=48, M=20, dtype="f16", lengths=("uniform", 0, 18)),
]


def nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def appended(x) -> list:
    """n_b: the leading True entries of each mask row."""
    return [int(v) for v in x.append_mask.to(torch.int64).cumprod(1).sum(1)]


@pytest.mark.parametrize("i", range(len(SPECS)))
def test_out_of_place_bytes_are_every_tensor_once(i):
    spec = SPECS[i]
    x = workloads.generate(spec, seed=i)
    B, Hq, Q, _ = x.query.shape
    es = x.key_cache.element_size()
    inputs = sum(nbytes(t) for t in (x.query, x.new_key, x.new_value, x.key_cache,
                                      x.value_cache, x.lengths))
    inputs += B * Q  # the mask, one byte per entry
    outputs = (nbytes(x.key_cache) + nbytes(x.value_cache) + nbytes(x.lengths)
               + B * Hq * Q * spec.M * es + B * Hq * Q * spec.Dv * es)
    model = bench.algorithmic_bytes(spec)
    assert model["total"] == inputs + outputs
    assert model["fused_kernel"] + model["finalize_kernel"] == model["total"]


@pytest.mark.parametrize("i", range(len(SPECS)))
def test_inplace_bytes_count_the_valid_prefix_slot_by_slot(i):
    spec = SPECS[i]
    x = workloads.generate(spec, seed=10 + i)
    es = x.key_cache.element_size()
    n = appended(x)
    prefix = appended_rows = 0
    for b in range(spec.B):
        N = int(x.lengths[b]) + n[b]
        for k in range(spec.Hk):
            for j in range(N):
                prefix += (spec.D + spec.Dv) * es       # K and V rows read
                if j >= int(x.lengths[b]):
                    appended_rows += (spec.D + spec.Dv) * es  # new rows written in place
    others = (nbytes(x.query) + nbytes(x.new_key) + nbytes(x.new_value) + 2 * nbytes(x.lengths)
              + spec.B * spec.Q + spec.B * spec.Hq * spec.Q * (spec.M + spec.Dv) * es)
    model = bench.algorithmic_bytes_inplace(spec, x.lengths.tolist(), n)
    assert model["total"] == prefix + appended_rows + others


@pytest.mark.parametrize("i", range(len(SPECS)))
def test_backward_flops_enumerate_the_allowed_pairs(i):
    spec = SPECS[i]
    x = workloads.generate(spec, seed=20 + i)
    n = appended(x)
    pairs = 0
    for b in range(spec.B):
        L = int(x.lengths[b])
        for h in range(spec.Hq):
            for t in range(n[b]):           # valid query rows
                for j in range(spec.M):
                    if j <= L + t:          # the lower-right causal rule
                        pairs += 1
    assert bench.flops_backward(spec, x.lengths.tolist(), n) == 4 * (spec.D + spec.Dv) * pairs


@pytest.mark.parametrize("i", range(len(SPECS)))
def test_backward_bytes_split_at_the_new_length(i):
    """The slot kernel's share and the tail copy's share cover every cache
    slot once: below N_b the prefix, both gradient tensors and the allowed
    attention gradients; from N_b on the gradient read and write."""
    spec = SPECS[i]
    x = workloads.generate(spec, seed=30 + i)
    es = x.key_cache.element_size()
    n = appended(x)
    row = spec.Hk * (spec.D + spec.Dv) * es
    below = tail = allowed = 0
    for b in range(spec.B):
        L = int(x.lengths[b])
        N = L + n[b]
        for j in range(spec.M):
            if j < N:
                below += 3 * row        # prefix read, returned gradient read, gradient written
            else:
                tail += 2 * row         # returned gradient read, gradient written
        allowed += spec.Hq * sum(L + t + 1 for t in range(n[b]))
    qrows = spec.B * spec.Hq * spec.Q
    model = bench.algorithmic_bytes_backward(spec, x.lengths.tolist(), n)
    assert model["bwd_copy_kernel"] == tail
    assert model["bwd_kv_kernel"] == below + allowed * es + qrows * (spec.D + spec.Dv) * es


def test_traffic_keys_separate_token_and_dtype_overrides():
    """A kernel's DRAM traffic is recorded per workload face; the attention rows
    a step writes grow with Q, so a capture taken at the workload's own Q must
    not be scaled onto a run with another Q (or dtype)."""
    import argparse

    def args(**kw):
        base = dict(backward=False, readonly=False, paged=None, inplace=False,
                    workload="gqa_decode", q=None, dtype=None)
        base.update(kw)
        return argparse.Namespace(**base)

    assert bench.mode_key(args()) == "gqa_decode"
    assert bench.mode_key(args(inplace=True)) == "inplace:gqa_decode"
    assert bench.mode_key(args(paged=16)) == "paged16:gqa_decode"
    assert bench.mode_key(args(inplace=True, q=8)) == "inplace:gqa_decode:Q8"
    assert bench.mode_key(args(workload="chunked_append", dtype="f32")) == "chunked_append:f32"
    keys = {bench.mode_key(args(**kw)) for kw in
            ({}, {"q": 8}, {"dtype": "f16"}, {"inplace": True}, {"inplace": True, "q": 8},
             {"readonly": True}, {"backward": True}, {"paged": 64})}
    assert len(keys) == 8
