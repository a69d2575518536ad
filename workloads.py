"""Seeded synthetic inputs for the KV-cache append + causal attention step.

This module only draws tensors: shapes, value distributions, length mixes and
append counts of the step's workloads. It holds none of the step's arithmetic,
and both sides of every parity check (the CUDA library and the fp64 oracle)
take their inputs from here.

Workloads (sizes as named; "N(0, s)" means a normal with standard deviation s):

* ``tiny_fp32``       B=2 Hq=4 Hk=2 Q=3 D=Dv=16 M=32 fp32; length ~ U{0..M-Q};
                      the row's append count n ~ U{0..3}; N(0,1) everywhere,
                      including the cache tail; default scale.
* ``gqa_decode``      B=64 Hq=32 Hk=8 Q=1 D=Dv=128 M=8192 bf16 (a Llama-3-8B-like
                      decode batch); length ~ U{1024..8191}; all-True masks.
* ``chunked_append``  B=2 Hq=8 Hk=2 D=Dv=64 M=4096, bf16 or fp32; initial length
                      ~ U{100..2000}; three chained steps with Q = 40, 32, 24 and
                      all-True masks, each step consuming the previous outputs.
* ``ragged_specdec``  B=256 Hq=32 Hk=8 Q=4 D=Dv=128 M=16384 bf16; length =
                      min(Zipf(1.2), M-4); n ~ U{0..4}; N(0,1) with 1% of the
                      (b, h, t) query rows scaled by 50 (raw dots above 1000).
* ``long_mqa``        B=8 Hq=16 Hk=1 Q=8 D=192 Dv=128 M=65536 fp16; length ~
                      U{60000..65528}; all-True masks; N(0, 0.5); scale 0.05.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass
class Spec:
    B: int
    Hq: int
    Hk: int
    Q: int
    D: int
    Dv: int
    M: int
    dtype: str = "bf16"
    # lengths: ("uniform", lo, hi) inclusive, or ("zipf", a) clipped to [0, M-Q],
    # or ("fixed", value)
    lengths: tuple = ("uniform", 0, None)
    # append counts: ("all",) = Q, ("uniform", lo, hi) inclusive, ("fixed", n)
    counts: tuple = ("all",)
    std: float = 1.0
    hot_frac: float = 0.0     # fraction of (b, h, t) query rows scaled by hot_scale
    hot_scale: float = 1.0
    scale: Optional[float] = None   # None = the step's default 1/sqrt(D)

    def replace(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


SPECS = {
    "tiny_fp32": Spec(B=2, Hq=4, Hk=2, Q=3, D=16, Dv=16, M=32, dtype="f32",
                      lengths=("uniform", 0, 29), counts=("uniform", 0, 3)),
    "gqa_decode": Spec(B=64, Hq=32, Hk=8, Q=1, D=128, Dv=128, M=8192, dtype="bf16",
                       lengths=("uniform", 1024, 8191), counts=("all",)),
    "chunked_append": Spec(B=2, Hq=8, Hk=2, Q=40, D=64, Dv=64, M=4096, dtype="bf16",
                           lengths=("uniform", 100, 2000), counts=("all",)),
    "ragged_specdec": Spec(B=256, Hq=32, Hk=8, Q=4, D=128, Dv=128, M=16384, dtype="bf16",
                           lengths=("zipf", 1.2), counts=("uniform", 0, 4),
                           hot_frac=0.01, hot_scale=50.0),
    "long_mqa": Spec(B=8, Hq=16, Hk=1, Q=8, D=192, Dv=128, M=65536, dtype="f16",
                     lengths=("uniform", 60000, 65528), counts=("all",), std=0.5, scale=0.05),
}
CHUNKS = (40, 32, 24)   # chained append sizes of ``chunked_append``


@dataclasses.dataclass
class StepInputs:
    query: torch.Tensor
    new_key: torch.Tensor
    new_value: torch.Tensor
    key_cache: torch.Tensor
    value_cache: torch.Tensor
    lengths: torch.Tensor
    append_mask: torch.Tensor
    options: dict

    def args(self):
        return (self.query, self.new_key, self.new_value, self.key_cache, self.value_cache,
                self.lengths, self.append_mask)

    def to(self, device) -> "StepInputs":
        return StepInputs(*(t.to(device) for t in self.args()), options=dict(self.options))


def _draw_lengths(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    kind = spec.lengths[0]
    hi_cap = spec.M - spec.Q
    if kind == "uniform":
        lo, hi = spec.lengths[1], spec.lengths[2]
        hi = hi_cap if hi is None else hi
        return rng.integers(lo, hi + 1, size=spec.B, dtype=np.int64)
    if kind == "zipf":
        k = rng.zipf(spec.lengths[1], size=spec.B).astype(np.int64)
        return np.clip(k, 0, hi_cap)
    if kind == "fixed":
        return np.full(spec.B, spec.lengths[1], dtype=np.int64)
    raise ValueError(kind)


def _draw_counts(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    kind = spec.counts[0]
    if kind == "all":
        return np.full(spec.B, spec.Q, dtype=np.int64)
    if kind == "uniform":
        return rng.integers(spec.counts[1], spec.counts[2] + 1, size=spec.B, dtype=np.int64)
    if kind == "fixed":
        return np.full(spec.B, spec.counts[1], dtype=np.int64)
    raise ValueError(kind)


def prefix_mask(counts: Sequence[int], Q: int) -> torch.Tensor:
    """Bool [B, Q] whose row b is counts[b] True values followed by False."""
    c = torch.as_tensor(np.asarray(counts, dtype=np.int64))
    return torch.arange(Q)[None, :] < c[:, None]


def _normal(shape, std, dtype, gen, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(DTYPES[dtype])


def generate(spec: Spec, seed: int, device="cpu", Q: Optional[int] = None) -> StepInputs:
    """Draw one step's inputs. Large tensors come from a torch generator on
    ``device`` (seeded), small integer draws from numpy's PCG64 (seeded)."""
    if Q is not None:
        spec = spec.replace(Q=Q)
    device = torch.device(device)
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B, Hq, Hk, Q, D, Dv, M = spec.B, spec.Hq, spec.Hk, spec.Q, spec.D, spec.Dv, spec.M
    lengths = _draw_lengths(spec, rng)
    counts = np.minimum(_draw_counts(spec, rng), spec.Q)
    key_cache = _normal((B, Hk, M, D), spec.std, spec.dtype, gen, device)
    value_cache = _normal((B, Hk, M, Dv), spec.std, spec.dtype, gen, device)
    query = _normal((B, Hq, Q, D), spec.std, spec.dtype, gen, device)
    new_key = _normal((B, Hk, Q, D), spec.std, spec.dtype, gen, device)
    new_value = _normal((B, Hk, Q, Dv), spec.std, spec.dtype, gen, device)
    if spec.hot_frac > 0 and Q > 0:
        hot = torch.as_tensor(rng.random((B, Hq, Q)) < spec.hot_frac)
        factor = torch.where(hot, spec.hot_scale, 1.0).to(device=device, dtype=torch.float32)
        query = (query.float() * factor[..., None]).to(DTYPES[spec.dtype])
    options = {} if spec.scale is None else {"scale": float(spec.scale)}
    return StepInputs(query, new_key, new_value, key_cache, value_cache,
                      torch.as_tensor(lengths).to(device),
                      prefix_mask(counts, Q).to(device), options)


def chain_chunks(spec: Spec, seed: int, device="cpu", chunks=CHUNKS):
    """Inputs for chained multi-token appends: the first step's full inputs
    (Q = chunks[0]), then per later step (query, new_key, new_value, mask)
    drawn with its own Q. Each later step consumes the previous outputs."""
    first = generate(spec, seed, device, Q=chunks[0])
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed + 1000)
    rest = []
    for q in chunks[1:]:
        s = spec.replace(Q=q)
        rest.append((
            _normal((s.B, s.Hq, q, s.D), s.std, s.dtype, gen, device),
            _normal((s.B, s.Hk, q, s.D), s.std, s.dtype, gen, device),
            _normal((s.B, s.Hk, q, s.Dv), s.std, s.dtype, gen, device),
            prefix_mask(np.full(s.B, q), q).to(device),
        ))
    return first, rest
