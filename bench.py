"""Benchmark of the KV-cache append + causal attention step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload gqa_decode|ragged_specdec|long_mqa|chunked_append|tiny_fp32]

One step = one kvc_step over one batch of the workload: copy + scatter of
both caches, attention partials, split combine, attention rows and context.
Inputs are seeded synthetic tensors (workloads.py) resident in HBM before the
timed region; the caches alone are far larger than the 129 MB L2, so no L2
flush is needed between steps. Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "effective HBM GB/s (and % of 8 TB/s) + kv steps/s per config, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# CUDA-core fp32 peak: 152 SMs x 128 FP32 lanes x 2 flops per FMA x 2070 MHz
# (the maximum SM clock); the roofline of the backward's slot kernel when its
# products, not its bytes, bound it
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
_CSRC = "kv_cache_append_gb300/csrc/"
# The first kernel of each path and the sources that define it.
STEP_KERNEL = {"fused": "fused_step_kernel", "tensor": "tc_step_kernel",
               "tensor_2pass": "tc_step_kernel",
               "decode_tc": "decode_tc_kernel", "generic": "generic_copy_kernel"}
# Every kernel of a step with query rows, in launch order (in place: the
# cache write comes first and the generic path has no copy kernel).
PATH_KERNELS_INPLACE = {
    "fused": ["inplace_rows_kernel", "fused_step_kernel", "finalize_merge_kernel",
              "finalize_rows_kernel"],
    "tensor": ["inplace_rows_kernel", "tc_step_kernel", "finalize_merge_kernel",
               "finalize_rows_kernel"],
    "decode_tc": ["inplace_rows_kernel", "decode_tc_kernel", "finalize_merge_kernel",
                  "finalize_rows_kernel"],
    "generic": ["inplace_rows_kernel", "generic_attend_kernel", "finalize_merge_kernel",
                "finalize_rows_kernel"]}
PATH_KERNELS_PAGED = {
    path: ["paged_prep_kernel"] + PATH_KERNELS_INPLACE[path] for path in PATH_KERNELS_INPLACE}
PATH_KERNELS_READONLY = {
    path: ["attend_prep_kernel", STEP_KERNEL[path] if path != "generic" else "generic_attend_kernel",
           "finalize_merge_kernel", "attend_unpack_kernel"]
    for path in ("fused", "tensor", "decode_tc", "generic")}
# the backward: the statistics pass (step kernel and merge with no copy, or the tensor-core
# step with its row writer), then its own four; kvc_backward_plan_info names the path and
# the slot kernel ("bwd_kv_kernel" below stands for it)
PATH_KERNELS_BACKWARD = {
    path: first + ["bwd_rowdot_kernel", "bwd_kv_kernel", "bwd_copy_kernel", "bwd_dq_kernel"]
    for path, first in (("fused", ["fused_step_kernel", "finalize_merge_kernel"]),
                        ("decode", ["decode_tc_kernel", "finalize_merge_kernel"]),
                        ("generic", ["generic_attend_kernel", "finalize_merge_kernel"]),
                        ("tensor", ["tc_step_kernel", "finalize_merge_kernel",
                                    "finalize_rows_kernel"]))}


PATH_KERNELS = {"fused": ["fused_step_kernel", "finalize_merge_kernel", "finalize_rows_kernel"],
                "tensor": ["tc_step_kernel", "finalize_merge_kernel", "finalize_rows_kernel"],
                # two passes: the step kernel writes the attention rows itself
                "tensor_2pass": ["tc_step_kernel", "finalize_merge_kernel"],
                "generic": ["generic_copy_kernel", "generic_attend_kernel",
                            "finalize_merge_kernel", "finalize_rows_kernel"]}
KERNEL_SOURCES = {
    "fused_step_kernel": [_CSRC + f for f in ("kvc_fused.cu", "kvc_internal.cuh",
                                              "kvc_pipeline.cuh")],
    "tc_step_kernel": [_CSRC + f for f in ("kvc_fused_tc.cu", "kvc_internal.cuh",
                                           "kvc_pipeline.cuh", "kvc_tcgen05.cuh")],
    "decode_tc_kernel": [_CSRC + f for f in ("kvc_decode_tc.cu", "kvc_internal.cuh",
                                             "kvc_pipeline.cuh", "kvc_tcgen05.cuh")],
    "bwd_kv_kernel": [_CSRC + f for f in ("kvc_backward.cu", "kvc_internal.cuh")],
    "bwd_kv_rows_kernel": [_CSRC + f for f in ("kvc_backward.cu", "kvc_internal.cuh")],
    "bwd_kv_tiled_kernel": [_CSRC + f for f in ("kvc_backward_tiled.cu", "kvc_internal.cuh")],
    "bwd_kv_tc_kernel": [_CSRC + f for f in ("kvc_backward_tc.cu", "kvc_internal.cuh",
                                             "kvc_tcgen05.cuh")],
    "bwd_copy_kernel": [_CSRC + f for f in ("kvc_backward.cu", "kvc_internal.cuh")],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")


# ----------------------------------------------------------------- bytes model
def algorithmic_bytes(spec: workloads.Spec, batch_rows: int | None = None) -> dict:
    """Bytes the step must move at minimum: full cache read + write, the
    attention and context writes, the query / new key / new value reads,
    lengths and mask (read) and lengths (write)."""
    B = spec.B if batch_rows is None else batch_rows
    es = 4 if spec.dtype == "f32" else 2
    cache = B * spec.Hk * spec.M * (spec.D + spec.Dv) * es
    qkv = (B * spec.Hq * spec.Q * spec.D + B * spec.Hk * spec.Q * (spec.D + spec.Dv)) * es
    small = B * 8 * 2 + B * spec.Q
    att = B * spec.Hq * spec.Q * spec.M * es
    ctx = B * spec.Hq * spec.Q * spec.Dv * es
    fused = 2 * cache + qkv + small
    return {"total": fused + att + ctx, "fused_kernel": fused, "finalize_kernel": att + ctx,
            "attention": att}


def step_kernel_bytes(nbytes: dict, path: str) -> int:
    """Algorithmic bytes of the step kernel: the copy and its inputs, plus the
    attention rows where the step kernel writes them (the two-pass form)."""
    return nbytes["fused_kernel"] + (nbytes.get("attention", 0) if path == "tensor_2pass" else 0)


def algorithmic_bytes_inplace(spec: workloads.Spec, lengths, counts) -> dict:
    """Bytes the in-place step must move at minimum: the valid prefix of both
    caches read (new length N_b = L_b + n_b slots per KV head), the appended
    rows written, query / new rows / lengths / mask read, attention and
    context written. ``lengths``/``counts`` are the batch rows' L_b and n_b."""
    es = 4 if spec.dtype == "f32" else 2
    B = len(lengths)
    row = spec.Hk * (spec.D + spec.Dv) * es
    N = int(sum(lengths)) + int(sum(counts))
    prefix = N * row
    appended = int(sum(counts)) * row
    qkv = (B * spec.Hq * spec.Q * spec.D + B * spec.Hk * spec.Q * (spec.D + spec.Dv)) * es
    small = B * 8 * 2 + B * spec.Q
    att = B * spec.Hq * spec.Q * spec.M * es
    ctx = B * spec.Hq * spec.Q * spec.Dv * es
    step = prefix + qkv + small
    return {"total": step + appended + att + ctx, "fused_kernel": step,
            "finalize_kernel": att + ctx}


def algorithmic_bytes_readonly(spec: workloads.Spec, lengths, counts) -> dict:
    """Bytes the read-only re-attention must move at minimum: each sequence's
    cached prefix (K_b = L_b + n_b slots per KV head) read, its n_b packed
    query rows read and output rows written, and the per-sequence offsets,
    lengths and slots."""
    es = 4 if spec.dtype == "f32" else 2
    B = len(lengths)
    K = int(sum(lengths)) + int(sum(counts))
    tq = int(sum(counts))
    prefix = K * spec.Hk * (spec.D + spec.Dv) * es
    step = prefix + tq * spec.Hq * spec.D * es + (B + 1) * 4 + B * 8
    out = tq * spec.Hq * spec.Dv * es
    return {"total": step + out, "fused_kernel": prefix + tq * spec.Hq * spec.D * es,
            "finalize_kernel": out}


def algorithmic_bytes_backward(spec: workloads.Spec, lengths, counts) -> dict:
    """Bytes the step's backward must move at minimum, all four upstream
    gradients given: the returned caches' gradient read and the caches'
    gradient written in full; the valid prefix of both caches (N_b = L_b + n_b
    slots per KV head) read; the attention gradient on the allowed slots, the
    context gradient and the query read; the query and new-row gradients
    written, the new rows read. Per kernel: bwd_kv_kernel covers the slots
    below the new length (prefix, the two cache gradients there, the
    attention gradient, query and context gradient rows), bwd_copy_kernel the
    slots from it on (cache gradients read and written)."""
    es = 4 if spec.dtype == "f32" else 2
    B = len(lengths)
    row = spec.Hk * (spec.D + spec.Dv) * es
    N = [int(l) + int(c) for l, c in zip(lengths, counts)]
    allowed = sum(spec.Hq * sum(int(l) + t + 1 for t in range(int(c)))
                  for l, c in zip(lengths, counts))
    qrows = B * spec.Hq * spec.Q
    kv = sum(N) * row * 3 + allowed * es + qrows * (spec.D + spec.Dv) * es
    copy = sum(spec.M - n for n in N) * row * 2
    rest = qrows * spec.D * es + 2 * B * spec.Hk * spec.Q * (spec.D + spec.Dv) * es + B * (16 + spec.Q)
    return {"total": kv + copy + rest, "bwd_kv_kernel": kv, "bwd_copy_kernel": copy}


def flops_backward(spec: workloads.Spec, lengths, counts) -> int:
    """Arithmetic of the backward's slot kernel: for every allowed (query row,
    slot) pair, dcontext . V'_j (2 Dv flops), ds q into dK'_j (2 D), a dcontext
    into dV'_j (2 Dv) and ds K'_j into dq (2 D)."""
    allowed = sum(spec.Hq * sum(int(l) + t + 1 for t in range(int(c)))
                  for l, c in zip(lengths, counts))
    return 4 * (spec.D + spec.Dv) * allowed


def source_digest(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def mode_key(args) -> str:
    """Key of a workload and step face in the traffic record, e.g.
    "gqa_decode", "inplace:gqa_decode", "paged64:gqa_decode", and with a
    token or dtype override "inplace:gqa_decode:Q8" (the attention rows a
    step writes grow with Q, so a capture holds for its own Q only)."""
    mode = ("backward" if args.backward else "readonly" if args.readonly else
            f"paged{args.paged}" if args.paged else "inplace" if args.inplace else "")
    key = f"{mode}:{args.workload}" if mode else args.workload
    if args.q is not None:
        key += f":Q{args.q}"
    if args.dtype is not None:
        key += f":{args.dtype}"
    return key


def kernel_traffic(key: str, kernel: str, algorithmic: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary for
    `key`, scaled from the captured launch to this one by their algorithmic
    bytes, if the capture was taken on the kernel's current source; else None."""
    if kernel not in KERNEL_SOURCES:
        return None
    try:
        with open(TRAFFIC_FILE) as f:
            entry = json.load(f)["workloads"][key]
        cap = entry["captured"]
    except Exception:
        return None
    if entry.get("kernel") != kernel or \
            entry.get("kernel_source_sha256") != source_digest(KERNEL_SOURCES[kernel]):
        return None
    return round(float(cap["dram_bytes"]) * algorithmic / float(cap["algorithmic_bytes"]))


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.t:
            self.t.join(timeout=5)

    def summary(self, t0, t1):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = [s for (ts, s) in self.samples if len(s) >= 9]
        window = [s for (ts, s) in self.samples if t0 - 0.25 <= ts <= t1 + 0.25 and len(s) >= 9]
        busy = [s for s in rows if _num(s[4]) and _num(s[4]) >= 50]
        use = window if window else busy
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [_num(s[1]) for s in use if _num(s[1])]
        reasons = sorted({names[i] for s in use for i in range(4) if s[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": _num(use[0][2]), "reasons": reasons, "samples": len(use),
                "window": "timed region" if window else "busy samples (timed region < 200 ms)",
                "power_w_max": max((_num(s[3]) or 0.0) for s in use)}


def _num(x):
    try:
        return float(x)
    except Exception:
        return None


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle leg
def backward_grads(spec, x, seed, device):
    """Seeded upstream gradients of the four outputs, in the inputs' dtype."""
    g = torch.Generator(device=device).manual_seed(seed)
    B, Hq, Q, _ = x.query.shape
    M, Dv = x.key_cache.shape[2], x.value_cache.shape[-1]
    dt = x.query.dtype
    return {"key_cache": torch.randn(tuple(x.key_cache.shape), generator=g, device=device).to(dt),
            "value_cache": torch.randn(tuple(x.value_cache.shape), generator=g,
                                       device=device).to(dt),
            "attention": torch.randn(B, Hq, Q, M, generator=g, device=device).to(dt),
            "context": torch.randn(B, Hq, Q, Dv, generator=g, device=device).to(dt)}


def oracle_call(x_cpu, k: int, backward: bool, grads=None):
    """One oracle step (or its backward) on the first k batch rows."""
    import oracle
    sub = [t[:k] for t in x_cpu.args()]
    if backward:
        return oracle.step_backward(*sub, options=x_cpu.options,
                                    **{f"d_{n}": g[:k] for n, g in grads.items()})
    return oracle.step(*sub, x_cpu.options)


def oracle_sample(spec: workloads.Spec, x_cpu: workloads.StepInputs, budget_s: float,
                  backward: bool = False):
    """Time the fp64 oracle on the first k batch rows, k grown until the run
    takes about budget_s. Returns (seconds, rows, threads)."""
    import oracle
    oracle.build()
    grads = backward_grads(spec, x_cpu, 5, "cpu") if backward else None
    k = 1
    while True:
        t0 = time.perf_counter()
        oracle_call(x_cpu, k, backward, grads)
        dt = time.perf_counter() - t0
        if dt >= budget_s or k >= spec.B:
            return dt, k, oracle.threads()
        grow = max(2, int(math.ceil(budget_s / max(dt, 1e-3) * k)))
        k = min(spec.B, grow)


def cpu_inputs(spec, seed):
    """Seeded inputs on the host for the oracle legs (independent of any GPU)."""
    return workloads.generate(spec, seed, device="cpu")


def run_reference(args, spec, world, rank):
    if rank != 0:
        return
    x = cpu_inputs(spec, seed=1)
    per_step_budget = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    # size the sample once, then time W + K steps of that sample
    _, rows, threads = oracle_sample(spec, x, per_step_budget, args.backward)
    grads = backward_grads(spec, x, 5, "cpu") if args.backward else None
    for _ in range(args.warmup):
        oracle_call(x, rows, args.backward, grads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_call(x, rows, args.backward, grads)
    dt = (time.perf_counter() - t0) / args.steps
    if args.backward:
        nbytes = algorithmic_bytes_backward(spec, x.lengths[:rows].tolist(),
                                            x.append_mask[:rows].to(torch.int64).sum(1).tolist()
                                            )["total"]
    elif args.inplace or args.readonly:  # the same attention, counted with that face's bytes
        f = algorithmic_bytes_readonly if args.readonly else algorithmic_bytes_inplace
        nbytes = f(spec, x.lengths[:rows].tolist(),
                   x.append_mask[:rows].to(torch.int64).sum(1).tolist())["total"]
    else:
        nbytes = algorithmic_bytes(spec, rows)["total"]
    value = nbytes / dt / 1e9
    sample = f"first {rows} of {spec.B} batch rows of {args.workload} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, spec),
        "steps_per_s": round(1.0 / dt * rows / spec.B, 6),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(name, spec):
    return {"workload": name, "B": spec.B, "Hq": spec.Hq, "Hk": spec.Hk, "Q": spec.Q,
            "D": spec.D, "Dv": spec.Dv, "M": spec.M, "dtype": spec.dtype,
            "lengths": list(spec.lengths), "append_counts": list(spec.counts),
            "scale": spec.scale if spec.scale is not None else "1/sqrt(D)",
            "l2": "inputs (caches) larger than the 129 MB L2; no flush between steps"}


# ----------------------------------------------------------------- GPU leg
def run_ours(args, spec, world, rank, local):
    import kv_cache_append_gb300 as kvc
    from kv_cache_append_gb300 import build as kbuild
    if not os.path.exists(kbuild.LIB):
        kbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = workloads.generate(spec, seed=1 + rank, device=dev)
    q, nk, nv, kc, vc, ln, mk = x.args()
    mk = mk.view(torch.uint8)
    scale = x.options.get("scale", kvc.default_scale(spec.D))
    dims = kvc.dims_of(q, kc, vc)
    out = kvc.allocate_outputs(q, kc, vc)
    nws = kvc.workspace_bytes(dims)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
    stream = torch.cuda.current_stream(dev)
    if args.paged:
        # the caches as a pool of block_size-slot blocks in a shuffled order
        bs = args.paged
        Bn, Hk_, M_ = kc.shape[:3]
        mb = M_ // bs
        g = torch.Generator().manual_seed(17 + rank)
        perm = torch.randperm(Bn * mb, generator=g).to(dev)
        table = perm.reshape(Bn, mb).to(torch.int32)

        def to_pool(c):
            W = c.shape[-1]
            blocks = c.reshape(Bn, Hk_, mb, bs, W).permute(0, 2, 1, 3, 4).reshape(Bn * mb, Hk_, bs, W)
            pool = torch.empty_like(blocks)
            pool[perm] = blocks
            return pool
        kc_p, vc_p = to_pool(kc), to_pool(vc)
        del out["key_cache"], out["value_cache"]
        x.key_cache = x.value_cache = None
        kc = vc = None
        torch.cuda.empty_cache()
        ws = torch.empty(kvc.paged_workspace_bytes(dims), dtype=torch.uint8, device=dev)
        nkern = 5 if spec.Q > 0 else 2
        path = kvc.plan_info_inplace(dims, kc_p, vc_p, nk, nv)[1]
        if path in ("tensor", "decode_tc") and not (bs % 64 == 0 or (64 % bs == 0 and bs >= 8)):
            path = "fused"

        def step(events=None):
            kvc.step_paged_into(dims, table, q, nk, nv, kc_p, vc_p, ln, mk, scale, out, ws, None,
                                stream.cuda_stream, events)
    elif args.readonly:
        # packed queries = the step's valid query rows; each sequence's cached
        # length = its new length; cache rows visited through a permutation
        counts_d = x.append_mask.to(torch.int64).sum(1)
        Bn = spec.B
        rows_q = [q[b, :, :int(counts_d[b])].permute(1, 0, 2) for b in range(Bn)]
        q_packed = torch.cat(rows_q, 0).contiguous()
        cu = torch.zeros(Bn + 1, dtype=torch.int32, device=dev)
        cu[1:] = torch.cumsum(counts_d, 0).to(torch.int32)
        kl = (x.lengths + counts_d).to(torch.int32)
        g = torch.Generator().manual_seed(11 + rank)
        perm = torch.randperm(Bn, generator=g)
        kc_p, vc_p = kc[perm].contiguous(), vc[perm].contiguous()   # sequence b in row inv[b]
        slots = torch.argsort(perm).to(torch.int32).to(dev)
        del out
        out_ro = torch.empty(q_packed.shape[0], spec.Hq, spec.Dv, dtype=q.dtype, device=dev)
        ws = torch.empty(kvc.attend_cache_workspace_bytes(dims), dtype=torch.uint8, device=dev)
        torch.cuda.empty_cache()
        nkern = 4
        path = kvc.plan_info_inplace(dims, kc_p, vc_p, nk, nv)[1]

        def step(events=None):
            kvc.attend_cache_into(dims, Bn, q_packed, kc_p, vc_p, cu, kl, False, slots, scale,
                                  out_ro, ws, None, stream.cuda_stream, events)
    elif args.backward:
        # the step's gradients for seeded upstream gradients of all four outputs
        grads = backward_grads(spec, x, 5 + rank, dev)
        outb = {"query": torch.empty_like(q), "new_key": torch.empty_like(nk),
                "new_value": torch.empty_like(nv), "key_cache": torch.empty_like(kc),
                "value_cache": torch.empty_like(vc)}
        del out
        torch.cuda.empty_cache()
        ws = torch.empty(kvc.backward_workspace_bytes(dims), dtype=torch.uint8, device=dev)
        nkern, path, slot_kernel = kvc.backward_plan_info(dims)

        def step(events=None):
            kvc.step_backward_into(dims, q, nk, nv, kc, vc, ln, mk, scale, grads, outb, ws, None,
                                   stream.cuda_stream, events)
    elif args.inplace:
        # donated caches: every step appends the same rows at the same slots,
        # so repeated steps leave the caches as the first one did
        nkern, path = kvc.plan_info_inplace(dims, kc, vc, nk, nv)
        del out["key_cache"], out["value_cache"]
        torch.cuda.empty_cache()

        def step(events=None):
            kvc.step_inplace_into(dims, q, nk, nv, kc, vc, ln, mk, scale, out, ws, None,
                                  stream.cuda_stream, events)
    else:
        nkern, path = kvc.plan_info(dims, kc, vc, nk, nv, out["key_cache"], out["value_cache"])

        def step(events=None):
            kvc.step_into(dims, q, nk, nv, kc, vc, ln, mk, scale, out, ws, None,
                          stream.cuda_stream, events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # the timed steps carry no events between their kernels (an event there
    # would keep the row writer from starting before the merge ends); a
    # separate run of steps with events between the kernels gives the split
    nev = nkern + 1
    nsplit = min(args.steps, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(nsplit)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    for e in [ev for row in evs for ev in row] + [start, end]:
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    ms_total = start.elapsed_time(end)
    time.sleep(0.25)
    clocks.stop()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    for i in range(nsplit):
        step(evs[i])
    torch.cuda.synchronize(dev)
    kern_ms = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evs) for k in range(nkern)]

    lengths_h = x.lengths.cpu().tolist()
    counts_h = x.append_mask.to(torch.int64).sum(1).cpu().tolist()
    nbytes = (algorithmic_bytes_backward(spec, lengths_h, counts_h) if args.backward else
              algorithmic_bytes_readonly(spec, lengths_h, counts_h) if args.readonly else
              algorithmic_bytes_inplace(spec, lengths_h, counts_h) if (args.inplace or args.paged)
              else algorithmic_bytes(spec))
    value = world * nbytes["total"] / (ms_step * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    if args.backward:  # the longer of the two HBM kernels of the gradients
        names_b = list(PATH_KERNELS_BACKWARD[path] if spec.Q > 0
                       else ["bwd_kv_kernel", "bwd_copy_kernel"])
        assert len(names_b) == nkern, (names_b, nkern)
        ks = max((i for i, nm in enumerate(names_b) if nm in ("bwd_kv_kernel", "bwd_copy_kernel")),
                 key=lambda i: kern_ms[i])
        nbytes["fused_kernel"] = nbytes[names_b[ks]]
        names_b = [slot_kernel if nm == "bwd_kv_kernel" else nm for nm in names_b]
        kname = names_b[ks]
    else:
        ks = (2 if args.paged and nkern > 2 else
              1 if (args.inplace or args.readonly) and nkern > 1 else 0)  # index of the step kernel
        kname = STEP_KERNEL[path]
        if args.readonly and path == "generic":
            kname = "generic_attend_kernel"
        nbytes["fused_kernel"] = step_kernel_bytes(nbytes, path)
    fused_ms = kern_ms[ks]
    achieved = nbytes["fused_kernel"] / (fused_ms * 1e-3) / 1e9
    traffic = kernel_traffic(mode_key(args), kname, nbytes["fused_kernel"])
    roof = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": traffic}
    if args.backward and kname.startswith("bwd_kv") and kname != "bwd_kv_tc_kernel":
        # a CUDA-core slot kernel: bound by its fp32 products when they take
        # longer at the CUDA-core peak than its bytes at the HBM peak (the
        # tensor-core one is HBM-bound: its products take ~1/20 of its bytes' time)
        flops = flops_backward(spec, lengths_h, counts_h)
        if flops / (FP32_PEAK_TFLOPS * 1e12) > nbytes["fused_kernel"] / (peak * 1e9):
            tf = flops / (fused_ms * 1e-3) / 1e12
            roof = {"bound": "alu", "kernel": kname, "achieved": round(tf, 2),
                    "peak": round(FP32_PEAK_TFLOPS, 2), "unit": "TFLOP/s",
                    "frac": round(tf / FP32_PEAK_TFLOPS, 4),
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x 2070 MHz",
                    "flops": flops, "hbm_frac": round(achieved / peak, 4), "traffic": traffic}

    # ---- end to end through the public API: pinned host in, pinned host out
    e2e = None
    if args.readonly or args.paged or args.backward:
        e2e = None  # these faces have no host-buffer leg here
    elif not args.no_e2e:
        e2e = (measure_e2e_inplace(kvc, x, dev, max(3, min(args.steps, 10)), nbytes["total"],
                                   world) if args.inplace else
               measure_e2e(kvc, x, dev, spec, max(3, min(args.steps, 10)), nbytes["total"], world))

    # ---- CPU oracle baseline, rank 0 at N = 1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xc = cpu_inputs(spec, seed=1)
        dt, rows, threads = oracle_sample(spec, xc, args.cpu_budget, args.backward)
        sample_bytes = (algorithmic_bytes_backward(spec, lengths_h[:rows], counts_h[:rows])
                        if args.backward else
                        algorithmic_bytes_readonly(spec, lengths_h[:rows], counts_h[:rows])
                        if args.readonly else
                        algorithmic_bytes_inplace(spec, lengths_h[:rows], counts_h[:rows])
                        if (args.inplace or args.paged) else algorithmic_bytes(spec, rows))
        cpu = {"value": round(sample_bytes["total"] / dt / 1e9, 4),
               "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"first {rows} of {spec.B} batch rows of {args.workload}, one "
                         + ("backward" if args.backward else "step")
                         + (" (the oracle's step: the same attention plus the cache copy)"
                            if args.readonly else "")}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": spec.dtype, "data": "synthetic",
        "config": config_of(args.workload, spec),
        "pct_of_8TBs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "steps_per_s": round(world * 1e3 / ms_step, 2),
        "bytes_per_step": nbytes["total"],
        "path": path,
        "kernels": {kname: {"ms": round(kern_ms[ks], 4),
                            "algorithmic_bytes": nbytes["fused_kernel"],
                            "algorithmic_GBps": round(achieved, 1)}},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": nkern * args.steps,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    names = (names_b if args.backward else
             (PATH_KERNELS_READONLY if args.readonly else PATH_KERNELS_PAGED if args.paged else
              PATH_KERNELS_INPLACE if args.inplace else PATH_KERNELS)[path])
    for k in range(nkern):
        if k != ks:
            line["kernels"][names[k]] = {"ms": round(kern_ms[k], 4)}
    if args.inplace:
        line["config"]["mode"] = ("in place: donated caches, only the appended rows written, "
                                  "the attention reads the valid prefix")
    if args.paged:
        line["config"]["mode"] = (f"paged: pools of {args.paged}-slot blocks in a shuffled "
                                  "order, updated in place through the block table")
    if args.readonly:
        line["config"]["mode"] = ("read-only re-attention: packed queries (the step's valid "
                                  "rows) over the cached prefix through a slot permutation; "
                                  "context only, no attention rows, cache not written")
    if args.backward:
        line["config"]["mode"] = ("backward: gradients of all four outputs given (seeded), "
                                  "the statistics pass over the inputs, then the gradients")
    if nkern > 2 and not args.backward:
        fin_ms = kern_ms[-1] + kern_ms[-2]
        line["kernels"]["merge + unpack" if args.readonly else "finalize (merge + rows)"] = {
            "ms": round(fin_ms, 4),
            "algorithmic_GBps": round(nbytes["finalize_kernel"] / (fin_ms * 1e-3) / 1e9, 1)}
    default_face = not (args.inplace or args.paged or args.readonly or args.backward)
    if (world == 1 and default_face and not args.no_per_config and args.batch is None
            and args.q is None and args.dtype is None):
        x = out = ws = q = nk = nv = kc = vc = ln = mk = step = None
        torch.cuda.empty_cache()
        line["per_config"] = run_per_config(args, kvc, dev, stream)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- the other configs
# Every configuration the metric is quoted per, measured in the same run as the
# headline: (name, workload, dtype override).
PER_CONFIG = [("tiny_fp32", "tiny_fp32", None), ("chunked_append_bf16", "chunked_append", "bf16"),
              ("chunked_append_f32", "chunked_append", "f32"),
              ("ragged_specdec", "ragged_specdec", None), ("long_mqa", "long_mqa", None)]
L2_FLUSH_BYTES = 512 << 20   # written between timed steps of the L2-sized configs


def _roofline_entry(kname, kern_ms, kbytes, key, peak, peak_src):
    achieved = kbytes / (kern_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": kernel_traffic(key, kname, kbytes)}


def _split_kernels(step, nkern, reps, stream, dev, flush=None):
    """Mean time of each kernel of a step: events recorded between them."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nkern + 1)] for _ in range(reps)]
    for e in [ev for row in evs for ev in row]:
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize(dev)
    for i in range(reps):
        if flush is not None:
            flush()
        step(evs[i])
    torch.cuda.synchronize(dev)
    return [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evs) for k in range(nkern)]


def _cpu_entry(spec, x_cpu, budget, what):
    dt, rows, threads = oracle_sample(spec, x_cpu, budget)
    sample_bytes = algorithmic_bytes(spec, rows)["total"]
    return {"value": round(sample_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"first {rows} of {spec.B} batch rows of {what}, one step"}


def measure_config(kvc, name, spec, steps, warmup, dev, stream, cpu_budget, peak, peak_src):
    """ms/step, GB/s, steps/s, the step kernel's roofline and the oracle's
    GB/s for one configuration. Inputs larger than L2 are timed back to back;
    smaller ones with an L2 flush (a write larger than L2) before each step,
    events around the step only."""
    x = workloads.generate(spec, seed=1, device=dev)
    q, nk, nv, kc, vc, ln, mk = x.args()
    mk = mk.view(torch.uint8)
    scale = x.options.get("scale", kvc.default_scale(spec.D))
    dims = kvc.dims_of(q, kc, vc)
    out = kvc.allocate_outputs(q, kc, vc)
    ws = torch.empty(max(1, kvc.workspace_bytes(dims)), dtype=torch.uint8, device=dev)
    nkern, path = kvc.plan_info(dims, kc, vc, nk, nv, out["key_cache"], out["value_cache"])
    nbytes = algorithmic_bytes(spec)
    small = 2 * nbytes["fused_kernel"] < (128 << 20)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if small else None

    def flush():
        flush_buf.fill_(1)

    def step(events=None):
        kvc.step_into(dims, q, nk, nv, kc, vc, ln, mk, scale, out, ws, None, stream.cuda_stream,
                      events)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    if small:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / steps
    kern_ms = _split_kernels(step, nkern, min(steps, 20), stream, dev, flush if small else None)
    kname = STEP_KERNEL[path]
    entry = {"workload": name, "path": path, "ms_per_step": round(ms, 4),
             "GBps": round(nbytes["total"] / (ms * 1e-3) / 1e9, 2),
             "pct_of_8TBs": round(100.0 * nbytes["total"] / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 2),
             "steps_per_s": round(1e3 / ms, 2), "bytes_per_step": nbytes["total"],
             "kernels_ms": {nm: round(t, 4) for nm, t in zip(PATH_KERNELS[path], kern_ms)},
             "roofline": _roofline_entry(kname, kern_ms[0], step_kernel_bytes(nbytes, path), name,
                                         peak, peak_src),
             "timed_steps": steps,
             "l2": ("inputs smaller than L2: a 512 MB write flushes it before each timed step"
                    if small else "inputs larger than the 129 MB L2; no flush")}
    del x, out, ws, flush_buf
    torch.cuda.empty_cache()
    if cpu_budget > 0:
        entry["cpu_baseline"] = _cpu_entry(spec, cpu_inputs(spec, seed=1), cpu_budget, name)
    return entry


def measure_chain(kvc, name, spec, steps, warmup, dev, stream, cpu_budget, peak, peak_src):
    """The chunked append as the configuration defines it: three chained steps
    (Q = 40, 32, 24), each consuming the previous step's returned caches and
    lengths. L2 is flushed before each chain; each step is timed with events."""
    first, rest = workloads.chain_chunks(spec, seed=1, device=dev)
    qs = [first.query] + [r[0] for r in rest]
    nks = [first.new_key] + [r[1] for r in rest]
    nvs = [first.new_value] + [r[2] for r in rest]
    mks = [first.append_mask.view(torch.uint8)] + [r[3].view(torch.uint8) for r in rest]
    scale = first.options.get("scale", kvc.default_scale(spec.D))
    outs, dims, plans = [], [], []
    kc, vc, ln = first.key_cache, first.value_cache, first.lengths
    for k in range(len(qs)):
        d = kvc.dims_of(qs[k], kc, vc)
        o = kvc.allocate_outputs(qs[k], kc, vc)
        plans.append(kvc.plan_info(d, kc, vc, nks[k], nvs[k], o["key_cache"], o["value_cache"]))
        outs.append(o)
        dims.append(d)
        kc, vc, ln = o["key_cache"], o["value_cache"], o["lengths"]
    ws = torch.empty(max(kvc.workspace_bytes(d) for d in dims), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def one(k, events=None):
        src = {"key_cache": first.key_cache, "value_cache": first.value_cache,
               "lengths": first.lengths} if k == 0 else outs[k - 1]
        kvc.step_into(dims[k], qs[k], nks[k], nvs[k], src["key_cache"], src["value_cache"],
                      src["lengths"], mks[k], scale, outs[k], ws, None, stream.cuda_stream, events)

    for _ in range(warmup):
        for k in range(len(qs)):
            one(k)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(qs) + 1)] for _ in range(steps)]
    for e in ev:
        flush_buf.fill_(1)
        e[0].record(stream)
        for k in range(len(qs)):
            one(k)
            e[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    per_q = {}
    for k, Q in enumerate(workloads.CHUNKS):
        ms = statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev)
        nkern, path = plans[k]
        sk = spec.replace(Q=Q)
        nbytes = algorithmic_bytes(sk)

        def step_k(events=None, k=k):
            one(k, events)

        def prep(k=k):   # the chain up to step k, after a flush
            flush_buf.fill_(1)
            for j in range(k):
                one(j)
        kern_ms = _split_kernels(step_k, nkern, min(steps, 20), stream, dev, prep)
        kname = STEP_KERNEL[path]
        per_q[f"Q{Q}"] = {
            "path": path, "ms_per_step": round(ms, 4),
            "GBps": round(nbytes["total"] / (ms * 1e-3) / 1e9, 2),
            "steps_per_s": round(1e3 / ms, 2), "bytes_per_step": nbytes["total"],
            "kernels_ms": {nm: round(t, 4) for nm, t in zip(PATH_KERNELS[path], kern_ms)},
            "roofline": _roofline_entry(kname, kern_ms[0], step_kernel_bytes(nbytes, path),
                                        f"{name}:Q{Q}", peak, peak_src)}
    chain_ms = sum(v["ms_per_step"] for v in per_q.values())
    entry = {"workload": "chunked_append", "dtype": spec.dtype, "chain": list(workloads.CHUNKS),
             "per_step": per_q, "chain_ms": round(chain_ms, 4),
             "chains_per_s": round(1e3 / chain_ms, 2), "timed_chains": steps,
             "l2": "inputs smaller than L2: a 512 MB write flushes it before each chain",
             "note": "L2-sized and launch-bound by design; GB/s is reported, steps/s is the figure"}
    del outs, ws, flush_buf, first, rest
    torch.cuda.empty_cache()
    if cpu_budget > 0:
        s40 = spec.replace(Q=workloads.CHUNKS[0])
        entry["cpu_baseline"] = _cpu_entry(s40, cpu_inputs(s40, seed=1), cpu_budget,
                                           f"{name} (the Q=40 step)")
    return entry


def run_per_config(args, kvc, dev, stream):
    """Every other configuration, measured after the headline one."""
    peak, peak_src = measured_peak()
    budget = 0.0 if args.no_cpu_baseline else min(args.cpu_budget, 4.0)
    res = {}
    for name, wl, dt in PER_CONFIG:
        if wl == args.workload and dt is None:
            continue
        spec = workloads.SPECS[wl] if dt is None else workloads.SPECS[wl].replace(dtype=dt)
        slow = wl == "ragged_specdec"
        steps = max(5, min(args.steps, 40 if slow else 200))
        warm = max(3, min(args.warmup, 5))
        if wl == "chunked_append":
            res[name] = measure_chain(kvc, name, spec, steps, warm, dev, stream, budget, peak,
                                      peak_src)
        else:
            res[name] = measure_config(kvc, name, spec, steps, warm, dev, stream, budget, peak,
                                       peak_src)
    return res


def measure_e2e(kvc, x, dev, spec, steps, nbytes, world):
    """The public call with host buffers: every step copies the inputs from
    pinned host memory, runs kv_cache_attention_step and copies every output
    back. Two input and two output buffers alternate, the host-to-device
    copies run on one copy stream and the device-to-host copies on another, so
    step i+1's inputs stream in while step i's outputs stream out; every copy
    of every step is inside the timed region."""
    host_in = [t.to("cpu").pin_memory() for t in x.args()]
    out0 = kvc.kv_cache_attention_step(*x.args(), x.options)
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out0.items()}
                for _ in range(2)]
    del out0
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    stream = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]     # dev_in[s] consumed by its step
    drained = [torch.cuda.Event() for _ in range(2)]   # host_out[s] written back
    for e in freed + drained:
        e.record(stream)

    def one(i):
        s_ = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(freed[s_])
            for d, h in zip(dev_in[s_], host_in):
                d.copy_(h, non_blocking=True)
        stream.wait_stream(s_in)
        out = kvc.kv_cache_attention_step(*dev_in[s_], x.options)
        freed[s_].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_stream(stream)
            s_out.wait_event(drained[s_])
            for k, v in out.items():
                host_out[s_][k].copy_(v, non_blocking=True)
                v.record_stream(s_out)
            drained[s_].record(s_out)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(steps):
        one(i)
    stream.wait_stream(s_out)
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(s.elapsed_time(e) / steps, world)
    return {"value": round(world * nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": steps, "copies": "double-buffered; H2D and D2H on two copy streams"}


def measure_e2e_inplace(kvc, x, dev, steps, nbytes, world):
    """The in-place public call with host buffers for everything but the
    donated caches, which stay resident on the device as a serving loop keeps
    them: every step copies query, new rows, lengths and mask in from pinned
    host memory and copies lengths, attention and context back."""
    kc, vc = x.key_cache, x.value_cache
    host_in = [t.to("cpu").pin_memory() for t in (x.query, x.new_key, x.new_value, x.lengths,
                                                  x.append_mask)]
    out0 = kvc.kv_cache_attention_step_inplace(x.query, x.new_key, x.new_value, kc, vc,
                                               x.lengths, x.append_mask, x.options)
    keys = ("lengths", "attention", "context")
    host_out = {k: torch.empty(out0[k].shape, dtype=out0[k].dtype, pin_memory=True) for k in keys}
    del out0
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    stream = torch.cuda.current_stream(dev)

    def one():
        q, nk, nv, ln, mk = (t.to(dev, non_blocking=True) for t in host_in)
        out = kvc.kv_cache_attention_step_inplace(q, nk, nv, kc, vc, ln, mk, x.options)
        for k in keys:
            host_out[k].copy_(out[k], non_blocking=True)

    one()
    torch.cuda.synchronize(dev)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        one()
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(s.elapsed_time(e) / steps, world)
    return {"value": round(world * nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "steps": steps, "resident": "key_cache, value_cache (donated, updated in place)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_decode", choices=sorted(workloads.SPECS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only --workload (no per_config block for the other configs)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size B (profiling captures)")
    ap.add_argument("--q", type=int, default=None,
                    help="override the tokens per step Q (the 32- and 24-token chunked appends)")
    ap.add_argument("--dtype", choices=["f32", "bf16", "f16"], default=None,
                    help="override the workload's dtype (the fp32 chunked append)")
    ap.add_argument("--inplace", action="store_true",
                    help="time kvc_step_inplace (donated caches updated in place)")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK_SIZE",
                    help="time kvc_step_paged on pools of BLOCK_SIZE-slot blocks")
    ap.add_argument("--readonly", action="store_true",
                    help="time kvc_attend_cache (read-only re-attention over the cache)")
    ap.add_argument("--backward", action="store_true",
                    help="time kvc_step_backward (gradients of the step's outputs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    spec = workloads.SPECS[args.workload]
    if args.batch:
        spec = spec.replace(B=args.batch)
    if args.q is not None:
        spec = spec.replace(Q=args.q)
    if args.dtype:
        spec = spec.replace(dtype=args.dtype)
    if args.impl == "reference":
        run_reference(args, spec, world, rank)
    else:
        run_ours(args, spec, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
