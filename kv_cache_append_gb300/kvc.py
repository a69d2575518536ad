"""ctypes binding of libkvc (include/kvc.h).

Argument marshalling only: every step of the operation runs in libkvc's CUDA
kernels. PyTorch supplies device memory and the current stream. There is no
CPU fallback: if libkvc.so is missing or the tensors are not on a CUDA
device, the call raises.

Python face of the step, as on the page "Autoregressive KV-cache append and
causal attention" (Function signature / Return):

    kv_cache_attention_step(query, new_key, new_value, key_cache, value_cache,
                            lengths, append_mask, options)
        -> {"key_cache", "value_cache", "lengths", "attention", "context"}
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVC_LIBRARY names another build of the same library (e.g. one compiled with
# other compile-time options by build.build_variant); default: the in-tree build.
LIB_PATH = os.environ.get("KVC_LIBRARY") or os.path.join(_HERE, "libkvc.so")

DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}

KVC_OK = 0
STATUS_NAMES = {0: "KVC_OK", -1: "KVC_E_NULL", -2: "KVC_E_SHAPE", -3: "KVC_E_DTYPE",
                -4: "KVC_E_SCALE", -5: "KVC_E_WORKSPACE", -6: "KVC_E_ALIAS",
                -7: "KVC_E_DEVICE", -8: "KVC_E_CUDA", -9: "KVC_E_STATIC_LIMIT"}
DEV_OVERFLOW, DEV_MASK, DEV_TIMEOUT = 1, 2, 4


class KvcError(ValueError):
    """A libkvc call returned a KVC_E_* status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hk", ctypes.c_int64),
                ("Q", ctypes.c_int64), ("D", ctypes.c_int64), ("Dv", ctypes.c_int64),
                ("M", ctypes.c_int64), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvc.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m kv_cache_append_gb300.build` "
                    "(needs nvcc); there is no CPU fallback")
            lib = ctypes.CDLL(path)
            vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            dp = ctypes.POINTER(Dims)
            lib.kvc_workspace_bytes.restype = sz
            lib.kvc_workspace_bytes.argtypes = [dp]
            step_args = [dp] + [vp] * 7 + [ctypes.c_double] + [vp] * 6 + [sz, vp, vp]
            lib.kvc_step.restype = i32
            lib.kvc_step.argtypes = step_args
            lib.kvc_step_timed.restype = i32
            lib.kvc_step_timed.argtypes = step_args + [ctypes.POINTER(vp), i32]
            lib.kvc_step_static.restype = i32
            lib.kvc_step_static.argtypes = [dp] + [vp] * 7 + [ctypes.c_double] + [vp] * 7
            lib.kvc_plan_info.restype = i32
            lib.kvc_plan_info.argtypes = [dp] + [vp] * 6 + [ctypes.POINTER(ctypes.c_char_p)]
            inplace_args = [dp] + [vp] * 7 + [ctypes.c_double] + [vp] * 4 + [sz, vp, vp]
            lib.kvc_step_inplace.restype = i32
            lib.kvc_step_inplace.argtypes = inplace_args
            lib.kvc_step_inplace_timed.restype = i32
            lib.kvc_step_inplace_timed.argtypes = inplace_args + [ctypes.POINTER(vp), i32]
            lib.kvc_plan_info_inplace.restype = i32
            lib.kvc_plan_info_inplace.argtypes = [dp] + [vp] * 4 + [ctypes.POINTER(ctypes.c_char_p)]
            lib.kvc_backward_plan_info.restype = i32
            lib.kvc_backward_plan_info.argtypes = [dp] + [ctypes.POINTER(ctypes.c_char_p)] * 2
            i64 = ctypes.c_int64
            attend_args = ([dp, i64, i64] + [vp] * 5 + [i32, vp, ctypes.c_double, vp, vp, sz, vp,
                                                         vp])
            lib.kvc_attend_cache_workspace_bytes.restype = sz
            lib.kvc_attend_cache_workspace_bytes.argtypes = [dp]
            lib.kvc_attend_cache.restype = i32
            lib.kvc_attend_cache.argtypes = attend_args
            lib.kvc_attend_cache_timed.restype = i32
            lib.kvc_attend_cache_timed.argtypes = attend_args + [ctypes.POINTER(vp), i32]
            paged_args = ([dp, i64, i64] + [vp] * 8 + [ctypes.c_double] + [vp] * 4 +
                          [sz, vp, vp])
            lib.kvc_paged_workspace_bytes.restype = sz
            lib.kvc_paged_workspace_bytes.argtypes = [dp]
            lib.kvc_step_paged.restype = i32
            lib.kvc_step_paged.argtypes = paged_args
            lib.kvc_step_paged_timed.restype = i32
            lib.kvc_step_paged_timed.argtypes = paged_args + [ctypes.POINTER(vp), i32]
            lib.kvc_backward_workspace_bytes.restype = sz
            lib.kvc_backward_workspace_bytes.argtypes = [dp]
            lib.kvc_step_backward.restype = i32
            lib.kvc_step_backward.argtypes = ([dp] + [vp] * 7 + [ctypes.c_double] + [vp] * 9 +
                                              [vp, sz, vp, vp])
            lib.kvc_step_backward_timed.restype = i32
            lib.kvc_step_backward_timed.argtypes = (lib.kvc_step_backward.argtypes +
                                                    [ctypes.POINTER(vp), i32])
            lib.kvc_selftest_wait_timeout.restype = i32
            lib.kvc_selftest_wait_timeout.argtypes = [vp, i64, vp]
            lib.kvc_status_string.restype = ctypes.c_char_p
            lib.kvc_status_string.argtypes = [i32]
            lib.kvc_version.restype = i32
            lib.kvc_version.argtypes = []
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().kvc_status_string(status).decode()


def selftest_wait_timeout(status, limit_ns: int = 5_000_000, stream=None) -> None:
    """kvc_selftest_wait_timeout: a kernel whose pipeline wait is never
    satisfied gives up after limit_ns and ORs DEV_TIMEOUT into `status` (a
    device int32 tensor of one element)."""
    if not (status.is_cuda and status.dtype == torch.int32 and status.numel() >= 1):
        raise ValueError("status must be a device int32 tensor")
    s = torch.cuda.current_stream(status.device).cuda_stream if stream is None else stream
    rc = library().kvc_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), int(limit_ns),
                                             ctypes.c_void_p(s))
    if rc != 0:
        raise KvcError(rc, status_string(rc))


def make_dims(B, Hq, Hk, Q, D, Dv, M, dtype) -> Dims:
    code = DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return Dims(B, Hq, Hk, Q, D, Dv, M, code)


def dims_of(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor) -> Dims:
    B, Hq, Q, D = query.shape
    _, Hk, M, _ = key_cache.shape
    return make_dims(B, Hq, Hk, Q, D, value_cache.shape[-1], M, key_cache.dtype)


def workspace_bytes(dims: Dims) -> int:
    return int(library().kvc_workspace_bytes(ctypes.byref(dims)))


def plan_info(dims: Dims, key_cache, value_cache, new_key, new_value, out_key_cache,
              out_value_cache):
    """(kernel count, path name) kvc_step takes for these tensors."""
    name = ctypes.c_char_p()
    n = library().kvc_plan_info(ctypes.byref(dims), *(_p(t) for t in (
        key_cache, value_cache, new_key, new_value, out_key_cache, out_value_cache)),
        ctypes.byref(name))
    if n < 0:
        raise KvcError(n, status_string(n))
    return n, name.value.decode()


def plan_info_inplace(dims: Dims, key_cache, value_cache, new_key, new_value):
    """(kernel count, path name) kvc_step_inplace takes for these tensors."""
    name = ctypes.c_char_p()
    n = library().kvc_plan_info_inplace(ctypes.byref(dims), *(_p(t) for t in (
        key_cache, value_cache, new_key, new_value)), ctypes.byref(name))
    if n < 0:
        raise KvcError(n, status_string(n))
    return n, name.value.decode()


def backward_plan_info(dims: Dims):
    """(kernel count, statistics path, slot kernel) kvc_step_backward takes
    for these shapes with 16-byte aligned buffers."""
    stats, slot = ctypes.c_char_p(), ctypes.c_char_p()
    n = library().kvc_backward_plan_info(ctypes.byref(dims), ctypes.byref(stats),
                                         ctypes.byref(slot))
    if n < 0:
        raise KvcError(n, status_string(n))
    return n, stats.value.decode(), slot.value.decode()


def _p(t: Optional[torch.Tensor]):
    if t is None or t.numel() == 0:
        return None
    return ctypes.c_void_p(t.data_ptr())


def default_scale(D: int) -> float:
    """The page's default scale 1/sqrt(D)."""
    return 1.0 / math.sqrt(D)


def _scale_from(options: Optional[dict], D: int) -> float:
    options = dict(options or {})
    scale = options.pop("scale", None)
    if options:
        raise ValueError(f"unknown option keys {sorted(options)}: 'scale' is the only key")
    if scale is None:
        return default_scale(D)
    scale = float(scale)
    if not (scale > 0.0 and math.isfinite(scale)):
        raise ValueError("scale must be positive and finite")
    return scale


def check_inputs(query, new_key, new_value, key_cache, value_cache, lengths, append_mask):
    """Shape/dtype/device contract of the step (Required behavior, bullet 1)."""
    for name, t in (("query", query), ("new_key", new_key), ("new_value", new_value),
                    ("key_cache", key_cache), ("value_cache", value_cache)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D, got {tuple(t.shape)}")
        if t.dtype not in DTYPES:
            raise ValueError(f"{name}: dtype {t.dtype} not in float32/bfloat16/float16")
        if t.dtype != query.dtype:
            raise ValueError("query, new_key, new_value and the caches need one dtype")
        if t.device != query.device:
            raise ValueError("all tensors must be on one device")
    if query.device.type != "cuda":
        raise ValueError("kv_cache_attention_step runs on a CUDA device only (no CPU path)")
    B, Hq, Q, D = query.shape
    _, Hk, M, _ = key_cache.shape
    Dv = value_cache.shape[-1]
    if tuple(key_cache.shape) != (B, Hk, M, D):
        raise ValueError(f"key_cache shape {tuple(key_cache.shape)} != {(B, Hk, M, D)}")
    if tuple(value_cache.shape) != (B, Hk, M, Dv):
        raise ValueError(f"value_cache shape {tuple(value_cache.shape)} != {(B, Hk, M, Dv)}")
    if tuple(new_key.shape) != (B, Hk, Q, D):
        raise ValueError(f"new_key shape {tuple(new_key.shape)} != {(B, Hk, Q, D)}")
    if tuple(new_value.shape) != (B, Hk, Q, Dv):
        raise ValueError(f"new_value shape {tuple(new_value.shape)} != {(B, Hk, Q, Dv)}")
    if min(B, Hq, Hk, D, Dv, M) < 1 or Hq % Hk:
        raise ValueError("need B,Hq,Hk,D,Dv,M >= 1 and Hq a multiple of Hk")
    if tuple(lengths.shape) != (B,) or lengths.device != query.device:
        raise ValueError("lengths must be [B] on the same device")
    if lengths.dtype.is_floating_point or lengths.dtype == torch.bool:
        raise ValueError("lengths must be integers")
    if tuple(append_mask.shape) != (B, Q) or append_mask.device != query.device:
        raise ValueError("append_mask must be [B, Q] on the same device")
    if append_mask.dtype not in (torch.bool, torch.uint8):
        raise ValueError("append_mask must be bool")
    return B, Hq, Hk, Q, D, Dv, M


def allocate_outputs(query, key_cache, value_cache) -> dict:
    B, Hq, Q, _ = query.shape
    M, Dv = key_cache.shape[2], value_cache.shape[-1]
    dev, dt = query.device, query.dtype
    return {
        "key_cache": torch.empty_like(key_cache, memory_format=torch.contiguous_format),
        "value_cache": torch.empty_like(value_cache, memory_format=torch.contiguous_format),
        "lengths": torch.empty(B, dtype=torch.int64, device=dev),
        "attention": torch.empty(B, Hq, Q, M, dtype=dt, device=dev),
        "context": torch.empty(B, Hq, Q, Dv, dtype=dt, device=dev),
    }


def step_into(dims: Dims, query, new_key, new_value, key_cache, value_cache, lengths,
              append_mask, scale: float, out: dict, workspace: Optional[torch.Tensor],
              status: Optional[torch.Tensor] = None, stream: Optional[int] = None,
              events: Optional[Sequence] = None) -> None:
    """Enqueue one kvc_step into preallocated outputs (no checks beyond libkvc's).

    All tensors must be contiguous CUDA tensors; lengths int64, append_mask
    one byte per entry. ``events`` (torch.cuda.Event, enable_timing) are
    recorded before the first kernel and after each kernel."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(query.device).cuda_stream
    ws_ptr = _p(workspace)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [ctypes.byref(dims), _p(query), _p(new_key), _p(new_value), _p(key_cache),
            _p(value_cache), _p(lengths), _p(append_mask), ctypes.c_double(scale),
            _p(out["key_cache"]), _p(out["value_cache"]), _p(out["lengths"]),
            _p(out["attention"]), _p(out["context"]), ws_ptr, ws_len, _p(status),
            ctypes.c_void_p(stream)]
    if events:
        handles = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
        rc = lib.kvc_step_timed(*args, handles, len(events))
    else:
        rc = lib.kvc_step(*args)
    if rc != KVC_OK:
        raise KvcError(rc, status_string(rc))


def kv_cache_attention_step(query: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor,
                            key_cache: torch.Tensor, value_cache: torch.Tensor,
                            lengths: torch.Tensor, append_mask: torch.Tensor,
                            options: Optional[dict] = None,
                            status: Optional[torch.Tensor] = None) -> dict:
    """One autoregressive KV-cache step on the GPU.

    Returns {"key_cache", "value_cache", "lengths", "attention", "context"}:
    the whole updated caches (new rows at slots length + t for the True-prefix
    of append_mask), lengths + n, attention [B,Hq,Q,M] and context
    [B,Hq,Q,Dv] under the lower-right causal rule. ``options`` may hold
    "scale" only (default 1/sqrt(D)). ``status`` is an optional int32 CUDA
    tensor of one element into which the kernels OR contract-violation bits
    (1 = capacity overflow, 2 = non-prefix mask); it is not synchronized.

    Differentiable: when gradients are enabled and query, new_key, new_value
    or a cache requires grad, the outputs carry a backward (kvc_step_backward)
    to all five (lengths has none).
    """
    if torch.is_grad_enabled() and any(
            t.requires_grad for t in (query, new_key, new_value, key_cache, value_cache)):
        kc, vc, ln, att, ctx = _Step.apply(query, new_key, new_value, key_cache, value_cache,
                                           lengths, append_mask, options, status)
        return {"key_cache": kc, "value_cache": vc, "lengths": ln, "attention": att,
                "context": ctx}
    return _step_forward(query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
                         options, status)


def _step_forward(query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
                  options, status) -> dict:
    check_inputs(query, new_key, new_value, key_cache, value_cache, lengths, append_mask)
    scale = _scale_from(options, query.shape[-1])
    q, nk, nv, kc, vc = (t.contiguous() for t in (query, new_key, new_value, key_cache,
                                                   value_cache))
    ln = lengths.to(torch.int64).contiguous()
    mk = append_mask.contiguous()
    mk = mk.view(torch.uint8) if mk.dtype == torch.bool else mk
    dims = dims_of(q, kc, vc)
    out = allocate_outputs(q, kc, vc)
    nbytes = workspace_bytes(dims)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    with torch.cuda.device(q.device):
        step_into(dims, q, nk, nv, kc, vc, ln, mk, scale, out, ws, status)
    return out


class _Step(torch.autograd.Function):
    """The step as an autograd node: forward kvc_step, backward kvc_step_backward."""

    @staticmethod
    def forward(ctx, query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
                options, status):
        out = _step_forward(query.detach(), new_key.detach(), new_value.detach(),
                            key_cache.detach(), value_cache.detach(), lengths, append_mask,
                            options, status)
        ctx.save_for_backward(query, new_key, new_value, key_cache, value_cache, lengths,
                              append_mask)
        ctx.options = options
        ctx.set_materialize_grads(False)
        ctx.mark_non_differentiable(out["lengths"])
        return (out["key_cache"], out["value_cache"], out["lengths"], out["attention"],
                out["context"])

    @staticmethod
    def backward(ctx, d_key_cache, d_value_cache, _d_lengths, d_attention, d_context):
        q, nk, nv, kc, vc, ln, mk = ctx.saved_tensors
        g = kv_cache_attention_step_backward(q.detach(), nk.detach(), nv.detach(), kc.detach(),
                                             vc.detach(), ln, mk, ctx.options,
                                             d_key_cache=d_key_cache, d_value_cache=d_value_cache,
                                             d_attention=d_attention, d_context=d_context)
        return (g["query"], g["new_key"], g["new_value"], g["key_cache"], g["value_cache"],
                None, None, None, None)


def backward_workspace_bytes(dims: Dims) -> int:
    return int(library().kvc_backward_workspace_bytes(ctypes.byref(dims)))


def step_backward_into(dims: Dims, query, new_key, new_value, key_cache, value_cache, lengths,
                       append_mask, scale: float, grads: dict, out: dict,
                       workspace: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream: Optional[int] = None, events: Optional[Sequence] = None) -> None:
    """Enqueue one kvc_step_backward (no checks beyond libkvc's). grads holds
    the gradients reaching "key_cache", "value_cache", "attention" and
    "context" (each a contiguous tensor of the inputs' dtype, or None for
    zero); out receives "query", "new_key", "new_value", "key_cache" and
    "value_cache"."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(query.device).cuda_stream
    args = [ctypes.byref(dims), _p(query), _p(new_key), _p(new_value), _p(key_cache),
            _p(value_cache), _p(lengths), _p(append_mask), ctypes.c_double(scale),
            *(_p(grads.get(k)) for k in ("key_cache", "value_cache", "attention", "context")),
            *(_p(out[k]) for k in ("query", "new_key", "new_value", "key_cache", "value_cache")),
            _p(workspace), workspace.numel(), _p(status), ctypes.c_void_p(stream)]
    if events:
        handles = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
        rc = lib.kvc_step_backward_timed(*args, handles, len(events))
    else:
        rc = lib.kvc_step_backward(*args)
    if rc != KVC_OK:
        raise KvcError(rc, status_string(rc))


def kv_cache_attention_step_backward(query, new_key, new_value, key_cache, value_cache, lengths,
                                     append_mask, options: Optional[dict] = None,
                                     d_key_cache=None, d_value_cache=None, d_attention=None,
                                     d_context=None, status: Optional[torch.Tensor] = None
                                     ) -> dict:
    """Gradients of the step's outputs (key_cache, value_cache, attention,
    context) with respect to query, new_key, new_value, key_cache and
    value_cache, given the gradients reaching those outputs (None = zero).
    Returns {"query", "new_key", "new_value", "key_cache", "value_cache"}."""
    check_inputs(query, new_key, new_value, key_cache, value_cache, lengths, append_mask)
    scale = _scale_from(options, query.shape[-1])
    q, nk, nv, kc, vc = (t.contiguous() for t in (query, new_key, new_value, key_cache,
                                                   value_cache))
    ln = lengths.to(torch.int64).contiguous()
    mk = append_mask.contiguous()
    mk = mk.view(torch.uint8) if mk.dtype == torch.bool else mk
    B, Hq, Q, D = q.shape
    M, Dv = kc.shape[2], vc.shape[-1]
    shapes = {"key_cache": tuple(kc.shape), "value_cache": tuple(vc.shape),
              "attention": (B, Hq, Q, M), "context": (B, Hq, Q, Dv)}
    grads = {}
    for name, g in (("key_cache", d_key_cache), ("value_cache", d_value_cache),
                    ("attention", d_attention), ("context", d_context)):
        if g is None:
            grads[name] = None
            continue
        if tuple(g.shape) != shapes[name] or g.device != q.device:
            raise ValueError(f"gradient of {name}: shape {tuple(g.shape)} != {shapes[name]}")
        grads[name] = g.to(q.dtype).contiguous()
    dims = dims_of(q, kc, vc)
    out = {"query": torch.empty_like(q), "new_key": torch.empty_like(nk),
           "new_value": torch.empty_like(nv), "key_cache": torch.empty_like(kc),
           "value_cache": torch.empty_like(vc)}
    ws = torch.empty(backward_workspace_bytes(dims), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        step_backward_into(dims, q, nk, nv, kc, vc, ln, mk, scale, grads, out, ws, status)
    return out


def step_inplace_into(dims: Dims, query, new_key, new_value, key_cache, value_cache, lengths,
                      append_mask, scale: float, out: dict, workspace: Optional[torch.Tensor],
                      status: Optional[torch.Tensor] = None, stream: Optional[int] = None,
                      events: Optional[Sequence] = None) -> None:
    """Enqueue one kvc_step_inplace: key_cache/value_cache are updated in
    place; out holds "lengths", "attention" and "context" (no checks beyond
    libkvc's)."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(query.device).cuda_stream
    ws_ptr = _p(workspace)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [ctypes.byref(dims), _p(query), _p(new_key), _p(new_value), _p(key_cache),
            _p(value_cache), _p(lengths), _p(append_mask), ctypes.c_double(scale),
            _p(out["lengths"]), _p(out["attention"]), _p(out["context"]), ws_ptr, ws_len,
            _p(status), ctypes.c_void_p(stream)]
    if events:
        handles = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
        rc = lib.kvc_step_inplace_timed(*args, handles, len(events))
    else:
        rc = lib.kvc_step_inplace(*args)
    if rc != KVC_OK:
        raise KvcError(rc, status_string(rc))


def kv_cache_attention_step_inplace(query: torch.Tensor, new_key: torch.Tensor,
                                    new_value: torch.Tensor, key_cache: torch.Tensor,
                                    value_cache: torch.Tensor, lengths: torch.Tensor,
                                    append_mask: torch.Tensor, options: Optional[dict] = None,
                                    status: Optional[torch.Tensor] = None) -> dict:
    """The step on donated caches, as a serving stack keeps them: key_cache
    and value_cache (contiguous CUDA tensors) are updated in place, only the
    appended rows [length, length + n) being written. Returns the same dict
    as kv_cache_attention_step, whose "key_cache"/"value_cache" are the
    arguments themselves."""
    check_inputs(query, new_key, new_value, key_cache, value_cache, lengths, append_mask)
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("the caches are updated in place and must be contiguous")
    scale = _scale_from(options, query.shape[-1])
    q, nk, nv = (t.contiguous() for t in (query, new_key, new_value))
    ln = lengths.to(torch.int64).contiguous()
    mk = append_mask.contiguous()
    mk = mk.view(torch.uint8) if mk.dtype == torch.bool else mk
    dims = dims_of(q, key_cache, value_cache)
    B, Hq, Q, _ = q.shape
    M, Dv = key_cache.shape[2], value_cache.shape[-1]
    out = {
        "key_cache": key_cache,
        "value_cache": value_cache,
        "lengths": torch.empty(B, dtype=torch.int64, device=q.device),
        "attention": torch.empty(B, Hq, Q, M, dtype=q.dtype, device=q.device),
        "context": torch.empty(B, Hq, Q, Dv, dtype=q.dtype, device=q.device),
    }
    nbytes = workspace_bytes(dims)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    with torch.cuda.device(q.device):
        step_inplace_into(dims, q, nk, nv, key_cache, value_cache, ln, mk, scale, out, ws, status)
    return out


def attend_cache_workspace_bytes(dims: Dims) -> int:
    return int(library().kvc_attend_cache_workspace_bytes(ctypes.byref(dims)))


def attend_cache_into(dims: Dims, num_slots: int, q, key_cache, value_cache, cu_seqlens_q,
                      seqlens_k, k_cumulative: bool, slot_ids, scale: float, out,
                      workspace: torch.Tensor, status: Optional[torch.Tensor] = None,
                      stream: Optional[int] = None, events: Optional[Sequence] = None) -> None:
    """Enqueue one kvc_attend_cache (no checks beyond libkvc's)."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(key_cache.device).cuda_stream
    ws_len = workspace.numel() * workspace.element_size()
    args = [ctypes.byref(dims), int(num_slots), int(q.shape[0]), _p(q), _p(key_cache),
            _p(value_cache), _p(cu_seqlens_q), _p(seqlens_k), int(bool(k_cumulative)),
            _p(slot_ids), ctypes.c_double(scale), _p(out), _p(workspace), ws_len, _p(status),
            ctypes.c_void_p(stream)]
    if events:
        handles = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
        rc = lib.kvc_attend_cache_timed(*args, handles, len(events))
    else:
        rc = lib.kvc_attend_cache(*args)
    if rc != KVC_OK:
        raise KvcError(rc, status_string(rc))


def attention_over_cache(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                         cu_seqlens_q: torch.Tensor, seqlens_k: torch.Tensor,
                         slot_ids: Optional[torch.Tensor] = None,
                         max_seqlen_q: Optional[int] = None, scale: Optional[float] = None,
                         status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Read-only re-attention of packed queries over an appended cache.

    q [total_q, Hq, D]; key_cache [num_slots, Hk, M, D] and value_cache
    [num_slots, Hk, M, Dv] (never written); cu_seqlens_q [B + 1] packing
    offsets; seqlens_k each sequence's total cached length, [B] or cumulative
    [B + 1]; slot_ids [B] cache row per sequence (default row b). Query t of a
    sequence with S queries and K cached positions attends slots
    j <= K - S + t. Returns out [total_q, Hq, Dv]. ``max_seqlen_q`` (the
    largest S) is read from cu_seqlens_q when not given (a device sync).
    """
    for name, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        if t.dtype not in DTYPES or t.dtype != q.dtype:
            raise ValueError(f"{name}: one dtype among float32/bfloat16/float16 is needed")
        if t.device.type != "cuda" or t.device != q.device:
            raise ValueError("attention_over_cache runs on one CUDA device only (no CPU path)")
    if q.dim() != 3 or key_cache.dim() != 4 or value_cache.dim() != 4:
        raise ValueError("q is [total_q, Hq, D]; the caches are [num_slots, Hk, M, D|Dv]")
    total_q, Hq, D = q.shape
    num_slots, Hk, M, Dk = key_cache.shape
    if Dk != D or tuple(value_cache.shape[:3]) != (num_slots, Hk, M):
        raise ValueError("cache shapes do not match q")
    B = cu_seqlens_q.numel() - 1
    if B < 1 or seqlens_k.numel() not in (B, B + 1):
        raise ValueError("cu_seqlens_q is [B + 1]; seqlens_k is [B] or cumulative [B + 1]")
    if Hq % Hk:
        raise ValueError("Hq must be a multiple of Hk")
    if scale is None:
        scale = default_scale(D)
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    Dv = value_cache.shape[-1]
    dims = make_dims(B, Hq, Hk, max(1, int(max_seqlen_q)), D, Dv, M, q.dtype)
    cu = cu_seqlens_q.to(device=q.device, dtype=torch.int32).contiguous()
    kl = seqlens_k.to(device=q.device, dtype=torch.int32).contiguous()
    sl = None if slot_ids is None else slot_ids.to(device=q.device,
                                                   dtype=torch.int32).contiguous()
    out = torch.empty(total_q, Hq, Dv, dtype=q.dtype, device=q.device)
    ws = torch.empty(attend_cache_workspace_bytes(dims), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        attend_cache_into(dims, num_slots, q.contiguous(), key_cache.contiguous(),
                          value_cache.contiguous(), cu, kl, seqlens_k.numel() == B + 1, sl,
                          float(scale), out, ws, status)
    return out


def paged_workspace_bytes(dims: Dims) -> int:
    return int(library().kvc_paged_workspace_bytes(ctypes.byref(dims)))


def step_paged_into(dims: Dims, block_table, query, new_key, new_value, key_pool, value_pool,
                    lengths, append_mask, scale: float, out: dict, workspace: torch.Tensor,
                    status: Optional[torch.Tensor] = None, stream: Optional[int] = None,
                    events: Optional[Sequence] = None) -> None:
    """Enqueue one kvc_step_paged (no checks beyond libkvc's); out holds
    "lengths", "attention" and "context"."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(key_pool.device).cuda_stream
    ws_len = workspace.numel() * workspace.element_size()
    args = [ctypes.byref(dims), int(key_pool.shape[0]), int(key_pool.shape[2]), _p(block_table),
            _p(query), _p(new_key), _p(new_value), _p(key_pool), _p(value_pool), _p(lengths),
            _p(append_mask), ctypes.c_double(scale), _p(out["lengths"]), _p(out["attention"]),
            _p(out["context"]), _p(workspace), ws_len, _p(status), ctypes.c_void_p(stream)]
    if events:
        handles = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
        rc = lib.kvc_step_paged_timed(*args, handles, len(events))
    else:
        rc = lib.kvc_step_paged(*args)
    if rc != KVC_OK:
        raise KvcError(rc, status_string(rc))


def kv_cache_attention_step_paged(query: torch.Tensor, new_key: torch.Tensor,
                                  new_value: torch.Tensor, key_pool: torch.Tensor,
                                  value_pool: torch.Tensor, block_table: torch.Tensor,
                                  lengths: torch.Tensor, append_mask: torch.Tensor,
                                  options: Optional[dict] = None,
                                  status: Optional[torch.Tensor] = None) -> dict:
    """The in-place step on a paged block pool: key_pool [num_blocks, Hk,
    block_size, D] / value_pool [..., Dv] are updated in place, batch row b's
    slot j living in block block_table[b, j // block_size] (capacity
    M = block_table.shape[1] * block_size). Returns {"key_cache": key_pool,
    "value_cache": value_pool, "lengths", "attention", "context"}."""
    if query.dim() != 4 or key_pool.dim() != 4 or value_pool.dim() != 4 or block_table.dim() != 2:
        raise ValueError("query [B,Hq,Q,D], pools [num_blocks,Hk,block_size,D|Dv], table [B,max_blocks]")
    for name, t in (("query", query), ("new_key", new_key), ("new_value", new_value),
                    ("key_pool", key_pool), ("value_pool", value_pool)):
        if t.dtype not in DTYPES or t.dtype != query.dtype:
            raise ValueError(f"{name}: one dtype among float32/bfloat16/float16 is needed")
        if t.device.type != "cuda" or t.device != query.device:
            raise ValueError("the paged step runs on one CUDA device only (no CPU path)")
    if not (key_pool.is_contiguous() and value_pool.is_contiguous()):
        raise ValueError("the pools are updated in place and must be contiguous")
    B, Hq, Q, D = query.shape
    num_blocks, Hk, bs, Dk = key_pool.shape
    Dv = value_pool.shape[-1]
    if Dk != D or tuple(value_pool.shape[:3]) != (num_blocks, Hk, bs) or block_table.shape[0] != B:
        raise ValueError("pool / table shapes do not match the query")
    if tuple(new_key.shape) != (B, Hk, Q, D) or tuple(new_value.shape) != (B, Hk, Q, Dv):
        raise ValueError("new_key / new_value shapes do not match")
    if tuple(append_mask.shape) != (B, Q) or tuple(lengths.shape) != (B,):
        raise ValueError("append_mask is [B, Q] and lengths [B]")
    scale = _scale_from(options, D)
    M = block_table.shape[1] * bs
    dims = make_dims(B, Hq, Hk, Q, D, Dv, M, query.dtype)
    q, nk, nv = (t.contiguous() for t in (query, new_key, new_value))
    tb = block_table.to(device=query.device, dtype=torch.int32).contiguous()
    ln = lengths.to(torch.int64).contiguous()
    mk = append_mask.contiguous()
    mk = mk.view(torch.uint8) if mk.dtype == torch.bool else mk
    out = {"key_cache": key_pool, "value_cache": value_pool,
           "lengths": torch.empty(B, dtype=torch.int64, device=q.device),
           "attention": torch.empty(B, Hq, Q, M, dtype=q.dtype, device=q.device),
           "context": torch.empty(B, Hq, Q, Dv, dtype=q.dtype, device=q.device)}
    ws = torch.empty(max(16, paged_workspace_bytes(dims)), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        step_paged_into(dims, tb, q, nk, nv, key_pool, value_pool, ln, mk, scale, out, ws, status)
    return out
