"""fp64 CPU oracle for the autoregressive KV-cache append + causal attention step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``kv_cache_append_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``kvc_oracle.c`` (plain C loops in double precision,
written from the page "Autoregressive KV-cache append and causal attention",
Required behavior). This module only compiles that file with gcc, marshals
arrays with ctypes and shapes the results.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kvc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvc_oracle.so")

DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
FLAG_OVERFLOW = 1
FLAG_MASK = 2


def compile_library(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: one C file to one shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``kvc_oracle.c`` into ``libkvc_oracle.so`` next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_library(SOURCE, _LIB_PATH)


def _host(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu").contiguous()


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def default_scale(D: int) -> float:
    """Positive default scale 1/sqrt(D), D the query/key width."""
    return 1.0 / math.sqrt(D)


def _dims(query, key_cache, value_cache):
    B, Hq, Q, D = query.shape
    _, Hk, M, _ = key_cache.shape
    Dv = value_cache.shape[-1]
    return B, Hq, Hk, Q, D, Dv, M


def _scale(options, D):
    options = dict(options or {})
    scale = float(options.pop("scale", default_scale(D)))
    if options:
        raise ValueError(f"unknown option keys: {sorted(options)}")
    return scale


class Oracle:
    """One loaded build of ``kvc_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        lib.kvo_step.restype = ctypes.c_int
        lib.kvo_step.argtypes = [ctypes.c_int] + [i64] * 7 + [vp] * 7 + [dbl] + [vp] * 7
        lib.kvo_rows.restype = ctypes.c_int
        lib.kvo_rows.argtypes = [ctypes.c_int] + [i64] * 7 + [vp] * 7 + [dbl, vp, i64] + [vp] * 3
        lib.kvo_widen_n.restype = None
        lib.kvo_widen_n.argtypes = [ctypes.c_int, vp, i64, vp]
        lib.kvo_threads.restype = ctypes.c_int
        lib.kvo_threads.argtypes = []
        lib.kvo_attend_cache.restype = ctypes.c_int
        lib.kvo_attend_cache.argtypes = [ctypes.c_int] + [i64] * 7 + [vp] * 6 + [dbl] + [vp] * 3
        lib.kvo_step_backward.restype = ctypes.c_int
        lib.kvo_step_backward.argtypes = ([ctypes.c_int] + [i64] * 7 + [vp] * 7 + [dbl] +
                                          [vp] * 11)
        self.lib = lib

    def threads(self) -> int:
        """OpenMP threads the oracle uses."""
        return int(self.lib.kvo_threads())

    def widen(self, t: torch.Tensor) -> np.ndarray:
        """Exact widening of an fp32/bf16/fp16 tensor to float64 by the oracle's decoder."""
        h = _host(t)
        out = np.empty(h.numel(), dtype=np.float64)
        self.lib.kvo_widen_n(DTYPE_CODES[h.dtype], _ptr(h), h.numel(), out.ctypes.data)
        return out.reshape(tuple(h.shape))

    def step(self, query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
             options: dict | None = None) -> dict:
        """The whole step on the CPU in fp64.

        Returns key_cache / value_cache (input dtype, the bytes the step
        leaves), lengths (int64), attention [B,Hq,Q,M] and context
        [B,Hq,Q,Dv] as float64 numpy arrays, and flags [B] (1 = overflow,
        2 = non-prefix mask; a flagged row appends nothing).
        """
        q, nk, nv, kc, vc = (_host(x) for x in (query, new_key, new_value, key_cache,
                                                 value_cache))
        B, Hq, Hk, Q, D, Dv, M = _dims(q, kc, vc)
        scale = _scale(options, D)
        ln = _host(lengths).to(torch.int64)
        mk = _host(append_mask).to(torch.uint8)
        out_k = torch.empty_like(kc)
        out_v = torch.empty_like(vc)
        out_len = torch.empty(B, dtype=torch.int64)
        att = np.zeros((B, Hq, Q, M), dtype=np.float64)
        ctx = np.zeros((B, Hq, Q, Dv), dtype=np.float64)
        flags = np.zeros(B, dtype=np.int32)
        work = np.empty(max(1, self.threads()) * max(1, M), dtype=np.float64)
        self.lib.kvo_step(DTYPE_CODES[q.dtype], B, Hq, Hk, Q, D, Dv, M, _ptr(q), _ptr(nk),
                          _ptr(nv), _ptr(kc), _ptr(vc), _ptr(ln), _ptr(mk), scale, _ptr(out_k),
                          _ptr(out_v), _ptr(out_len), att.ctypes.data, ctx.ctypes.data,
                          flags.ctypes.data, work.ctypes.data)
        return {"key_cache": out_k, "value_cache": out_v, "lengths": out_len,
                "attention": att, "context": ctx, "flags": flags}

    def rows(self, query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
             rows_bht, options: dict | None = None):
        """Attention rows [n, M] and context rows [n, Dv] (float64) for the listed (b, h, t)."""
        q, nk, nv, kc, vc = (_host(x) for x in (query, new_key, new_value, key_cache,
                                                 value_cache))
        B, Hq, Hk, Q, D, Dv, M = _dims(q, kc, vc)
        scale = _scale(options, D)
        ln = _host(lengths).to(torch.int64)
        mk = _host(append_mask).to(torch.uint8)
        idx = np.ascontiguousarray(np.asarray(rows_bht, dtype=np.int64).reshape(-1, 3))
        n = idx.shape[0]
        att = np.zeros((n, M), dtype=np.float64)
        ctx = np.zeros((n, Dv), dtype=np.float64)
        work = np.empty(max(1, self.threads()) * max(1, M), dtype=np.float64)
        self.lib.kvo_rows(DTYPE_CODES[q.dtype], B, Hq, Hk, Q, D, Dv, M, _ptr(q), _ptr(nk),
                          _ptr(nv), _ptr(kc), _ptr(vc), _ptr(ln), _ptr(mk), scale,
                          idx.ctypes.data, n, att.ctypes.data, ctx.ctypes.data,
                          work.ctypes.data)
        return att, ctx


    def attend_cache(self, q, cache_key, cache_value, cu_seqlens_q, seqlens_k, slot_ids=None,
                     scale: float | None = None):
        """Read-only re-attention of packed queries q [total_q, Hq, D] over the
        cache rows slot_ids[b] (default b) of cache_key [num_slots, Hk, M, D] /
        cache_value [num_slots, Hk, M, Dv]: out [total_q, Hq, Dv] float64 and
        flags [B] (1 = sequence outside the contract, zero rows)."""
        qh, kc, vc = (_host(x) for x in (q, cache_key, cache_value))
        total_q, Hq, D = qh.shape
        num_slots, Hk, M, _ = kc.shape
        Dv = vc.shape[-1]
        cu = _host(cu_seqlens_q).to(torch.int32)
        B = cu.numel() - 1
        kl = _host(seqlens_k).to(torch.int32)
        sl = None if slot_ids is None else _host(slot_ids).to(torch.int32)
        if scale is None:
            scale = default_scale(D)
        out = np.zeros((total_q, Hq, Dv), dtype=np.float64)
        flags = np.zeros(B, dtype=np.int32)
        work = np.empty(max(1, self.threads()) * max(1, M), dtype=np.float64)
        self.lib.kvo_attend_cache(DTYPE_CODES[qh.dtype], B, Hq, Hk, D, Dv, M, num_slots,
                                  _ptr(qh), _ptr(kc), _ptr(vc), _ptr(cu), _ptr(kl),
                                  None if sl is None else _ptr(sl), float(scale),
                                  out.ctypes.data, flags.ctypes.data, work.ctypes.data)
        return out, flags


    def step_backward(self, query, new_key, new_value, key_cache, value_cache, lengths,
                      append_mask, d_key_cache=None, d_value_cache=None, d_attention=None,
                      d_context=None, options: dict | None = None) -> dict:
        """Gradients of the step's outputs (key_cache, value_cache, attention,
        context) with respect to query, new_key, new_value, key_cache and
        value_cache, given the gradients reaching those outputs (tensors in
        the inputs' dtype, or None for zero). Returns float64 numpy arrays
        d_query, d_new_key, d_new_value, d_key_cache, d_value_cache and flags."""
        q, nk, nv, kc, vc = (_host(x) for x in (query, new_key, new_value, key_cache,
                                                 value_cache))
        B, Hq, Hk, Q, D, Dv, M = _dims(q, kc, vc)
        scale = _scale(options, D)
        ln = _host(lengths).to(torch.int64)
        mk = _host(append_mask).to(torch.uint8)
        grads = [None if g is None else _host(g).to(q.dtype)
                 for g in (d_key_cache, d_value_cache, d_attention, d_context)]
        out = {"d_query": np.zeros((B, Hq, Q, D)), "d_new_key": np.zeros((B, Hk, Q, D)),
               "d_new_value": np.zeros((B, Hk, Q, Dv)), "d_key_cache": np.zeros((B, Hk, M, D)),
               "d_value_cache": np.zeros((B, Hk, M, Dv))}
        flags = np.zeros(B, dtype=np.int32)
        work = np.empty(max(1, self.threads()) * 3 * max(1, M), dtype=np.float64)
        self.lib.kvo_step_backward(
            DTYPE_CODES[q.dtype], B, Hq, Hk, Q, D, Dv, M, _ptr(q), _ptr(nk), _ptr(nv), _ptr(kc),
            _ptr(vc), _ptr(ln), _ptr(mk), scale,
            *(None if g is None else _ptr(g) for g in grads),
            *(out[k].ctypes.data for k in ("d_query", "d_new_key", "d_new_value", "d_key_cache",
                                           "d_value_cache")),
            flags.ctypes.data, work.ctypes.data)
        out["flags"] = flags
        return out

    def step_paged(self, query, new_key, new_value, key_pool, value_pool, block_table,
                   lengths, append_mask, options: dict | None = None) -> dict:
        """The step on a paged block pool ("ClikaRT::ops::attention_over_cache":
        a paged block pool [num_blocks, H_kv, block_size, D] with a rank-2
        [B, max_blocks] block table). Batch row b's logical cache slot j lives in
        block block_table[b, j // block_size], row j % block_size; its capacity
        is M = max_blocks * block_size. By definition the step on the pool is the
        step (kvo_step) on each row's logical cache, gathered through the table,
        with the updated rows written back through it: the gather and scatter are
        plain indexing, the step is the pinned one. A row whose table entries for
        the blocks it would touch (slots [0, length + n)) fall outside
        [0, num_blocks) appends nothing, gets zero query rows and flag 1, like a
        capacity overflow. Blocks not written keep their bytes.

        Returns the pool after the step (key_pool, value_pool), lengths,
        attention [B,Hq,Q,M], context [B,Hq,Q,Dv] (float64) and flags [B].
        """
        kp, vp = _host(key_pool), _host(value_pool)
        table = _host(block_table).to(torch.int64)
        num_blocks, Hk, bs, D = kp.shape
        Dv = vp.shape[-1]
        B, max_blocks = table.shape
        M = max_blocks * bs
        ln = _host(lengths).to(torch.int64)
        mk = _host(append_mask).to(torch.bool)
        Q = mk.shape[1]
        # rows whose needed blocks are outside the pool: append nothing (n = 0)
        n_pref = torch.zeros(B, dtype=torch.int64)
        for b in range(B):
            n = 0
            while n < Q and bool(mk[b, n]):
                n += 1
            n_pref[b] = n
        bad = torch.zeros(B, dtype=torch.bool)
        for b in range(B):
            L, n = int(ln[b]), int(n_pref[b])
            if L < 0 or L + n > M or bool(mk[b, n:].any()):
                continue  # outside the step's contract: the step flags them and appends nothing
            last = (L + n + bs - 1) // bs if n > 0 else 0
            if last and bool(((table[b, :last] < 0) | (table[b, :last] >= num_blocks)).any()):
                bad[b] = True
        mk_eff = mk.clone()
        mk_eff[bad] = False
        # gather each row's logical cache (blocks outside the pool read as zeros; never used)
        safe = table.clamp(0, num_blocks - 1)
        kc = kp[safe].permute(0, 2, 1, 3, 4).reshape(B, Hk, M, D)
        vc = vp[safe].permute(0, 2, 1, 3, 4).reshape(B, Hk, M, Dv)
        ref = self.step(query, new_key, new_value, kc, vc, ln, mk_eff, options)
        ref["flags"] = ref["flags"] | np.where(bad.numpy(), 1, 0).astype(np.int32)
        # write back only the appended rows, through the table
        out_k, out_v = kp.clone(), vp.clone()
        nk_, nv_ = _host(new_key), _host(new_value)
        counts = mk_eff.to(torch.int64).cumprod(1).sum(1)
        for b in range(B):
            L, n = int(ln[b]), int(counts[b])
            if ref["flags"][b] or n == 0:
                continue
            for t in range(n):
                j = L + t
                blk, row = int(table[b, j // bs]), j % bs
                out_k[blk, :, row] = nk_[b, :, t]
                out_v[blk, :, row] = nv_[b, :, t]
        ref["key_cache"], ref["value_cache"] = out_k, out_v
        return ref


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def widen(t):
    return default().widen(t)


def step(*args, **kw):
    return default().step(*args, **kw)


def attend_cache(*args, **kw):
    return default().attend_cache(*args, **kw)


def step_paged(*args, **kw):
    return default().step_paged(*args, **kw)


def rows(*args, **kw):
    return default().rows(*args, **kw)


def step_backward(*args, **kw):
    return default().step_backward(*args, **kw)
