"""GB300-native autoregressive KV-cache append + causal attention step.

The operation ("Autoregressive KV-cache append and causal attention",
Required behavior) runs in hand-written sm_103a CUDA kernels behind the C ABI
of libkvc.so (include/kvc.h); this package is its thin Python binding.
"""
from .kvc import (DEV_MASK, DEV_OVERFLOW, DEV_TIMEOUT, DTYPES, Dims, KvcError,  # noqa: F401
                  allocate_outputs, check_inputs, default_scale, dims_of,
                  kv_cache_attention_step, library, make_dims, plan_info, status_string,
                  step_into, workspace_bytes)

__all__ = ["kv_cache_attention_step", "KvcError", "workspace_bytes", "step_into", "library"]
