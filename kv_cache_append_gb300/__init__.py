"""GB300-native autoregressive KV-cache append + causal attention step.

The operation ("Autoregressive KV-cache append and causal attention",
Required behavior) runs in hand-written sm_103a CUDA kernels behind the C ABI
of libkvc.so (include/kvc.h); this package is its thin Python binding.
"""
from .kvc import (DEV_MASK, DEV_OVERFLOW, DEV_TIMEOUT, DTYPES, Dims, KvcError,  # noqa: F401
                  allocate_outputs, attend_cache_into, attend_cache_workspace_bytes,
                  attention_over_cache, check_inputs, default_scale, dims_of,
                  kv_cache_attention_step, kv_cache_attention_step_inplace,
                  kv_cache_attention_step_backward, kv_cache_attention_step_paged,
                  backward_plan_info, backward_workspace_bytes, library, paged_workspace_bytes,
                  step_backward_into,
                  step_paged_into,
                  make_dims, plan_info, plan_info_inplace, selftest_wait_timeout, status_string,
                  step_inplace_into, step_into, workspace_bytes)

__all__ = ["kv_cache_attention_step", "kv_cache_attention_step_inplace",
           "kv_cache_attention_step_paged", "kv_cache_attention_step_backward",
           "attention_over_cache", "KvcError",
           "workspace_bytes", "step_into", "step_inplace_into", "library"]
