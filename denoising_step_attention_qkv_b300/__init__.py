"""Cached attention of one diffusion-LLM denoising step on B300 (sm_103a).

The compute lives in ``libdllmcache.so`` (C ABI declared in ``include/dllm_cache.h``);
``capi`` is its ctypes binding.  Build the library with ``build.build()``.
"""
from . import capi  # noqa: F401
from .capi import (  # noqa: F401
    Cache, DllmError, dllm_cache_alloc, dllm_cache_bytes, dllm_cache_free, dllm_cache_get_layout,
    dllm_cache_status, dllm_cache_step, dllm_cache_project, dllm_cache_attend, dllm_cache_attend_noalloc,
    dllm_cache_step_unfused, dllm_unfused_workspace_bytes, dllm_attention_mass, dllm_selftest_wait_timeout,
    dllm_cache_attend_ragged, dllm_cache_attend_partial, dllm_attend_merge, dllm_kv_drift, dllm_kv_topk, dllm_strerror,
    dllm_elastic_workspace_bytes, dllm_elastic_step,
)
