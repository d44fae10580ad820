"""Failure handling on the GPU without a fault: a pipeline wait that nothing satisfies
gives up after its time limit, the kernel reports DLLM_DEV_TIMEOUT through the cache's
status word and ends, and the context stays usable for the next step."""
import time

import pytest
import torch

import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    wl = W.make("llada8b-b1", batch=2, d_model=256, head_dim=128, max_pos=256, block=32, gen_lo=128, fixed_lo=None)
    cache = G.make_cache(wl)
    t0 = time.perf_counter()
    capi.dllm_selftest_wait_timeout(cache.handle)
    rc, bits = cache.status()  # synchronises
    dt = time.perf_counter() - t0
    assert rc == capi.DLLM_EDEVICE and bits == capi.DEV_TIMEOUT
    assert 0.5 < dt < 30.0, dt
    assert cache.status() == (capi.DLLM_OK, 0)  # the status read cleared the bit
    # the same context runs an ordinary step afterwards
    out, _ = G.run_gpu(wl, cache)
    o_out, ocache, _ = G.run_oracle(wl)
    G.assert_close(out.reshape(o_out.shape), o_out, G.TOL["bf16"], "step after a timeout")


def test_device_range_errors_are_reported_not_faulted():
    # a position outside [0, max_pos) is skipped by the kernels and reported
    wl = W.make("llada8b-b1", batch=2, d_model=256, head_dim=128, max_pos=256, block=32, gen_lo=128, fixed_lo=None)
    cache = G.make_cache(wl)
    w = G.tdev(wl.w, "bf16")
    x = G.tdev(wl.x, "bf16")
    pos = wl.positions.copy()
    pos[1, 3] = 10_000
    out = torch.empty_like(x)
    capi.dllm_cache_project(cache.handle, 0, x, w, G.idev(pos), None, out)
    rc, bits = cache.status()
    assert rc == capi.DLLM_EDEVICE and bits & capi.DEV_BAD_POSITION
    idx = torch.full((2, 4), 999, dtype=torch.int32, device="cuda")
    probe = torch.zeros((2, 4, 2, wl.shape.D), dtype=torch.bfloat16, device="cuda")
    cos = torch.empty((2, 4, 2), dtype=torch.float32, device="cuda")
    capi.dllm_kv_drift(cache.handle, 0, idx, probe, 0.9, cos)
    rc, bits = cache.status()
    assert rc == capi.DLLM_EDEVICE and bits & capi.DEV_BAD_INDEX
    assert torch.isnan(cos).all()
