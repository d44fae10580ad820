"""Failure handling on the GPU without a fault: a pipeline wait that nothing satisfies
gives up after its time limit, the kernel reports DLLM_DEV_TIMEOUT through the cache's
status word and ends, and the context stays usable for the next step; out-of-range
device indices are reported, not faulted; a device allocation that fails (made to
fail by the library's self-test hook) returns DLLM_EOOM and leaks nothing."""
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


@pytest.mark.parametrize("owned", [True, False], ids=["library-owned", "caller-buffer"])
def test_allocation_failure_returns_eoom_and_releases_everything(owned):
    # every device allocation of dllm_cache_alloc is made to fail in turn (the K/V buffer
    # when the library owns it, the rotary table, the status word, the drift counters,
    # the fused drift workspace, the split-KV workspace and its arrival counts); each attempt must return
    # DLLM_EOOM with a NULL handle and give back what it had allocated before the failure
    import ctypes
    L = capi.lib()
    B, S, H = 4, 4096, 8  # 64 MiB of K/V: a leak of it would show in the free memory
    ext = None if owned else torch.empty(capi.dllm_cache_bytes(capi.dllm_cache_desc(
        1, B, S, 0, H, 128, capi.DLLM_BF16, 1e4, None, 0)), dtype=torch.uint8, device="cuda")
    desc = capi.dllm_cache_desc(1, B, S, 0, H, 128, capi.DLLM_BF16, 1e4,
                                None if owned else ext.data_ptr(), 0 if owned else ext.numel())
    n_allocs = 7 if owned else 6
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for nth in range(1, n_allocs + 1):
        capi.dllm_selftest_fail_alloc(nth)
        h = ctypes.c_void_p(1)
        assert L.dllm_cache_alloc(ctypes.byref(desc), ctypes.byref(h)) == capi.DLLM_EOOM, nth
        assert h.value is None
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] >= free0 - (4 << 20), f"memory kept after failing allocation {nth}"
    # the hook fired each time: one more allocation than the call makes never fails
    capi.dllm_selftest_fail_alloc(n_allocs + 1)
    h = ctypes.c_void_p()
    assert L.dllm_cache_alloc(ctypes.byref(desc), ctypes.byref(h)) == capi.DLLM_OK and h.value
    capi.dllm_selftest_fail_alloc(0)
    assert L.dllm_cache_free(h) == capi.DLLM_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (4 << 20)
