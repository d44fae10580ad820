"""The no-allocation attention entry point against the ordinary one.

Some callers cannot call cudaMalloc: a serving engine that has already given its whole
device memory budget to its own pool, or a latency-critical loop that cannot take the
device-wide synchronisation an allocation may cause.  They call
dllm_cache_attend_noalloc, whose split-KV scratch is a fixed array inside the library.
It launches the same kernels with the same work split as dllm_cache_attend, so its
output must be bit-identical to that call's, call after call, even though every call
reuses the array left behind by the previous one.

This file is named to be collected last, so a run that stops at its first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _staged(wl):
    """Fill the cache and leave the rotated Q of the query rows in a staging tensor."""
    s = wl.shape
    cache = G.make_cache(wl)
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                         kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    pos = G.idev(wl.positions)
    view = G.idev(wl.view, torch.uint8) if wl.view is not None else None
    q = torch.empty_like(x)
    capi.dllm_cache_project(cache.handle, 0, x, w, pos, view, q)
    return cache, pos, view, q


def _pair(wl):
    cache, pos, view, q = _staged(wl)
    ref = q.clone()
    capi.dllm_cache_attend(cache.handle, 0, pos, view, ref)
    torch.cuda.synchronize()
    return cache, pos, view, q, ref.double().cpu().numpy()


def _noalloc(cache, pos, view, q):
    out = q.clone()
    capi.dllm_cache_attend_noalloc(cache.handle, 0, pos, view, out)
    torch.cuda.synchronize()
    rc, bits = cache.status()
    assert rc == capi.DLLM_OK, f"device status {bits:#x}"
    return out.double().cpu().numpy()


SPLIT_CASES = [
    # LLaDA-8B layer at batch 1: 32 (sequence, head) units of 6 key tiles shared by the
    # CTAs, each unit cut into pieces whose partial states meet in the scratch
    dict(workload="llada8b-b1", kw={}),
    # small batch, 5 key tiles, more than one query chunk, Flash-Verify tail
    dict(workload="llada8b-b16-verify", kw=dict(batch=2, d_model=256, head_dim=128, max_pos=600, block=48, gen_lo=400, search=20,
                        tail_slots=24)),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=["llada8b-b1", "verify-small"])
def test_noalloc_matches_attend_two_calls_in_a_row(case):
    wl = W.make(case["workload"], **case["kw"])
    cache, pos, view, q, ref = _pair(wl)
    for call in range(2):
        np.testing.assert_array_equal(_noalloc(cache, pos, view, q), ref, err_msg=f"no-alloc call {call}")


def test_noalloc_interleaved_workloads_reuse_the_scratch():
    a = _pair(W.make("llada8b-b1", batch=1, d_model=512, head_dim=128, max_pos=900, block=32, gen_lo=512, fixed_lo=None))
    b = _pair(W.make("llada8b-b1", batch=3, d_model=256, head_dim=128, max_pos=333, block=20, gen_lo=200, fixed_lo=None))
    for first, second in ((a, b), (b, a)):
        for case in (first, second):
            cache, pos, view, q, ref = case
            np.testing.assert_array_equal(_noalloc(cache, pos, view, q), ref, err_msg="interleaved no-alloc call")


def test_noalloc_largest_split_fits_the_scratch():
    """The schedule splits units over keys only as far as their partial states fit the
    scratch, so a request with one unit fewer than the SMs (the most split states a plain
    batch makes: every unit split in two) still runs, bit-identical to the ordinary call."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    B = sm - 1  # one head each: fewer units than SMs, every unit split over its keys
    wl = W.make("llada8b-b1", batch=B, d_model=128, head_dim=128, max_pos=384, block=16, gen_lo=256, fixed_lo=None)
    cache, pos, view, q, ref = _pair(wl)
    np.testing.assert_array_equal(_noalloc(cache, pos, view, q), ref, err_msg="largest split")
    np.testing.assert_equal(cache.status()[0], capi.DLLM_OK)
