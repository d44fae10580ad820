"""Attention under the balanced schedule: full waves of whole (sequence, head, query
chunk) units go round-robin over the SMs, and the units left over after at least one
full wave (fewer than the SMs) are cut into equal pieces of key tiles that all SMs share;
the CTA that completes such a unit (an arrival count per unit, reset by that CTA) merges
the pieces' partial softmax states.  The host picks the piece count that minimises the
most key tiles any CTA runs.  With fewer units than SMs, or an e4m3 cache, units stay
whole and only their keys are split (partial states merged by a second kernel).

Checked here against the fp64 oracle at the usual bounds: a batch one wave past the SM
count (the leftover units in 4 pieces), the Flash-Verify tail (3 pieces of a 9-tile
unit), and for contrast a long cache over few heads and an e4m3 cache (key splits).  The
merge adds the pieces in piece order whichever CTA finishes last, so repeated calls give
bit-identical outputs, which also shows that every arrival count is back at zero after
a call (else the next call would lose its merges and leave Q in the output).
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu

CASES = [
    # 4 units of 32 key tiles, no full wave: keys split 32 ways, merged by a second kernel
    ("long-few-units", "llada8b-b1", dict(batch=1, d_model=512, head_dim=128, max_pos=4000, block=32, gen_lo=3000,
                                          fixed_lo=None)),
    # 160 units of 8 tiles: one wave of whole units, the 12 left over in 4 pieces of 2
    # (10 tiles on the busiest SM instead of 16)
    ("b40-past-sm-count", "llada8b-b1", dict(batch=40, d_model=512, head_dim=128, max_pos=1024, block=32, gen_lo=512,
                                             fixed_lo=None)),
    # Flash-Verify: 9 tiles a unit (the last holds the draft tail), 48 query rows (32 block
    # rows, 16 draft views); the 12 units after the first wave in 3 pieces of 3 tiles
    ("verify-b40", "llada8b-b16-verify", dict(batch=40, d_model=512, head_dim=128, max_pos=1024, block=32, gen_lo=512,
                                              search=16, tail_slots=16)),
    # 100 query rows: two 64-row chunks per (sequence, head) (64 query columns), 320
    # units of 8 tiles, two full waves and the 24 left over in 4 pieces of 2
    ("b40-two-chunks", "llada8b-b1", dict(batch=40, d_model=512, head_dim=128, max_pos=1024, block=100, gen_lo=512,
                                          fixed_lo=None)),
    # e4m3 cache, 4 units of 24 tiles: keys split, partial states merged by a second kernel
    ("e4m3-long", "llada8b-b1", dict(kv="e4m3", batch=1, d_model=512, head_dim=128, max_pos=3072, block=32,
                                     gen_lo=2048, fixed_lo=None)),
]


@pytest.mark.parametrize("name,workload,kw", CASES, ids=[c[0] for c in CASES])
def test_tail_pieces_match_oracle(name, workload, kw):
    wl = W.make(workload, **kw)
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    o_out, ocache, _ = G.run_oracle(wl)
    tol = G.TOL[wl.shape.kv]
    G.assert_close(out.reshape(o_out.shape), o_out, tol, f"attention out ({name})")
    if wl.shape.kv == "e4m3":
        m_out, _, _ = G.run_oracle(wl, model_fp8=True)
        G.assert_close(out.reshape(m_out.shape), m_out, G.FP8_MODEL_TOL, f"out vs the e4m3 model ({name})")


@pytest.mark.parametrize("name,workload,kw", [c for c in CASES if c[0] != "verify-b40"],
                         ids=[c[0] for c in CASES if c[0] != "verify-b40"])
def test_tail_pieces_repeated_calls_bit_identical(name, workload, kw):
    wl = W.make(workload, **kw)
    s = wl.shape
    cache = G.make_cache(wl)
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                         kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    pos = G.idev(wl.positions)
    q = torch.empty_like(x)
    capi.dllm_cache_project(cache.handle, 0, x, w, pos, None, q)
    outs = []
    for _ in range(4):
        o = q.clone()
        capi.dllm_cache_attend(cache.handle, 0, pos, None, o)
        outs.append(o)
    torch.cuda.synchronize()
    rc, bits = cache.status()
    assert rc == capi.DLLM_OK and bits == 0, f"device status {bits:#x}"
    ref = outs[0].view(torch.int16).cpu().numpy()
    assert not np.array_equal(ref, q.view(torch.int16).cpu().numpy()), "output never written"
    for i, o in enumerate(outs[1:], 1):
        np.testing.assert_array_equal(o.view(torch.int16).cpu().numpy(), ref, err_msg=f"call {i}")
