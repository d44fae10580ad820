"""Full-size workloads through the C ABI, checked against the fp64 oracle on sampled
(sequence, head) pairs plus bit-exact slot sets and top-k indices."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _topk(wl):
    idx = torch.empty((wl.shape.batch, wl.drift_k), dtype=torch.int32, device="cuda")
    capi.dllm_kv_topk(torch.from_numpy(wl.mass).cuda(), torch.from_numpy(wl.block_lo).cuda(), wl.block_len,
                      wl.drift_k, idx)
    return idx


def test_config3_batch32_drift_fullsize():
    wl = W.make("llada8b-b32-drift")
    idx = _topk(wl)
    idx_np = idx.cpu().numpy()
    np.testing.assert_array_equal(idx_np, O.kv_topk(wl.mass, wl.block_lo, wl.block_len, wl.drift_k))
    cache = G.make_cache(wl)
    out, probe = G.run_gpu(wl, cache, probe_idx=idx_np)
    G.check_sampled(wl, cache, out, [(0, 0), (13, 7), (31, 31)], probe_gpu=probe, probe_idx=idx_np)
    # drift for two whole sequences (the cosine spans all heads)
    cos = torch.empty((wl.shape.batch, wl.drift_k, 2), dtype=torch.float32, device="cuda")
    refresh = torch.empty(wl.shape.batch, dtype=torch.int32, device="cuda")
    pk = torch.from_numpy(probe).to(torch.bfloat16).cuda()
    capi.dllm_kv_drift(cache.handle, 0, idx, pk, wl.gamma, cos, refresh)
    g_cos = cos.double().cpu().numpy()
    for b in (5, 30):
        s = wl.shape
        Kc = np.zeros((wl.drift_k, s.D))
        Vc = np.zeros((wl.drift_k, s.D))
        Kp = np.zeros((wl.drift_k, s.D))
        Vp = np.zeros((wl.drift_k, s.D))
        for h in range(s.n_heads):
            _, K, V, _, pr = G.oracle_head(wl, b, h, idx_np)
            sl = slice(h * s.head_dim, (h + 1) * s.head_dim)
            Kc[:, sl], Vc[:, sl] = K[idx_np[b]], V[idx_np[b]]
            Kp[:, sl], Vp[:, sl] = pr
        o_cos = np.array([[O.cosine(Kc[j], Kp[j]), O.cosine(Vc[j], Vp[j])] for j in range(wl.drift_k)])
        G.assert_close(g_cos[b], o_cos, G.TOL["bf16"], f"drift cos b={b}")
    assert set(np.unique(refresh.cpu().numpy())) <= {0, 1}


def test_config4_verify_fullsize():
    wl = W.make("llada8b-b16-verify")
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    G.check_sampled(wl, cache, out, [(0, 3), (9, 20), (15, 31)])


def test_config5_refresh_fp8_fullsize():
    wl = W.make("llada8b-b8-refresh-fp8")
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    G.check_sampled(wl, cache, out, [(0, 0), (4, 11), (7, 31)], exact_diag_tol=0.15)
