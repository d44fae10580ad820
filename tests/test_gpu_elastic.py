"""The multi-layer step with the depth-wise drift refresh (dllm_elastic_step) through
the C ABI, against the fp64 oracle's elastic_step: per-layer outputs, drift cosines,
refresh flags (exact), every cache slot after the step, and the attention mass."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu

KV = {"bf16": capi.DLLM_BF16, "e4m3": capi.DLLM_E4M3}


def _sigma(B):
    # per sequence, by b % 4: barely drifts; fails at layer 1; fails at layer 0; fails only at
    # the last layer (nothing left to refresh)
    pat = np.array([[0.05, 0.05, 3.0, 0.05], [0.05, 3.0, 3.0, 0.05], [0.05, 3.0, 3.0, 3.0]])
    return pat[:, np.arange(B) % 4]


CASES = [
    ("bf16", dict(batch=4, d_model=256, max_pos=384), True),
    ("e4m3", dict(batch=4, d_model=256, max_pos=384, kv="e4m3"), True),
    # enough refresh tiles for the CTA-pair projection kernel
    ("bf16-pairs", dict(batch=8, d_model=1024, max_pos=512), True),
]


@pytest.mark.parametrize("name,kw,with_mass", CASES, ids=[c[0] for c in CASES])
def test_elastic_step_matches_oracle(name, kw, with_mass):
    B = kw["batch"]
    wl = W.make_elastic(_sigma(B), seed=3, head_dim=128, beta=32, gen_lo=128, k=8, gamma=0.9, **kw)
    s, L = wl.shape, wl.n_layers
    S, D = s.max_pos, s.D
    all_pos = np.tile(np.arange(S, dtype=np.int32), (B, 1))

    # ---- GPU: prefill every layer from x_prev, then one step over the layers
    cache = capi.Cache(L, B, S, s.n_heads, s.head_dim, KV[s.kv], s.rope_theta, 0)
    w = [G.tdev(wl.w[l], s.act) for l in range(L)]
    x_all = [G.tdev(wl.x_all[l], s.act) for l in range(L)]
    for l in range(L):
        capi.dllm_cache_step(cache.handle, l, None, w[l], None, None, None, kv_x=G.tdev(wl.x_prev[l], s.act),
                             kv_positions=G.idev(all_pos))
    out = torch.empty((L, B, wl.beta, D), dtype=torch.bfloat16, device="cuda")
    cos = torch.empty((L, B, wl.k, 2), dtype=torch.float32, device="cuda")
    flags = torch.full((L, B), -7, dtype=torch.int32, device="cuda")
    mass_out = torch.empty((L, B, S), dtype=torch.float32, device="cuda") if with_mass else None
    ws = torch.empty(capi.dllm_elastic_workspace_bytes(cache.handle, wl.beta, wl.k), dtype=torch.uint8, device="cuda")
    capi.dllm_elastic_step(cache.handle, x_all, w, G.idev(wl.win_lo), wl.beta, torch.from_numpy(wl.mass).cuda(),
                           wl.k, wl.gamma, out, cos, flags, ws, mass_out=mass_out)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)

    # ---- oracle: unquantised caches (the tolerance reference); for an e4m3 cache also the
    # oracle's model of the encoding, against which the kernels' own error is held to
    # the bf16 bound
    def oracle(kvm):
        caches = []
        for l in range(L):
            c = O.OracleCache(B, S, 0, s.n_heads, s.head_dim, kv=kvm)
            O.write_rows(c, wl.w[l], wl.x_prev[l], all_pos, s.rope_theta)
            caches.append(c)
        res = O.elastic_step(caches, wl.w, s.rope_theta, wl.x_all, wl.win_lo, wl.beta, wl.mass, wl.k, wl.gamma,
                             with_mass=with_mass)
        return caches, res

    runs = [("oracle", oracle("exact"), G.TOL[s.kv])]
    if s.kv == "e4m3":
        runs.append(("e4m3 model", oracle("e4m3"), G.FP8_MODEL_TOL))
    g_out = out.double().cpu().numpy()
    g_cos = cos.double().cpu().numpy()
    for ref, (caches, (o_out, o_cos, o_flags, o_mass)), tol in runs:
        # the fixture keeps every drift decision far from the threshold
        margin = np.abs(o_cos.min(axis=(2, 3)) - wl.gamma)
        assert margin.min() > 0.02, margin.min()
        assert o_flags.any() and not o_flags.all()
        np.testing.assert_array_equal(flags.cpu().numpy(), o_flags, err_msg=f"refresh flags vs {ref}")
        G.assert_close(g_cos, o_cos, tol, f"drift cos ({name}) vs {ref}")
        for l in range(L):
            G.assert_close(g_out[l], o_out[l], tol, f"attention output layer {l} ({name}) vs {ref}")
            kv = G.gpu_kv(cache, l)
            G.assert_close(kv[:, :S, 0], caches[l].K, tol, f"cache K layer {l} ({name}) vs {ref}")
            G.assert_close(kv[:, :S, 1], caches[l].V, tol, f"cache V layer {l} ({name}) vs {ref}")
            if s.kv == "e4m3" and caches[l].kv == "exact":
                codes, scales = G.gpu_fp8_groups(cache, l)
                exact = np.stack([caches[l].K, caches[l].V], axis=2)
                G.fp8_code_check(codes[:, :S], scales[:, :S], exact, f"cache layer {l} e4m3 codes")
            if with_mass:
                G.assert_close(mass_out[l].double().cpu().numpy(), o_mass[l], min(tol, G.TOL["bf16"]),
                               f"mass layer {l} ({name}) vs {ref}")


def test_elastic_step_rejects_bad_arguments():
    cache = capi.Cache(2, 2, 256, 2, 128, capi.DLLM_BF16, 5e5, 0)
    D = 256
    x = [torch.zeros((2, 256, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    w = [torch.zeros((3 * D, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    win = torch.zeros(2, dtype=torch.int32, device="cuda")
    mass = torch.zeros((2, 2, 256), dtype=torch.float32, device="cuda")
    out = torch.empty((2, 2, 32, D), dtype=torch.bfloat16, device="cuda")
    cos = torch.empty((2, 2, 8, 2), dtype=torch.float32, device="cuda")
    flags = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    need = capi.dllm_elastic_workspace_bytes(cache.handle, 32, 8)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.DllmError):
        capi.dllm_elastic_step(cache.handle, x, w, win, 32, mass, 8, 0.9, out, cos, flags, small)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.DllmError):  # k larger than the candidates outside the window
        capi.dllm_elastic_step(cache.handle, x, w, win, 32, mass, 256 - 31, 0.9, out, cos, flags, ws)
    with pytest.raises(capi.DllmError):  # more layers than the cache holds
        capi.dllm_elastic_step(cache.handle, x * 2, w * 2, win, 32, mass, 8, 0.9, out, cos, flags, ws)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
