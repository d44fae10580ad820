"""The step's kernels (launched with programmatic dependent launch) captured into a
CUDA graph and replayed give the same bits as eager launches; so does the multi-layer
step, which synchronises nothing with the host."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _step_state(wl):
    s = wl.shape
    cache = G.make_cache(wl)  # filled first, so that the whole buffer is comparable
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None, kv_x=G.tdev(wl.pre_x, s.act),
                         kv_positions=G.idev(wl.pre_pos))
    k = wl.drift_k
    t = dict(cache=cache, w=w, x=G.tdev(wl.x, s.act), pos=G.idev(wl.positions), mass=torch.from_numpy(wl.mass).cuda(),
             lo=G.idev(wl.block_lo), idx=torch.empty((s.batch, k), dtype=torch.int32, device="cuda"),
             probe=torch.empty((s.batch, k, 2, s.D), dtype=torch.bfloat16, device="cuda"),
             cos=torch.empty((s.batch, k, 2), dtype=torch.float32, device="cuda"),
             ref=torch.empty(s.batch, dtype=torch.int32, device="cuda"))
    t["out"] = torch.empty_like(t["x"])
    t["xp"] = G.tdev(wl.probe_rows(np.tile(np.arange(k, dtype=np.int32), (s.batch, 1))), s.act)
    return t


def _run_step(wl, t, stream):
    capi.dllm_kv_topk(t["mass"], t["lo"], wl.block_len, wl.drift_k, t["idx"], stream)
    capi.dllm_cache_project(t["cache"].handle, 0, t["x"], t["w"], t["pos"], None, t["out"], kv_x=t["xp"],
                            kv_positions=t["idx"], probe_kv=t["probe"], stream=stream)
    capi.dllm_cache_attend(t["cache"].handle, 0, t["pos"], None, t["out"], stream=stream)
    capi.dllm_kv_drift(t["cache"].handle, 0, t["idx"], t["probe"], wl.gamma, t["cos"], t["ref"], stream=stream)


@pytest.mark.parametrize("batch,max_pos", [(4, 300), (40, 256)])
def test_step_graph_replay_matches_eager(batch, max_pos):
    wl = W.make("llada8b-b32-drift", batch=batch, d_model=512, head_dim=128, max_pos=max_pos, gen_lo=128, drift_k=8)
    eager, graphed = _step_state(wl), _step_state(wl)
    st = torch.cuda.current_stream()
    _run_step(wl, eager, st)
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        _run_step(wl, graphed, side)  # warm-up outside the capture (function attributes)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            _run_step(wl, graphed, side)
    st.wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for key in ("idx", "out", "probe", "cos", "ref"):
        assert torch.equal(eager[key], graphed[key]), key
    assert torch.equal(eager["cache"].buf, graphed["cache"].buf)
    assert eager["cache"].status() == (capi.DLLM_OK, 0) and graphed["cache"].status() == (capi.DLLM_OK, 0)


def test_multilayer_step_graph_replay_matches_eager():
    sigma = np.array([[0.05, 3.0, 0.05], [0.05, 3.0, 3.0]])
    wl = W.make_elastic(sigma, seed=4, batch=3, d_model=256, head_dim=128, max_pos=384, beta=32, gen_lo=128, k=8)
    s, L = wl.shape, wl.n_layers
    all_pos = G.idev(np.tile(np.arange(s.max_pos, dtype=np.int32), (s.batch, 1)))
    runs = []
    for mode in ("eager", "graph"):
        cache = capi.Cache(L, s.batch, s.max_pos, s.n_heads, s.head_dim, capi.DLLM_BF16, s.rope_theta, 0)
        w = [G.tdev(wl.w[l], s.act) for l in range(L)]
        xs = [G.tdev(wl.x_all[l], s.act) for l in range(L)]
        for l in range(L):
            capi.dllm_cache_step(cache.handle, l, None, w[l], None, None, None, kv_x=G.tdev(wl.x_prev[l], s.act),
                                 kv_positions=all_pos)
        t = dict(cache=cache, out=torch.empty((L, s.batch, wl.beta, s.D), dtype=torch.bfloat16, device="cuda"),
                 cos=torch.empty((L, s.batch, wl.k, 2), dtype=torch.float32, device="cuda"),
                 flags=torch.empty((L, s.batch), dtype=torch.int32, device="cuda"),
                 mass_out=torch.empty((L, s.batch, s.max_pos), dtype=torch.float32, device="cuda"),
                 ws=torch.empty(capi.dllm_elastic_workspace_bytes(cache.handle, wl.beta, wl.k), dtype=torch.uint8,
                                device="cuda"))
        win, mass = G.idev(wl.win_lo), torch.from_numpy(wl.mass).cuda()

        def run(stream):
            capi.dllm_elastic_step(cache.handle, xs, w, win, wl.beta, mass, wl.k, wl.gamma, t["out"], t["cos"],
                                   t["flags"], t["ws"], mass_out=t["mass_out"], stream=stream)

        if mode == "eager":
            run(torch.cuda.current_stream())
        else:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    run(side)
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
        torch.cuda.synchronize()
        assert cache.status() == (capi.DLLM_OK, 0)
        runs.append(t)
    a, b = runs
    assert a["flags"].any() and not a["flags"].all()
    for key in ("out", "cos", "flags", "mass_out"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["cache"].kv(), b["cache"].kv())


def test_host_staged_step_matches_device_inputs():
    """The end-to-end form of a step: inputs staged in dllm_host_alloc blocks, copied
    in on a side stream, results copied back into host blocks; the same bits as the
    step on device-resident inputs."""
    wl = W.make("llada8b-b32-drift", batch=6, d_model=512, head_dim=128, max_pos=300, gen_lo=128, drift_k=8)
    ref, staged = _step_state(wl), _step_state(wl)
    st = torch.cuda.current_stream()
    _run_step(wl, ref, st)
    keys_in, keys_out = ("x", "xp", "pos", "mass", "lo"), ("out", "cos", "ref", "idx")
    h_in = {k: capi.host_empty(staged[k].shape, staged[k].dtype) for k in keys_in}
    h_out = {k: capi.host_empty(staged[k].shape, staged[k].dtype) for k in keys_out}
    for k in keys_in:
        capi.dllm_host_stage(h_in[k], staged[k].cpu())
        assert h_in[k].is_pinned() and h_in[k].data_ptr() % 16 == 0
        staged[k].fill_(0)
    copy = torch.cuda.Stream()
    copy.wait_stream(st)
    with torch.cuda.stream(copy):
        for k in keys_in:
            staged[k].copy_(h_in[k], non_blocking=True)
    st.wait_stream(copy)
    _run_step(wl, staged, st)
    for k in keys_out:
        h_out[k].copy_(staged[k], non_blocking=True)
    torch.cuda.synchronize()
    for k in keys_out:
        assert torch.equal(h_out[k], ref[k].cpu()), k
    view = h_out["out"][1:3]
    del h_out
    assert torch.equal(view, ref["out"][1:3].cpu())  # a view keeps its block alive
