"""The conventional four-kernel pipeline (projection GEMM, rotary, cache write,
attention; the comparison the fused kernel is measured against) through the C ABI:
against the fp64 oracle on small cases, and against the fused step at full size."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _run_unfused(wl, cache, probe_idx=None):
    s = wl.shape
    w = G.tdev(wl.w, s.act)

    def step(x, pos, view, out, kv_x=None, kv_pos=None, probe=None):
        n_tok = 0 if pos is None else pos.shape[-1]
        n_kv = 0 if kv_pos is None else kv_pos.shape[-1]
        ws = torch.empty(capi.dllm_unfused_workspace_bytes(cache.handle, n_tok, n_kv), dtype=torch.uint8,
                         device="cuda")
        capi.dllm_cache_step_unfused(cache.handle, 0, x, w, pos, view, out, ws, kv_x=kv_x, kv_positions=kv_pos,
                                     probe_kv=probe)

    if wl.pre_x is not None:
        step(None, None, None, None, G.tdev(wl.pre_x, s.act), G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    out = torch.empty_like(x)
    view = G.idev(wl.view, torch.uint8) if wl.view is not None else None
    kv_x = kv_pos = probe = None
    if probe_idx is not None:
        kv_x = G.tdev(wl.probe_rows(probe_idx), s.act)
        kv_pos = G.idev(probe_idx)
        probe = torch.empty((s.batch, probe_idx.shape[1], 2, s.D), dtype=x.dtype, device="cuda")
    elif wl.kv_x is not None:
        kv_x, kv_pos = G.tdev(wl.kv_x, s.act), G.idev(wl.kv_pos)
    step(x, G.idev(wl.positions), view, out, kv_x, kv_pos, probe)
    torch.cuda.synchronize()
    rc, bits = cache.status()
    assert rc == capi.DLLM_OK, f"device status {bits:#x}"
    return out.double().cpu().numpy(), (None if probe is None else probe.double().cpu().numpy())


CASES = [
    ("bf16", "llada8b-b1", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=40, gen_lo=200, fixed_lo=None)),
    ("fp8-refresh", "llada8b-b8-refresh-fp8", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200)),
    ("verify", "llada8b-b16-verify", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200, search=6,
                       tail_slots=8)),
]


@pytest.mark.parametrize("name,workload,kw", CASES, ids=[c[0] for c in CASES])
def test_unfused_matches_oracle(name, workload, kw):
    wl = W.make(workload, **kw)
    cache = G.make_cache(wl)
    out, _ = _run_unfused(wl, cache)
    o_out, ocache, _ = G.run_oracle(wl)
    tol = G.TOL[wl.shape.kv]
    # for an e4m3 cache the pipeline quantises the fp32 rotated value, as the fused kernel
    # and the oracle do, so its codes are checked as theirs are (compare_cache)
    G.compare_cache(cache, ocache, tol)
    G.assert_close(out.reshape(o_out.shape), o_out, tol, f"unfused attention out ({name})")
    if wl.shape.kv == "e4m3":
        m_out = G.run_oracle(wl, model_fp8=True)[0]
        G.assert_close(out.reshape(m_out.shape), m_out, G.FP8_MODEL_TOL, f"unfused out vs the e4m3 model ({name})")


def test_unfused_probes_match_oracle():
    wl = W.make("llada8b-b32-drift", batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200, drift_k=8)
    idx = np.stack([np.arange(8, dtype=np.int32) * 3 for _ in range(3)])
    cache = G.make_cache(wl)
    out, probe = _run_unfused(wl, cache, probe_idx=idx)
    o_out, ocache, o_probe = G.run_oracle(wl, probe_idx=idx)
    G.compare_cache(cache, ocache, G.TOL["bf16"])
    G.assert_close(probe, o_probe, G.TOL["bf16"], "unfused probe K/V")


def test_unfused_agrees_with_fused_at_full_size():
    wl = W.make("llada8b-b32-drift")
    idx = np.stack([np.arange(32, dtype=np.int32) * 7 % 512 for _ in range(wl.shape.batch)])
    c1, c2 = G.make_cache(wl), G.make_cache(wl)
    out_f, probe_f = G.run_gpu(wl, c1, probe_idx=idx)
    out_u, probe_u = _run_unfused(wl, c2, probe_idx=idx)
    # the unfused pipeline rounds the projection to bf16 before rotating: a few bf16 ulps
    G.assert_close(out_u, out_f, 2e-2, "unfused vs fused attention output")
    G.assert_close(probe_u, probe_f, 2e-2, "unfused vs fused probes")
    kv_f, kv_u = c1.kv(0).float(), c2.kv(0).float()  # on the device: 512 MiB each
    written = torch.from_numpy(G.expected_written(wl, probe=True)).cuda()
    err = (kv_u - kv_f).abs()[written].max() / kv_f[written].abs().max()
    assert float(err) <= 2e-2, f"unfused vs fused cache: {float(err):.3g}"
