"""Per-position attention mass (what the next step's top-k reads) through the C ABI,
against the fp64 oracle's definition on small cases and on sampled sequences of the
batch-32 LLaDA-8B workload."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _gpu_mass(wl, cache):
    s = wl.shape
    w = G.tdev(wl.w, s.act)
    if wl.pre_x is not None:
        capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                             kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    pos = G.idev(wl.positions)
    view = G.idev(wl.view, torch.uint8) if wl.view is not None else None
    q = torch.empty_like(x)
    capi.dllm_cache_project(cache.handle, 0, x, w, pos, view, q)
    mass = torch.full((s.batch, s.max_pos), float("nan"), dtype=torch.float32, device="cuda")
    capi.dllm_attention_mass(cache.handle, 0, pos, view, q, mass)
    out = q.clone()
    capi.dllm_cache_attend(cache.handle, 0, pos, view, out)  # the step goes on as usual
    torch.cuda.synchronize()
    rc, bits = cache.status()
    assert rc == capi.DLLM_OK, f"device status {bits:#x}"
    return mass.double().cpu().numpy(), out.double().cpu().numpy()


def _oracle_mass(wl, model_fp8=False):
    """The oracle's mass over its unquantised cache, or over its model of the e4m3
    encoding (model_fp8)."""
    s = wl.shape
    kv = "e4m3" if (s.kv == "e4m3" and model_fp8) else "exact"
    cache = O.OracleCache(s.batch, s.max_pos, s.tail_slots, s.n_heads, s.head_dim, kv=kv)
    if wl.pre_x is not None:
        O.write_rows(cache, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    slots = np.stack([O.row_slots(wl.positions[b], None if wl.view is None else wl.view[b], s.max_pos)
                      for b in range(s.batch)])
    q = O.write_rows(cache, wl.w, wl.x, wl.positions, s.rope_theta, slots)
    return O.attention_mass(cache, q, wl.positions, wl.view)


CASES = [
    ("plain", "llada8b-b1", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=40, gen_lo=200, fixed_lo=None)),
    ("two-chunks", "llada8b-b1", dict(batch=2, d_model=256, head_dim=128, max_pos=400, block=100, gen_lo=200, fixed_lo=None)),
    ("verify", "llada8b-b16-verify", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200, search=6,
                       tail_slots=8)),
    # e4m3 caches: codes times group scales (32 and 48 query columns)
    ("e4m3", "llada8b-b1", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=40, gen_lo=200, fixed_lo=None,
                                kv="e4m3")),
    ("e4m3-verify", "llada8b-b16-verify", dict(batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200,
                                               search=6, tail_slots=8, kv="e4m3")),
]


@pytest.mark.parametrize("name,workload,kw", CASES, ids=[c[0] for c in CASES])
def test_mass_matches_oracle(name, workload, kw):
    wl = W.make(workload, **kw)
    cache = G.make_cache(wl)
    mass, _ = _gpu_mass(wl, cache)
    G.assert_close(mass, _oracle_mass(wl), G.TOL[wl.shape.kv], f"attention mass ({name})")
    if wl.shape.kv == "e4m3":
        G.assert_close(mass, _oracle_mass(wl, model_fp8=True), G.FP8_MODEL_TOL,
                       f"attention mass vs the e4m3 model ({name})")


def test_mass_fullsize_sampled_sequences():
    wl = W.make("llada8b-b32-drift")
    s = wl.shape
    cache = G.make_cache(wl)
    mass, _ = _gpu_mass(wl, cache)
    assert np.all(np.isfinite(mass))
    # every query's weights sum to one over the regular slots (no views here)
    np.testing.assert_allclose(mass.sum(axis=1), s.n_heads * wl.x.shape[1], rtol=2e-3)
    for b in (0, 19):
        ref = np.zeros(s.max_pos)
        for h in range(s.n_heads):
            _, K, _, written, _ = G.oracle_head(wl, b, h)
            qh, _, _ = O.project_head(wl.x[b], wl.w, s.n_heads, h)
            qh = O.rope(qh[:, None, :], wl.positions[b], s.rope_theta)
            ref += O.attention_weights(qh, K[:, None, :]).sum(axis=(0, 1))[:s.max_pos]
        G.assert_close(mass[b], ref, G.TOL["bf16"], f"attention mass (b={b})")
