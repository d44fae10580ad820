"""CUDA path vs fp64 oracle on identical seeded inputs, through the C ABI.

Bounds (max|gpu - oracle| <= tol * max|oracle|): 1e-4 fp32, 2e-2 bf16, 6e-2 FP8 cache,
always against the oracle's unquantised cache.  For an FP8 cache the e4m3 codes are
also checked against the oracle's quantisation (equal except at rounding ties) and the
outputs against the oracle's model of the encoding at the bf16 bound.  Slot sets and
top-k indices are compared bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _check_step(wl, probe_idx=None):
    """Returns (cache, out, probe, oracle cache, oracle probe, oracle e4m3-model cache or None)."""
    cache = G.make_cache(wl)
    out, probe = G.run_gpu(wl, cache, probe_idx)
    o_out, ocache, o_probe = G.run_oracle(wl, probe_idx)
    tol = G.TOL[wl.shape.kv]
    G.compare_cache(cache, ocache, tol)
    G.assert_close(out.reshape(o_out.shape), o_out, tol, "attention out")
    mcache = None
    if wl.shape.kv == "e4m3":
        m_out, mcache, _ = G.run_oracle(wl, probe_idx, model_fp8=True)
        G.assert_close(out.reshape(m_out.shape), m_out, G.FP8_MODEL_TOL, "attention out vs the e4m3 model")
    if probe_idx is not None:
        G.assert_close(probe, o_probe, G.TOL[wl.shape.act], "probe K/V")
    return cache, out, probe, ocache, o_probe, mcache


# ------------------------------------------------------------------------------ fp32
def test_config1_tiny_f32_full():
    _check_step(W.make("tiny-f32"))


def test_f32_ragged_small():
    wl = W.make("tiny-f32", batch=3, d_model=192, head_dim=64, max_pos=77, block=5, gen_lo=30, fixed_lo=None)
    _check_step(wl)


# ------------------------------------------------------------------------------ bf16
SMALL_BF16 = [
    # B, D, S, block: ragged GEMM row tiles, ragged key tile, split-KV + combine
    dict(batch=3, d_model=512, max_pos=300, block=40, gen_lo=200),
    # 128-key tiles exactly, one 32-row chunk, splits
    dict(batch=2, d_model=256, max_pos=256, block=32, gen_lo=128),
    # enough tiles for the 256-wide GEMM tile, 5 key tiles
    dict(batch=4, d_model=1024, max_pos=640, block=32, gen_lo=512),
    # many units: no key split
    dict(batch=40, d_model=512, max_pos=200, block=16, gen_lo=128),
    # more than one 64-query chunk
    dict(batch=2, d_model=256, max_pos=400, block=100, gen_lo=200),
    # 156 tiles of 128 x 256 on 148 SMs: the 8 left over run as 128-column halves
    dict(batch=52, d_model=1024, max_pos=160, block=32, gen_lo=128),
]


@pytest.mark.parametrize("kw", SMALL_BF16, ids=[f"B{k['batch']}-D{k['d_model']}-S{k['max_pos']}-n{k['block']}" for k in SMALL_BF16])
def test_bf16_step_small(kw):
    wl = W.make("llada8b-b1", head_dim=128, fixed_lo=None, **kw)
    _check_step(wl)


def test_bf16_config2_full():
    _check_step(W.make("llada8b-b1"))


# ------------------------------------------------------------------------------ FP8
def test_fp8_refresh_small():
    # full-sequence K/V refresh into an e4m3 cache, then the block attends over it
    wl = W.make("llada8b-b8-refresh-fp8", batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200)
    _check_step(wl)


def test_fp8_prefill_then_step_small():
    wl = W.make("llada8b-b1", kv="e4m3", batch=2, d_model=256, head_dim=128, max_pos=400, block=40, gen_lo=300, fixed_lo=None)
    _check_step(wl)


def test_fp8_more_than_one_chunk():
    # 100 query rows: two chunks of 64 columns, the widest query width, over an e4m3 cache
    wl = W.make("llada8b-b1", kv="e4m3", batch=2, d_model=256, head_dim=128, max_pos=400, block=100, gen_lo=200,
                fixed_lo=None)
    _check_step(wl)


def test_fp8_verify_small():
    wl = W.make("llada8b-b16-verify", kv="e4m3", batch=3, d_model=256, head_dim=128, max_pos=300, block=16, gen_lo=200, search=6,
                tail_slots=8)
    _check_step(wl)


def test_fp8_verify_48_rows():
    # the Flash-Verify width of 48 query columns (32 block rows, 16 draft views) over an
    # e4m3 cache: views, two softmax warpgroups and the converters together
    wl = W.make("llada8b-b16-verify", kv="e4m3", batch=3, d_model=256, head_dim=128, max_pos=300, block=32, gen_lo=200,
                search=16, tail_slots=16)
    assert wl.x.shape[1] == 48
    _check_step(wl)


# ---------------------------------------------------------------------- Flash-Verify
def test_verify_small():
    wl = W.make("llada8b-b16-verify", batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200, search=6, tail_slots=8)
    _check_step(wl)


def test_verify_draft_equals_mask_views_identical():
    wl = W.make("llada8b-b16-verify", batch=2, d_model=256, head_dim=128, max_pos=200, block=16, gen_lo=128, search=5, tail_slots=8)
    nb = wl.block_len
    for b in range(wl.shape.batch):
        for t in range(nb, wl.x.shape[1]):
            twin = np.where((wl.positions[b, :nb] == wl.positions[b, t]) & (wl.view[b, :nb] == W.VIEW_MASK))[0][0]
            wl.x[b, t] = wl.x[b, twin]
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    for b in range(wl.shape.batch):
        for t in range(nb, wl.x.shape[1]):
            twin = np.where((wl.positions[b, :nb] == wl.positions[b, t]) & (wl.view[b, :nb] == W.VIEW_MASK))[0][0]
            np.testing.assert_array_equal(out[b, t], out[b, twin])


# ----------------------------------------------------------------------- drift, top-k
def _topk_gpu(wl):
    mass = torch.from_numpy(wl.mass).cuda()
    lo = torch.from_numpy(wl.block_lo).cuda()
    idx = torch.empty((wl.shape.batch, wl.drift_k), dtype=torch.int32, device="cuda")
    capi.dllm_kv_topk(mass, lo, wl.block_len, wl.drift_k, idx)
    return idx.cpu().numpy()


def test_topk_bit_exact_with_ties():
    wl = W.make("llada8b-b32-drift", batch=5, d_model=256, head_dim=128, max_pos=1000, block=32, gen_lo=512, drift_k=32)
    wl.mass[1, 100:140] = 0.25  # ties across the cut
    wl.mass[2, :] = 0.0         # all equal
    wl.mass[3, wl.block_lo[3]:wl.block_lo[3] + 32] = 10.0  # block dominates but is excluded
    np.testing.assert_array_equal(_topk_gpu(wl), O.kv_topk(wl.mass, wl.block_lo, wl.block_len, wl.drift_k))


@pytest.mark.parametrize("k,n_pos", [(7, 5000), (32, 4100), (40, 700), (1, 33)])
def test_topk_sizes_bit_exact(k, n_pos):
    # k <= 32 merges per-warp top-32 lists (several rounds per warp above 1024
    # positions); larger k sorts every candidate
    wl = W.make("llada8b-b32-drift", batch=4, d_model=256, head_dim=128, max_pos=n_pos, block=min(32, n_pos - k - 1),
                gen_lo=0, drift_k=k)
    wl.mass[0, ::3] = wl.mass[0, 1]  # many ties
    np.testing.assert_array_equal(_topk_gpu(wl), O.kv_topk(wl.mass, wl.block_lo, wl.block_len, wl.drift_k))


DRIFT_CASES = [
    ("bf16", dict(d_model=512, head_dim=128, act="bf16", kv="bf16")),
    ("f32", dict(d_model=192, head_dim=64, act="f32", kv="f32")),
    ("e4m3", dict(d_model=512, head_dim=128, act="bf16", kv="e4m3")),
]


@pytest.mark.parametrize("name,kw", DRIFT_CASES, ids=[c[0] for c in DRIFT_CASES])
def test_drift_cache_types(name, kw):
    wl = W.make("llada8b-b32-drift", batch=5, max_pos=300, block=16, gen_lo=200, drift_k=24, **kw)
    idx = _topk_gpu(wl)
    cache, out, probe, ocache, o_probe, mcache = _check_step(wl, probe_idx=idx)
    ptype = torch.float32 if kw["act"] == "f32" else torch.bfloat16
    cos = torch.empty((wl.shape.batch, wl.drift_k, 2), dtype=torch.float32, device="cuda")
    refresh = torch.full((wl.shape.batch,), 7, dtype=torch.int32, device="cuda")
    pk = torch.from_numpy(probe).to(ptype).cuda()
    for _ in range(2):  # the per-sequence arrival counters reset themselves
        capi.dllm_kv_drift(cache.handle, 0, G.idev(idx), pk, 0.9, cos, refresh)
        o_cos = O.kv_drift(ocache, idx, o_probe)
        G.assert_close(cos.double().cpu().numpy(), o_cos, G.TOL[kw["kv"]], f"drift cos ({name})")
        if mcache is not None:
            G.assert_close(cos.double().cpu().numpy(), O.kv_drift(mcache, idx, o_probe), G.FP8_MODEL_TOL,
                           f"drift cos vs the e4m3 model ({name})")
        g_min = cos.cpu().numpy().reshape(wl.shape.batch, -1).min(1)
        np.testing.assert_array_equal(refresh.cpu().numpy(), (g_min < np.float32(0.9)).astype(np.int32))


def test_drift_refresh_flags_both_ways():
    # sequence 0 probes equal their cached tokens (cos = 1, no refresh); sequence 1 gets
    # unrelated probes (cos near 0, refresh)
    wl = W.make("llada8b-b32-drift", batch=2, d_model=256, head_dim=128, max_pos=200, block=16, gen_lo=128, drift_k=8)
    idx = _topk_gpu(wl)
    cache, out, probe, ocache, o_probe, _ = _check_step(wl, probe_idx=idx)
    kv = G.gpu_kv(cache)  # [B][slots][2][H][hd]
    probe = probe.copy()
    for j in range(wl.drift_k):
        probe[0, j] = kv[0, idx[0, j]].reshape(2, -1)
    probe[1] = np.random.default_rng(5).standard_normal(probe[1].shape)
    pk = torch.from_numpy(probe).to(torch.bfloat16).cuda()
    cos = torch.empty((2, wl.drift_k, 2), dtype=torch.float32, device="cuda")
    refresh = torch.empty(2, dtype=torch.int32, device="cuda")
    capi.dllm_kv_drift(cache.handle, 0, G.idev(idx), pk, 0.9, cos, refresh)
    c = cos.cpu().numpy()
    assert np.all(np.abs(c[0] - 1.0) < 1e-3) and np.all(np.abs(c[1]) < 0.2)
    np.testing.assert_array_equal(refresh.cpu().numpy(), [0, 1])


def test_drift_small():
    wl = W.make("llada8b-b32-drift", batch=3, d_model=512, head_dim=128, max_pos=300, block=16, gen_lo=200, drift_k=8)
    idx = _topk_gpu(wl)
    np.testing.assert_array_equal(idx, O.kv_topk(wl.mass, wl.block_lo, wl.block_len, wl.drift_k))
    cache, out, probe, ocache, o_probe, _ = _check_step(wl, probe_idx=idx)
    cos = torch.empty((wl.shape.batch, wl.drift_k, 2), dtype=torch.float32, device="cuda")
    refresh = torch.empty(wl.shape.batch, dtype=torch.int32, device="cuda")
    capi.dllm_kv_drift(cache.handle, 0, G.idev(idx), torch.from_numpy(probe).to(torch.bfloat16).cuda(), 0.9, cos,
                       refresh)
    o_cos = O.kv_drift(ocache, idx, o_probe)
    G.assert_close(cos.double().cpu().numpy(), o_cos, G.TOL["bf16"], "drift cos")
    g_cos = cos.cpu().numpy().reshape(wl.shape.batch, -1)
    # the flag is the kernel's own fp32 decision; away from the threshold it must match the oracle's
    np.testing.assert_array_equal(refresh.cpu().numpy(), (g_cos.min(1) < np.float32(0.9)).astype(np.int32))
    o_min = o_cos.reshape(wl.shape.batch, -1).min(1)
    far = np.abs(o_min - 0.9) > 1e-2
    np.testing.assert_array_equal(refresh.cpu().numpy()[far], (o_min[far] < 0.9).astype(np.int32))


# ------------------------------------------------------------------- tracked-row gather
@pytest.mark.parametrize("kv", ["bf16", "f32"])
def test_gather_rows_bit_exact(kv):
    # the tracked tokens' hidden states: x_rows[b][j] = x_all[b][idx[b][j]], a byte copy
    wl = W.make("llada8b-b32-drift", batch=3, max_pos=300, block=16, gen_lo=200, drift_k=24,
                **(dict(d_model=512, head_dim=128) if kv == "bf16" else dict(d_model=192, head_dim=64, act="f32",
                                                                              kv="f32")))
    s = wl.shape
    cache = G.make_cache(wl)
    idx = _topk_gpu(wl)
    x_all = G.tdev(wl.probe_rows(np.tile(np.arange(s.max_pos, dtype=np.int32), (s.batch, 1))), s.act)
    rows = torch.full((s.batch, wl.drift_k, s.D), 7.0, dtype=x_all.dtype, device="cuda")
    capi.dllm_gather_rows(cache.handle, x_all, G.idev(idx), rows)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    ref = x_all[torch.arange(s.batch, device="cuda")[:, None], G.idev(idx, torch.int64)]
    assert torch.equal(rows, ref)
    np.testing.assert_array_equal(rows.double().cpu().numpy(), wl.probe_rows(idx))  # the workload's rows
    # a position outside the sequence: a zero row and the status bit, nothing else touched
    bad = idx.copy()
    bad[1, 5] = s.max_pos
    capi.dllm_gather_rows(cache.handle, x_all, G.idev(bad), rows)
    rc, bits = cache.status()
    assert rc == capi.DLLM_EDEVICE and bits == capi.DEV_BAD_INDEX
    assert torch.count_nonzero(rows[1, 5]) == 0
    rows[1, 5] = ref[1, 5]
    assert torch.equal(rows, ref)


@pytest.mark.parametrize("kv,k", [("bf16", 32), ("bf16", 7), ("bf16", 40), ("f32", 24)])
def test_topk_gather_matches_the_two_calls(kv, k):
    # top-k and the row gather in one call: the oracle's top-k, bit-exact, and the byte
    # copy of those rows (one launch for k <= 32; k = 40 takes the two-launch path)
    wl = W.make("llada8b-b32-drift", batch=3, max_pos=300, block=16, gen_lo=200, drift_k=k,
                **(dict(d_model=512, head_dim=128) if kv == "bf16" else dict(d_model=192, head_dim=64, act="f32",
                                                                              kv="f32")))
    s = wl.shape
    cache = G.make_cache(wl)
    x_all = G.tdev(wl.probe_rows(np.tile(np.arange(s.max_pos, dtype=np.int32), (s.batch, 1))), s.act)
    mass = torch.from_numpy(wl.mass).cuda()
    lo = torch.from_numpy(wl.block_lo).cuda()
    idx = torch.full((s.batch, k), -5, dtype=torch.int32, device="cuda")
    rows = torch.full((s.batch, k, s.D), 7.0, dtype=x_all.dtype, device="cuda")
    capi.dllm_kv_topk_gather(cache.handle, mass, lo, wl.block_len, k, idx, x_all, rows)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    want = O.kv_topk(wl.mass, wl.block_lo, wl.block_len, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), want)
    ref = x_all[torch.arange(s.batch, device="cuda")[:, None], idx.long()]
    assert torch.equal(rows, ref)


# --------------------------------------------------------- drift fused into the projection
FUSED_DRIFT = [
    ("bf16", dict(d_model=512, head_dim=128, kv="bf16"), 24),
    ("e4m3", dict(d_model=512, head_dim=128, kv="e4m3"), 24),
    # 40 sequences x 37 tracked rows: 1480 probe rows over several 256-row tiles of the
    # CTA-pair projection (enough tiles at d_model 1024), a sequence's rows straddling two
    ("bf16-many", dict(batch=40, d_model=1024, head_dim=128, kv="bf16"), 37),
]


@pytest.mark.parametrize("name,kw,k", FUSED_DRIFT, ids=[c[0] for c in FUSED_DRIFT])
def test_fused_drift_matches_oracle(name, kw, k):
    kw = dict(kw)
    B = kw.pop("batch", 5)
    wl = W.make("llada8b-b32-drift", batch=B, max_pos=300, block=16, gen_lo=200, drift_k=k, **kw)
    s = wl.shape
    idx = _topk_gpu(wl)
    cache = G.make_cache(wl)
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                         kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    pos = G.idev(wl.positions)
    out = torch.empty_like(x)
    cos = torch.full((B, k, 2), 7.0, dtype=torch.float32, device="cuda")
    refresh = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    xp = G.tdev(wl.probe_rows(idx), s.act)
    o_out, ocache, o_probe = G.run_oracle(wl, probe_idx=idx)
    o_cos = O.kv_drift(ocache, idx, o_probe)
    for call in range(2):  # the workspace's counters and sums reset themselves
        capi.dllm_cache_step_drift(cache.handle, 0, x, w, pos, None, out, xp, G.idev(idx), 0.9, cos, refresh)
        torch.cuda.synchronize()
        assert cache.status() == (capi.DLLM_OK, 0)
        G.assert_close(out.double().cpu().numpy(), o_out, G.TOL[s.kv], f"attention out, call {call} ({name})")
        g_cos = cos.double().cpu().numpy()
        G.assert_close(g_cos, o_cos, G.TOL[s.kv], f"fused drift cos, call {call} ({name})")
        if s.kv == "e4m3":
            mcache = G.run_oracle(wl, probe_idx=idx, model_fp8=True)[1]
            G.assert_close(g_cos, O.kv_drift(mcache, idx, o_probe), G.FP8_MODEL_TOL,
                           f"fused drift cos vs the e4m3 model ({name})")
        np.testing.assert_array_equal(refresh.cpu().numpy(),
                                      (cos.cpu().numpy().reshape(B, -1).min(1) < np.float32(0.9)).astype(np.int32))
    G.compare_cache(cache, ocache, G.TOL[s.kv])  # probes never reach the cache


def test_fused_drift_bad_position_gives_nan_and_status():
    wl = W.make("llada8b-b32-drift", batch=3, d_model=256, head_dim=128, max_pos=300, block=16, gen_lo=200, drift_k=8)
    s = wl.shape
    idx = _topk_gpu(wl)
    cache = G.make_cache(wl, canary=False)
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                         kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    xp = G.tdev(wl.probe_rows(idx), s.act)
    bad = idx.copy()
    bad[1, 2] = s.max_pos + 5
    cos = torch.empty((3, 8, 2), dtype=torch.float32, device="cuda")
    refresh = torch.empty(3, dtype=torch.int32, device="cuda")
    capi.dllm_cache_project_drift(cache.handle, 0, None, w, None, None, None, xp, G.idev(bad), 0.9, cos, refresh)
    rc, bits = cache.status()
    assert rc == capi.DLLM_EDEVICE and bits == capi.DEV_BAD_POSITION
    c = cos.cpu().numpy()
    assert np.isnan(c[1, 2]).all() and np.isfinite(np.delete(c.reshape(-1, 2), 1 * 8 + 2, axis=0)).all()
    # the next call with good indices is unaffected (every counter was reset)
    capi.dllm_cache_project_drift(cache.handle, 0, None, w, None, None, None, xp, G.idev(idx), 0.9, cos, refresh)
    assert cache.status() == (capi.DLLM_OK, 0)
    ref = torch.empty_like(cos)
    probe = torch.empty((3, 8, 2, s.D), dtype=torch.bfloat16, device="cuda")
    capi.dllm_cache_project(cache.handle, 0, None, w, None, None, None, kv_x=xp, kv_positions=G.idev(idx),
                            probe_kv=probe)
    capi.dllm_kv_drift(cache.handle, 0, G.idev(idx), probe, 0.9, ref)
    torch.cuda.synchronize()
    # the separate path rounds the probes to bf16 first: cosines agree to that rounding
    assert float((cos - ref).abs().max()) < 2e-3
