"""Shared helpers of the GPU parity tests: run a workload through the C ABI and through
the fp64 oracle on identical seeded inputs, then compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as W
from denoising_step_attention_qkv_b300 import capi

KV = {"f32": capi.DLLM_F32, "bf16": capi.DLLM_BF16, "e4m3": capi.DLLM_E4M3}
# max|gpu - oracle| <= TOL * max|oracle|
TOL = {"f32": 1e-4, "bf16": 2e-2, "e4m3": 6e-2}


def tdev(a: np.ndarray, act: str) -> torch.Tensor:
    """Storage-rounded float32 array -> device tensor of the activation type (exact)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if act == "bf16":
        t = t.to(torch.bfloat16)  # exact: values are bf16-representable
    return t.cuda()


def idev(a: np.ndarray, dtype=torch.int32) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def make_cache(wl: W.Workload, canary: bool = True) -> capi.Cache:
    s = wl.shape
    c = capi.Cache(1, s.batch, s.max_pos, s.n_heads, s.head_dim, KV[s.kv], s.rope_theta, s.tail_slots)
    if canary:
        c.buf.fill_(0xFF)  # NaN in fp32, bf16 and e4m3: marks never-written slots
    return c


def gpu_kv(cache: capi.Cache, layer: int = 0) -> np.ndarray:
    """Dequantised cache contents as float64 [B][slots][2][H][hd] (NaN = canary)."""
    kv = cache.kv(layer)
    if cache.desc.kv_dtype == capi.DLLM_E4M3:
        vals = kv.view(torch.float8_e4m3fn).to(torch.float32)
        vals = vals * cache.scale(layer)[..., None]
        return vals.double().cpu().numpy()
    return kv.double().cpu().numpy()


def written_slots(cache: capi.Cache, layer: int = 0) -> np.ndarray:
    """bool [B][slots]: slot holds anything other than the canary in K or V."""
    raw = cache.kv(layer)
    if raw.dtype == torch.bfloat16:
        bits = raw.view(torch.int16) != -1
    elif raw.dtype == torch.float32:
        bits = raw.view(torch.int32) != -1
    else:
        bits = raw != 0xFF
    return bits.reshape(bits.shape[0], bits.shape[1], -1).any(-1).cpu().numpy()


def run_gpu(wl: W.Workload, cache: capi.Cache, probe_idx: np.ndarray = None, layer: int = 0):
    """Prefill (if any) then the step, through the C ABI.  Returns (out, probe_kv) numpy."""
    s = wl.shape
    w = tdev(wl.w, s.act)
    if wl.pre_x is not None:
        capi.dllm_cache_step(cache.handle, layer, None, w, None, None, None,
                             kv_x=tdev(wl.pre_x, s.act), kv_positions=idev(wl.pre_pos))
    x = tdev(wl.x, s.act)
    pos = idev(wl.positions)
    view = idev(wl.view, torch.uint8) if wl.view is not None else None
    out = torch.empty_like(x)
    kv_x = kv_pos = probe = None
    if probe_idx is not None:
        kv_x = tdev(wl.probe_rows(probe_idx), s.act)
        kv_pos = idev(probe_idx)
        probe = torch.empty((s.batch, probe_idx.shape[1], 2, s.D), dtype=x.dtype, device="cuda")
    elif wl.kv_x is not None:
        kv_x = tdev(wl.kv_x, s.act)
        kv_pos = idev(wl.kv_pos)
    capi.dllm_cache_step(cache.handle, layer, x, w, pos, view, out, kv_x=kv_x, kv_positions=kv_pos, probe_kv=probe)
    torch.cuda.synchronize()
    rc, bits = cache.status()
    assert rc == capi.DLLM_OK and bits == 0, f"device status bits {bits:#x}"
    return out.double().cpu().numpy(), (None if probe is None else probe.double().cpu().numpy())


def run_oracle(wl: W.Workload, probe_idx: np.ndarray = None, exact: bool = False):
    """Oracle of the workload; an FP8 cache is modelled (its quantisation is a step of the
    computation) unless ``exact`` asks for the unquantised diagnostic."""
    s = wl.shape
    kv = "e4m3" if (s.kv == "e4m3" and not exact) else "exact"
    cache = O.OracleCache(s.batch, s.max_pos, s.tail_slots, s.n_heads, s.head_dim, kv=kv)
    if wl.pre_x is not None:
        O.write_rows(cache, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    probe = None
    if probe_idx is not None:
        _, probe = O.step(cache, wl.w, s.rope_theta, wl.x[:, :0], wl.positions[:, :0],
                          kv_x=wl.probe_rows(probe_idx), kv_pos=probe_idx, probe=True)
        out, _ = O.step(cache, wl.w, s.rope_theta, wl.x, wl.positions, wl.view)
    else:
        out, _ = O.step(cache, wl.w, s.rope_theta, wl.x, wl.positions, wl.view, kv_x=wl.kv_x, kv_pos=wl.kv_pos)
    return out, cache, probe


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(gpu - ref)) / scale)


def assert_close(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max|gpu-oracle|/max|oracle| = {e:.3g} > {tol}"
    return e


def compare_cache(cache: capi.Cache, ocache: O.OracleCache, tol: float):
    """Slot set bit-exact; K and V values at written slots within tol."""
    written = written_slots(cache)
    np.testing.assert_array_equal(written, ocache.written, err_msg="set of written cache slots")
    kv = gpu_kv(cache)
    B, n, _, H, hd = kv.shape
    ek = assert_close(kv[:, :, 0][written], ocache.K[written], tol, "cache K")
    ev = assert_close(kv[:, :, 1][written], ocache.V[written], tol, "cache V")
    return ek, ev


# ------------------------------------------------------------------------------------
# Full-size workloads: the GPU runs the whole step; the oracle recomputes sampled
# (sequence, head) pairs one by one.
# ------------------------------------------------------------------------------------

def expected_written(wl: W.Workload, probe: bool = False) -> np.ndarray:
    """bool [B][slots]: slots the step (and its prefill) must write - index logic only."""
    s = wl.shape
    n = s.max_pos + s.tail_slots
    w = np.zeros((s.batch, n), bool)
    for b in range(s.batch):
        if wl.pre_pos is not None:
            w[b, wl.pre_pos[b]] = True
        if wl.kv_pos is not None and not probe:
            w[b, wl.kv_pos[b]] = True
        vb = None if wl.view is None else wl.view[b]
        w[b, O.row_slots(wl.positions[b], vb, s.max_pos)] = True
    return w


def written_slots_fast(cache: capi.Cache, layer: int = 0) -> np.ndarray:
    raw = cache.kv(layer)
    if raw.dtype == torch.bfloat16:
        bits = raw.view(torch.int16) != -1
    elif raw.dtype == torch.float32:
        bits = raw.view(torch.int32) != -1
    else:
        bits = raw != 0xFF
    return bits.flatten(2).any(-1).cpu().numpy()


def gpu_head(cache: capi.Cache, b: int, h: int, layer: int = 0) -> np.ndarray:
    """Dequantised K/V of one (sequence, head): float64 [slots][2][hd]."""
    kv = cache.kv(layer)[b, :, :, h, :]
    if cache.desc.kv_dtype == capi.DLLM_E4M3:
        vals = kv.view(torch.float8_e4m3fn).to(torch.float32) * cache.scale(layer)[b, :, :, h][..., None]
        return vals.double().cpu().numpy()
    return kv.double().cpu().numpy()


def oracle_head(wl: W.Workload, b: int, h: int, probe_idx: np.ndarray = None, exact: bool = False):
    """fp64 oracle restricted to head h of sequence b.

    Returns (out [n_tok][hd], K [slots][hd], V [slots][hd], written [slots], probe or None)
    with probe = (K [k][hd], V [k][hd]) of the tracked tokens."""
    s = wl.shape
    hd = s.head_dim
    n = s.max_pos + s.tail_slots
    K = np.zeros((n, hd))
    V = np.zeros((n, hd))
    written = np.zeros(n, bool)
    store = O.OracleCache(1, 1, 0, 1, hd, kv="e4m3" if (s.kv == "e4m3" and not exact) else "exact").stored

    def put(x_rows, pos, slots):
        q, k, v = O.project_head(x_rows, wl.w, s.n_heads, h)
        q = O.rope(q[:, None, :], pos, s.rope_theta)[:, 0]
        k = O.rope(k[:, None, :], pos, s.rope_theta)[:, 0]
        K[slots] = np.stack([store(r) for r in k])
        V[slots] = np.stack([store(r) for r in v])
        written[slots] = True
        return q

    if wl.pre_x is not None:
        put(wl.pre_x[b], wl.pre_pos[b], wl.pre_pos[b])
    if wl.kv_x is not None and probe_idx is None:
        put(wl.kv_x[b], wl.kv_pos[b], wl.kv_pos[b])
    vb = None if wl.view is None else wl.view[b]
    slots = O.row_slots(wl.positions[b], vb, s.max_pos)
    q = put(wl.x[b], wl.positions[b], slots)
    kview = O.key_views(wl.positions[b], vb, s.max_pos, n)
    qview = np.zeros(len(slots), np.int64) if vb is None else vb.astype(np.int64)
    vis = O.visible(qview, kview)
    assert written[vis.any(0)].all()
    out = O.attention(q[:, None, :], K[:, None, :], V[:, None, :], vis)[:, 0]
    probe = None
    if probe_idx is not None:
        xp = wl.probe_rows(probe_idx[b:b + 1], b0=b)[0]
        _, kp, vp = O.project_head(xp, wl.w, s.n_heads, h)
        kp = O.rope(kp[:, None, :], probe_idx[b], s.rope_theta)[:, 0]
        probe = (kp, vp)
    return out, K, V, written, probe


def check_sampled(wl: W.Workload, cache: capi.Cache, out: np.ndarray, samples, probe_gpu: np.ndarray = None,
                  probe_idx: np.ndarray = None, exact_diag_tol: float = None):
    """Written-slot set in full (bit-exact), then cache, output and probes on sampled heads."""
    s = wl.shape
    np.testing.assert_array_equal(written_slots_fast(cache), expected_written(wl, probe_idx is not None),
                                  err_msg="set of written cache slots")
    tol = TOL[s.kv]
    hd = s.head_dim
    errs = []
    for b, h in samples:
        o, K, V, written, probe = oracle_head(wl, b, h, probe_idx)
        g = gpu_head(cache, b, h)
        errs.append(assert_close(g[written, 0], K[written], tol, f"cache K (b={b}, h={h})"))
        errs.append(assert_close(g[written, 1], V[written], tol, f"cache V (b={b}, h={h})"))
        errs.append(assert_close(out[b][:, h * hd:(h + 1) * hd], o, tol, f"out (b={b}, h={h})"))
        if exact_diag_tol is not None:  # FP8 cache against the unquantised oracle: the encoding's own error
            oe = oracle_head(wl, b, h, exact=True)[0]
            assert_close(out[b][:, h * hd:(h + 1) * hd], oe, exact_diag_tol, f"out vs unquantised (b={b}, h={h})")
        if probe is not None:
            pg = probe_gpu[b][:, :, h * hd:(h + 1) * hd]
            errs.append(assert_close(pg[:, 0], probe[0], TOL[s.act], f"probe K (b={b}, h={h})"))
            errs.append(assert_close(pg[:, 1], probe[1], TOL[s.act], f"probe V (b={b}, h={h})"))
    return max(errs)
