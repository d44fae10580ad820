"""Shared helpers of the GPU parity tests: run a workload through the C ABI and through
the fp64 oracle on identical seeded inputs, then compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as W
from denoising_step_attention_qkv_b300 import capi

KV = {"f32": capi.DLLM_F32, "bf16": capi.DLLM_BF16, "e4m3": capi.DLLM_E4M3}
# max|gpu - oracle| <= TOL * max|oracle|, the oracle being the plain definition with an
# unquantised cache (the FP8 bound covers the e4m3 encoding's own error).
TOL = {"f32": 1e-4, "bf16": 2e-2, "e4m3": 6e-2}
# Tighter diagnostics of an e4m3 cache: against the oracle's model of the encoding
# (each group quantised with its scale), whatever the GPU does beyond that encoding is
# bf16/f16 operand rounding, so outputs and cosines are held to the bf16 bound; the
# codes themselves may differ only where the unquantised value lies within FP8_TIE of a
# rounding boundary (in units of the group's scale), which fp32 sums in another order
# can cross.
FP8_MODEL_TOL = TOL["bf16"]
FP8_TIE = 2.0 ** -8

# Every comparison made through assert_close: (what, measured, bound).  The test
# session prints the largest ratio per test and, with DLLM_PARITY_LOG set, writes every
# record to that file.
RECORDS = []


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


def run_oracle(wl: W.Workload, probe_idx: np.ndarray = None, model_fp8: bool = False):
    """Oracle of the workload.  Its cache keeps the unquantised values (the tolerance
    reference, also for an FP8 cache) unless ``model_fp8`` asks for the oracle's model of
    the e4m3 encoding (each group quantised with scale amax/448), the tighter diagnostic."""
    s = wl.shape
    kv = "e4m3" if (s.kv == "e4m3" and model_fp8) else "exact"
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


def record(what: str, measured: float, bound: float):
    RECORDS.append((what, float(measured), float(bound)))


def assert_close(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    e = rel_err(gpu, ref)
    record(what, e, tol)
    assert e <= tol, f"{what}: max|gpu-oracle|/max|oracle| = {e:.3g} > {tol}"
    return e


def fp8_code_check(codes: np.ndarray, scales: np.ndarray, exact: np.ndarray, what: str):
    """e4m3 groups against the oracle's quantisation of their unquantised values.

    codes: decoded e4m3 code values [..., hd] (without the scale); scales: the stored
    group scales [...]; exact: the oracle's unquantised values [..., hd].  The scale must
    be amax/448 of the group up to fp32 rounding, and every code must equal the oracle's
    round-to-nearest-even e4m3 code of value/scale, except where that value lies within
    FP8_TIE of the midpoint between the two neighbouring codes (a rounding tie that fp32
    arithmetic in another order may resolve either way).  Returns the number of such
    tie-side codes."""
    exact = np.asarray(exact, np.float64)
    amax = np.max(np.abs(exact), axis=-1)
    so = np.where(amax > 0, amax / 448.0, 1.0)
    s_err = float(np.max(np.abs(scales - so) / so)) if so.size else 0.0
    record(f"{what}: group scale vs amax/448", s_err, 1e-4)
    assert s_err <= 1e-4, f"{what}: group scale differs from amax/448 by {s_err:.3g} (relative)"
    t = exact / so[..., None]
    co = O.e4m3_quantize(t)
    diff = codes != co
    n = int(diff.sum())
    if n:
        cg, cm, tm = codes[diff], co[diff], t[diff]
        # neighbours on the e4m3 grid: no representable value strictly between them
        table = O.e4m3_table()
        grid = np.unique(table[np.isfinite(table)])
        lo, hi = np.minimum(cg, cm), np.maximum(cg, cm)
        between = np.searchsorted(grid, hi, "left") - np.searchsorted(grid, lo, "right")
        assert np.all(between == 0), f"{what}: a code differs from the oracle's by more than one e4m3 step"
        tie = float(np.max(np.abs(tm - (cg + cm) / 2.0)))
        record(f"{what}: farthest code flip from a rounding tie (scale units)", tie, FP8_TIE)
        assert tie <= FP8_TIE, f"{what}: a code flip {tie:.3g} scale units from the rounding tie > {FP8_TIE}"
    record(f"{what}: codes differing at rounding ties (count of {codes.size})", n, codes.size)
    return n


def gpu_fp8_groups(cache: capi.Cache, layer: int = 0):
    """(decoded code values [B][slots][2][H][hd], scales [B][slots][2][H]) as float64."""
    codes = cache.kv(layer).view(torch.float8_e4m3fn).to(torch.float32).double().cpu().numpy()
    return codes, cache.scale(layer).double().cpu().numpy()


def compare_cache(cache: capi.Cache, ocache: O.OracleCache, tol: float, layer: int = 0, what: str = "cache"):
    """Slot set bit-exact; K and V values at written slots within tol.  For an e4m3 cache
    against an unquantised oracle cache, also the codes (fp8_code_check)."""
    written = written_slots(cache, layer)
    np.testing.assert_array_equal(written, ocache.written, err_msg=f"set of written {what} slots")
    kv = gpu_kv(cache, layer)
    ek = assert_close(kv[:, :, 0][written], ocache.K[written], tol, f"{what} K")
    ev = assert_close(kv[:, :, 1][written], ocache.V[written], tol, f"{what} V")
    if cache.desc.kv_dtype == capi.DLLM_E4M3 and ocache.kv == "exact":
        codes, scales = gpu_fp8_groups(cache, layer)
        exact = np.stack([ocache.K, ocache.V], axis=2)  # [B][slots][2][H][hd]
        fp8_code_check(codes[written], scales[written], exact[written], f"{what} e4m3 codes")
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


def oracle_head(wl: W.Workload, b: int, h: int, probe_idx: np.ndarray = None, model_fp8: bool = False):
    """fp64 oracle restricted to head h of sequence b (unquantised cache unless
    ``model_fp8``, as in run_oracle).

    Returns (out [n_tok][hd], K [slots][hd], V [slots][hd], written [slots], probe or None)
    with probe = (K [k][hd], V [k][hd]) of the tracked tokens."""
    s = wl.shape
    hd = s.head_dim
    n = s.max_pos + s.tail_slots
    K = np.zeros((n, hd))
    V = np.zeros((n, hd))
    written = np.zeros(n, bool)
    store = O.OracleCache(1, 1, 0, 1, hd, kv="e4m3" if (s.kv == "e4m3" and model_fp8) else "exact").stored

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


def oracle_seq(wl: W.Workload, b: int, probe_idx: np.ndarray = None, model_fp8: bool = False):
    """The oracle's step for sequence b alone, every head: (out [n][D], cache, probe).

    cache is the oracle's one-sequence cache after the step (unquantised unless
    ``model_fp8``); probe is [k][2][D] of the tracked tokens or None."""
    s = wl.shape
    kv = "e4m3" if (s.kv == "e4m3" and model_fp8) else "exact"
    c = O.OracleCache(1, s.max_pos, s.tail_slots, s.n_heads, s.head_dim, kv=kv)
    one = slice(b, b + 1)
    if wl.pre_x is not None:
        O.write_rows(c, wl.w, wl.pre_x[one], wl.pre_pos[one], s.rope_theta)
    view = None if wl.view is None else wl.view[one]
    probe = None
    if probe_idx is not None:
        _, probe = O.step(c, wl.w, s.rope_theta, wl.x[one, :0], wl.positions[one, :0],
                          kv_x=wl.probe_rows(probe_idx[one], b0=b), kv_pos=probe_idx[one], probe=True)
        out, _ = O.step(c, wl.w, s.rope_theta, wl.x[one], wl.positions[one], view)
    else:
        kv_x = None if wl.kv_x is None else wl.kv_x[one]
        kv_pos = None if wl.kv_pos is None else wl.kv_pos[one]
        out, _ = O.step(c, wl.w, s.rope_theta, wl.x[one], wl.positions[one], view, kv_x=kv_x, kv_pos=kv_pos)
    return out[0], c, (None if probe is None else probe[0])


def check_sequences(wl: W.Workload, cache: capi.Cache, out: np.ndarray, seqs, probe_gpu: np.ndarray = None,
                    probe_idx: np.ndarray = None, whole_output: bool = False):
    """Full-size check: the written-slot set of every sequence bit-exactly, then every head
    of the sequences ``seqs``: cache K/V at written slots, the attention output and the
    probes against the oracle of that sequence (unquantised; for an e4m3 cache also the
    codes, and the output against the oracle's model of the encoding at the bf16 bound).
    Returns (largest error, {sequence: oracle_seq result}) for the callers' further checks.

    ``whole_output``: the output of every sequence is compared with the oracle's as one
    tensor, i.e. against max|oracle| over the workload's whole output, which is how the
    bound is stated (per sequence the bound is stricter than stated)."""
    s = wl.shape
    np.testing.assert_array_equal(written_slots_fast(cache), expected_written(wl, probe_idx is not None),
                                  err_msg="set of written cache slots")
    tol = TOL[s.kv]
    fp8 = s.kv == "e4m3"
    errs = []
    oracles = {}  # the oracle of each sequence, computed once
    if whole_output:
        for b in range(s.batch):
            oracles[b] = oracle_seq(wl, b, probe_idx)
        o_all = np.stack([oracles[b][0] for b in range(s.batch)])
        errs.append(assert_close(out, o_all, tol, "out (every sequence and head, one tensor)"))
    for b in seqs:
        if b not in oracles:
            oracles[b] = oracle_seq(wl, b, probe_idx)
        o, oc, pr = oracles[b]
        written = oc.written[0]
        kv = cache.kv(0)[b]
        if fp8:
            codes = kv.view(torch.float8_e4m3fn).to(torch.float32).double().cpu().numpy()  # [slots][2][H][hd]
            scales = cache.scale(0)[b].double().cpu().numpy()  # [slots][2][H]
            g = codes * scales[..., None]
        else:
            g = kv.double().cpu().numpy()
        errs.append(assert_close(g[written, 0], oc.K[0][written], tol, f"cache K (b={b}, all heads)"))
        errs.append(assert_close(g[written, 1], oc.V[0][written], tol, f"cache V (b={b}, all heads)"))
        if not whole_output:
            errs.append(assert_close(out[b], o, tol, f"out (b={b}, all heads)"))
        if fp8:
            exact = np.stack([oc.K[0], oc.V[0]], axis=1)  # [slots][2][H][hd]
            fp8_code_check(codes[written], scales[written], exact[written], f"e4m3 codes (b={b})")
            om = oracle_seq(wl, b, probe_idx, model_fp8=True)[0]
            assert_close(out[b], om, FP8_MODEL_TOL, f"out vs the e4m3 model (b={b}, all heads)")
        if pr is not None:
            errs.append(assert_close(probe_gpu[b], pr, TOL[s.act], f"probe K/V (b={b}, all heads)"))
    return max(errs), oracles
