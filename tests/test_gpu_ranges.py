"""Key ranges through the C ABI: ragged batches (each sequence attends to its first
key_len[b] slots) and partial softmax states over slot ranges with their merge (the
FACache combination), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu


def _staged(wl):
    """GPU cache filled (prefill + the step's rows) and the rotated Q of the step's rows."""
    s = wl.shape
    cache = G.make_cache(wl)
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None,
                         kv_x=G.tdev(wl.pre_x, s.act), kv_positions=G.idev(wl.pre_pos))
    x = G.tdev(wl.x, s.act)
    pos = G.idev(wl.positions)
    q = torch.empty_like(x)
    capi.dllm_cache_project(cache.handle, 0, x, w, pos, None, q)
    return cache, pos, q


def _oracle(wl, model_fp8=False):
    """The oracle's cache after the step's writes (unquantised unless model_fp8) and the
    step's rotated Q."""
    s = wl.shape
    kv = "e4m3" if (s.kv == "e4m3" and model_fp8) else "exact"
    cache = O.OracleCache(s.batch, s.max_pos, s.tail_slots, s.n_heads, s.head_dim, kv=kv)
    O.write_rows(cache, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    q = O.write_rows(cache, wl.w, wl.x, wl.positions, s.rope_theta)
    return cache, q


def _ragged_reference(wl, key_len, model_fp8=False):
    cache, q = _oracle(wl, model_fp8)
    n = wl.x.shape[1]
    ref = np.zeros((wl.shape.batch, n, wl.shape.D))
    for b in range(wl.shape.batch):
        L = int(min(max(key_len[b], 0), wl.shape.max_pos))
        if L == 0:
            continue
        vis = O.range_visible(n, cache.S + cache.T, 0, L)
        ref[b] = O.attention(q[b], cache.K[b], cache.V[b], vis).reshape(n, -1)
    return ref


RAGGED = [
    ("bf16", dict(batch=4, d_model=512, head_dim=128, max_pos=600, block=32, gen_lo=300), [600, 333, 129, 0]),
    ("e4m3", dict(batch=4, d_model=512, head_dim=128, max_pos=600, block=32, gen_lo=300, kv="e4m3"),
     [1, 600, 257, 450]),
    # few units: the keys are split across CTAs and most splits of short sequences are empty
    ("splits", dict(batch=2, d_model=256, head_dim=128, max_pos=640, block=16, gen_lo=300), [100, 640]),
    # more units than SMs with every other sequence empty: consecutive empty units per CTA
    ("empty-runs", dict(batch=40, d_model=512, head_dim=128, max_pos=256, block=16, gen_lo=128),
     [0 if b % 2 else 70 + 4 * b for b in range(40)]),
    # more sequences than the length ranking holds (256): units in plain order
    ("many", dict(batch=300, d_model=256, head_dim=128, max_pos=256, block=16, gen_lo=128),
     [(37 * b) % 257 for b in range(300)]),
]


@pytest.mark.parametrize("name,kw,lens", RAGGED, ids=[r[0] for r in RAGGED])
def test_ragged_matches_oracle(name, kw, lens):
    wl = W.make("llada8b-b1", fixed_lo=None, **kw)
    cache, pos, q = _staged(wl)
    key_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = q.clone()
    capi.dllm_cache_attend_ragged(cache.handle, 0, pos, key_len, out)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    got = out.double().cpu().numpy()
    ref = _ragged_reference(wl, lens)
    G.assert_close(got, ref, G.TOL[wl.shape.kv], f"ragged attention ({name})")
    if wl.shape.kv == "e4m3":
        G.assert_close(got, _ragged_reference(wl, lens, model_fp8=True), G.FP8_MODEL_TOL,
                       f"ragged attention vs the e4m3 model ({name})")
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(got[b] == 0.0)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_partial_states_and_merge(kv):
    wl = W.make("llada8b-b1", batch=3, d_model=512, head_dim=128, max_pos=600, block=40, gen_lo=300, fixed_lo=None, kv=kv)
    s = wl.shape
    cache, pos, q = _staged(wl)
    q_before = q.clone()
    n = wl.x.shape[1]
    st_a = torch.empty((s.batch, n, s.n_heads, s.head_dim + 2), dtype=torch.float32, device="cuda")
    st_b = torch.empty_like(st_a)
    st_ab = torch.empty_like(st_a)
    cut = 250  # not a tile boundary
    capi.dllm_cache_attend_partial(cache.handle, 0, pos, q, 0, cut, st_a)
    capi.dllm_cache_attend_partial(cache.handle, 0, pos, q, cut, s.max_pos, st_b)
    merged = torch.empty_like(q)
    capi.dllm_attend_merge(st_a, st_b, out=merged, state_out=st_ab)
    full = q.clone()
    capi.dllm_cache_attend(cache.handle, 0, pos, None, full)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    assert torch.equal(q, q_before)  # partial calls leave Q alone
    refs = [("oracle", _oracle(wl), G.TOL[kv])]
    if kv == "e4m3":
        # also against the oracle's model of the encoding, which holds the values the
        # kernel reads (up to rounding ties): the kernel's own error at the bf16 bound
        refs.append(("e4m3 model", _oracle(wl, model_fp8=True), G.FP8_MODEL_TOL))
    G.assert_close(merged.double().cpu().numpy(), full.double().cpu().numpy(), G.TOL["bf16"], "merged vs one-pass")
    for ref_name, (ocache, oq), tol in refs:
        full_ref = np.stack([O.attention(oq[b], ocache.K[b], ocache.V[b]).reshape(n, -1) for b in range(s.batch)])
        G.assert_close(merged.double().cpu().numpy(), full_ref, tol, f"merged partial states vs {ref_name}")
        # each state against the oracle's: the normalised output and the base-2 log-sum-exp
        for st, lo, hi in ((st_a, 0, cut), (st_b, cut, s.max_pos)):
            g = st.double().cpu().numpy()
            for b in range(s.batch):
                vis = O.range_visible(n, s.max_pos, lo, hi)
                ost = O.attention_partial(oq[b], ocache.K[b], ocache.V[b], vis)
                o_out = O.state_output(ost)
                g_out = g[b, :, :, :s.head_dim] / g[b, :, :, s.head_dim + 1][..., None]
                G.assert_close(g_out, o_out, tol, f"partial state output [{lo}, {hi}) b={b} vs {ref_name}")
                lse_g = g[b, :, :, s.head_dim] + np.log2(g[b, :, :, s.head_dim + 1])
                lse_o = ost[1] + np.log2(ost[2])
                G.record(f"partial state log2-sum-exp [{lo}, {hi}) b={b} vs {ref_name} (absolute)",
                         np.max(np.abs(lse_g - lse_o)), 0.05)
                assert np.max(np.abs(lse_g - lse_o)) < 0.05, np.max(np.abs(lse_g - lse_o))
        # the merged state normalises to the same output
        g = st_ab.double().cpu().numpy()
        G.assert_close(g[..., :s.head_dim] / g[..., s.head_dim + 1:], full_ref.reshape(g[..., :s.head_dim].shape),
                       tol, f"merged state vs {ref_name}")


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_facache_reuse_after_a_step_rewrites_the_tail(kv):
    # An invariant query block (q fixed) over a cache whose slots [lo, max_pos) are
    # rewritten by the next step: the state of [0, lo) is cached once, and after the
    # rewrite one call attends over [lo, max_pos) only and merges the cached state.
    wl = W.make("llada8b-b1", batch=3, d_model=512, head_dim=128, max_pos=600, block=40, gen_lo=300, fixed_lo=None, kv=kv)
    s = wl.shape
    cache, pos, q = _staged(wl)
    n = wl.x.shape[1]
    lo = 300  # not a tile boundary; the block sits in the rewritten range
    st_c = torch.empty((s.batch, n, s.n_heads, s.head_dim + 2), dtype=torch.float32, device="cuda")
    capi.dllm_cache_attend_partial(cache.handle, 0, pos, q, 0, lo, st_c)
    # the step rewrites every slot of [lo, max_pos) with new hidden states
    rng = np.random.default_rng(7)
    tail = np.arange(lo, s.max_pos, dtype=np.int32)
    x_new = W.round_bf16(rng.standard_normal((s.batch, len(tail), s.D)).astype(np.float32))
    w = G.tdev(wl.w, s.act)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None, kv_x=G.tdev(x_new, s.act),
                         kv_positions=G.idev(np.tile(tail, (s.batch, 1))))
    out = torch.full_like(q, float("nan"))
    q_before = q.clone()
    capi.dllm_cache_attend_with_state(cache.handle, 0, pos, q, lo, s.max_pos, st_c, out)
    full = q.clone()
    capi.dllm_cache_attend(cache.handle, 0, pos, None, full)  # one pass over the updated cache
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    assert torch.equal(q, q_before)
    got = out.double().cpu().numpy()
    # oracle: the same q over the updated cache, every slot
    for ref_name, model_fp8, tol in [("oracle", False, G.TOL[kv])] + (
            [("e4m3 model", True, G.FP8_MODEL_TOL)] if kv == "e4m3" else []):
        ocache, oq = _oracle(wl, model_fp8)
        O.write_rows(ocache, wl.w, x_new, np.tile(tail, (s.batch, 1)), s.rope_theta)
        ref = np.stack([O.attention(oq[b], ocache.K[b], ocache.V[b]).reshape(n, -1) for b in range(s.batch)])
        G.assert_close(got, ref, tol, f"FACache reuse vs {ref_name} ({kv})")
    G.assert_close(got, full.double().cpu().numpy(), G.TOL["bf16"], f"FACache reuse vs one pass ({kv})")
