"""Pins for the fp64 oracle: closed forms, invariants, brute force, one library routine.

None of these re-type the oracle's own formula: each checks a property or value that
the mathematics of the step fixes independently of how the oracle computes it.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

with open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")) as _f:
    GOLD = json.load(_f)


def _rng(s=0):
    return np.random.default_rng(1234 + s)


# ----------------------------------------------------------------------------- RoPE
def test_rope_golden_hd2():
    for c in GOLD["rope_hd2"]["cases"]:
        y = O.rope(np.array(c["x"])[None, None, :], np.array([c["p"]]), theta=10000.0)
        np.testing.assert_allclose(y[0, 0], c["y"], rtol=0, atol=1e-15)


def test_rope_golden_pairing_and_frequency():
    g = GOLD["rope_hd4_theta100"]
    for c in g["cases"]:
        y = O.rope(np.array(c["x"])[None, None, :], np.array([g["p"]]), theta=100.0)
        np.testing.assert_allclose(y[0, 0], c["y"], rtol=0, atol=1e-15)


def test_rope_preserves_norm():
    r = _rng()
    v = r.standard_normal((50, 3, 128))
    p = r.integers(0, 5000, 50)
    y = O.rope(v, p, 500000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(v, axis=-1), rtol=1e-13)


def test_rope_dot_depends_only_on_offset():
    r = _rng(1)
    q = r.standard_normal((1, 2, 64))
    k = r.standard_normal((1, 2, 64))
    for p, pk, c in [(5, 3, 100), (0, 70, 1000), (127, 0, 2500)]:
        d1 = np.sum(O.rope(q, np.array([p]), 1e4) * O.rope(k, np.array([pk]), 1e4), axis=-1)
        d2 = np.sum(O.rope(q, np.array([p + c]), 1e4) * O.rope(k, np.array([pk + c]), 1e4), axis=-1)
        np.testing.assert_allclose(d1, d2, rtol=1e-10, atol=1e-10)


def test_rope_position_zero_is_identity():
    v = _rng(2).standard_normal((4, 2, 16))
    np.testing.assert_array_equal(O.rope(v, np.zeros(4, int), 1e4), v)


# ----------------------------------------------------------------------- projection
def test_projection_identity_weights():
    D, H = 8, 2
    eye = np.eye(D)
    w = np.concatenate([eye, 2 * eye, 3 * eye])  # [3D][D]
    x = _rng(3).standard_normal((5, D))
    q, k, v = O.project_qkv(x, w, H)
    np.testing.assert_array_equal(q.reshape(5, D), x)
    np.testing.assert_array_equal(k.reshape(5, D), 2 * x)
    np.testing.assert_array_equal(v.reshape(5, D), 3 * x)


def test_projection_row_permutation_permutes_features():
    D, H = 8, 2
    r = _rng(4)
    w = r.standard_normal((3 * D, D))
    perm = r.permutation(3 * D)
    x = r.standard_normal((3, D))
    q, k, v = O.project_qkv(x, w, H)
    y = np.concatenate([q.reshape(3, D), k.reshape(3, D), v.reshape(3, D)], axis=1)
    q2, k2, v2 = O.project_qkv(x, w[perm], H)
    y2 = np.concatenate([q2.reshape(3, D), k2.reshape(3, D), v2.reshape(3, D)], axis=1)
    np.testing.assert_allclose(y2, y[:, perm], rtol=1e-14)


def test_projection_head_split_brute_force():
    D, H, hd = 6, 3, 2
    r = _rng(5)
    w = r.standard_normal((3 * D, D))
    x = r.standard_normal((2, D))
    q, k, v = O.project_qkv(x, w, H)
    heads = [O.project_head(x, w, H, h) for h in range(H)]
    for t in range(2):
        for part, arr in enumerate((q, k, v)):
            for h in range(H):
                for i in range(hd):
                    n = part * D + h * hd + i
                    ref = sum(x[t, c] * w[n, c] for c in range(D))
                    assert abs(arr[t, h, i] - ref) < 1e-12
                    assert abs(heads[h][part][t, i] - ref) < 1e-12


# ------------------------------------------------------------------------ attention
def test_attention_golden_weights():
    g = GOLD["attention_weights_1234"]
    q = np.array(g["q"])[None, None, :]
    K = np.array([[math.log(a), 0, 0, 0] for a in g["a"]])[:, None, :]
    V = np.array(g["v"], float)[:, None, :]
    o = O.attention(q, K, V)
    np.testing.assert_allclose(o[0, 0], g["o"], rtol=1e-13)


def test_attention_identical_keys_gives_mean_of_v():
    r = _rng(6)
    k = r.standard_normal(16)
    K = np.tile(k, (9, 2, 1))  # 9 keys, 2 heads
    V = r.standard_normal((9, 2, 16))
    q = r.standard_normal((3, 2, 16))
    np.testing.assert_allclose(O.attention(q, K, V), np.broadcast_to(V.mean(0), (3, 2, 16)), rtol=1e-12)


def test_attention_single_visible_key():
    r = _rng(7)
    K, V = r.standard_normal((6, 1, 8)), r.standard_normal((6, 1, 8))
    q = r.standard_normal((2, 1, 8))
    vis = np.zeros((2, 6), bool)
    vis[0, 4] = vis[1, 1] = True
    o = O.attention(q, K, V, vis)
    np.testing.assert_allclose(o[0, 0], V[4, 0], rtol=1e-14)
    np.testing.assert_allclose(o[1, 0], V[1, 0], rtol=1e-14)


def test_attention_permutation_invariant_and_shift_stable():
    r = _rng(8)
    q, K, V = r.standard_normal((4, 2, 8)), r.standard_normal((10, 2, 8)), r.standard_normal((10, 2, 8))
    perm = r.permutation(10)
    np.testing.assert_allclose(O.attention(q, K[perm], V[perm]), O.attention(q, K, V), rtol=1e-12)
    # huge logits must not overflow (max subtraction): scale q by 1e3
    o = O.attention(1e3 * q, K, V)
    assert np.all(np.isfinite(o))


def test_attention_brute_force_tiny_python_loops():
    # B=1, H=1, hd=8, S=4, 2-token block: pure-Python step against the oracle step.
    r = _rng(9)
    D, H, hd, S = 8, 1, 8, 4
    theta = 10000.0
    w = r.standard_normal((3 * D, D)) * 0.3
    x_pre = r.standard_normal((1, 2, D))
    x = r.standard_normal((1, 2, D))
    pre_pos = np.array([[0, 3]])
    pos = np.array([[1, 2]])

    def proj(row):
        return [sum(row[c] * w[n, c] for c in range(D)) for n in range(3 * D)]

    def rot(vec, p):
        half = hd // 2
        out = list(vec)
        for i in range(half):
            a = p * theta ** (-2.0 * i / hd)
            out[i] = vec[i] * math.cos(a) - vec[i + half] * math.sin(a)
            out[i + half] = vec[i + half] * math.cos(a) + vec[i] * math.sin(a)
        return out

    Kc = [None] * S
    Vc = [None] * S
    for t in range(2):
        y = proj(x_pre[0, t])
        Kc[pre_pos[0, t]] = rot(y[D:2 * D], pre_pos[0, t])
        Vc[pre_pos[0, t]] = y[2 * D:]
    qs = []
    for t in range(2):
        y = proj(x[0, t])
        Kc[pos[0, t]] = rot(y[D:2 * D], pos[0, t])
        Vc[pos[0, t]] = y[2 * D:]
        qs.append(rot(y[:D], pos[0, t]))
    expect = []
    for t in range(2):
        s = [sum(qs[t][i] * Kc[j][i] for i in range(hd)) / math.sqrt(hd) for j in range(S)]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        z = sum(e)
        expect.append([sum(e[j] / z * Vc[j][i] for j in range(S)) for i in range(hd)])

    cache = O.OracleCache(1, S, 0, H, hd)
    O.write_rows(cache, w, x_pre, pre_pos, theta)
    out, _ = O.step(cache, w, theta, x, pos)
    np.testing.assert_allclose(out[0], np.array(expect), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------- Flash-Verify
def test_visibility_truth_table():
    # rows: query view BASE, DRAFT, MASK; columns: key view SHARED, MASK, DRAFT, NONE
    qv = np.array([O.VIEW_BASE, O.VIEW_DRAFT, O.VIEW_MASK])
    kv = np.array([O.KVIEW_SHARED, O.KVIEW_MASK, O.KVIEW_DRAFT, O.KVIEW_NONE])
    expect = np.array([[1, 1, 0, 0],
                       [1, 0, 1, 0],
                       [1, 1, 0, 0]], bool)
    np.testing.assert_array_equal(O.visible(qv, kv), expect)


def _verify_case(seed=0, **kw):
    args = dict(batch=2, d_model=256, head_dim=128, max_pos=96, block=16, gen_lo=48, search=6, tail_slots=8)
    args.update(kw)
    return W.make("llada8b-b16-verify", seed=seed, **args)


def _run(wl, x=None, positions=None, view=None):
    s = wl.shape
    cache = O.OracleCache(s.batch, s.max_pos, s.tail_slots, s.n_heads, s.head_dim)
    O.write_rows(cache, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    return O.step(cache, wl.w, s.rope_theta, wl.x if x is None else x,
                  wl.positions if positions is None else positions, view)[0], cache


def test_verify_draft_equal_mask_gives_identical_views():
    wl = _verify_case()
    x = wl.x.copy()
    n_blk = wl.block_len
    for b in range(wl.shape.batch):
        # draft rows take exactly the x of their mask-view twin
        for t in range(n_blk, x.shape[1]):
            twin = np.where((wl.positions[b, :n_blk] == wl.positions[b, t]) & (wl.view[b, :n_blk] == O.VIEW_MASK))[0]
            assert len(twin) == 1
            x[b, t] = x[b, twin[0]]
    out, _ = _run(wl, x=x, view=wl.view)
    for b in range(wl.shape.batch):
        for t in range(n_blk, x.shape[1]):
            twin = np.where((wl.positions[b, :n_blk] == wl.positions[b, t]) & (wl.view[b, :n_blk] == O.VIEW_MASK))[0][0]
            np.testing.assert_allclose(out[b, t], out[b, twin], rtol=1e-12, atol=1e-14)


def test_verify_empty_search_set_is_the_ordinary_step():
    wl = _verify_case()
    n_blk = wl.block_len
    x, pos = wl.x[:, :n_blk], wl.positions[:, :n_blk]
    base_view = np.zeros_like(wl.view[:, :n_blk])
    out_a, _ = _run(wl, x=x, positions=pos, view=base_view)
    out_b, _ = _run(wl, x=x, positions=pos, view=None)
    np.testing.assert_array_equal(out_a, out_b)


def test_verify_base_rows_never_see_draft_views():
    wl = _verify_case()
    n_blk = wl.block_len
    full, _ = _run(wl, view=wl.view)
    plain, _ = _run(wl, x=wl.x[:, :n_blk], positions=wl.positions[:, :n_blk], view=wl.view[:, :n_blk])
    base = wl.view[:, :n_blk] != O.VIEW_DRAFT
    np.testing.assert_allclose(full[:, :n_blk][base], plain[base], rtol=1e-12, atol=1e-14)


def test_verify_draft_rows_use_tail_slots():
    wl = _verify_case()
    _, cache = _run(wl, view=wl.view)
    S = wl.shape.max_pos
    n_draft = int((wl.view[0] == O.VIEW_DRAFT).sum())
    assert cache.written[0, S:S + n_draft].all() and not cache.written[0, S + n_draft:].any()


def test_verify_rth_draft_row_writes_tail_slot_r():
    """Flash-dLLM, paragraph 3: a DRAFT row keeps its absolute position for the rotary
    embedding but goes to the tail; the r-th DRAFT row of a sequence (row order) fills
    tail slot max_pos + r, which then holds that row's own K and V."""
    wl = _verify_case()
    _, cache = _run(wl, view=wl.view)
    s = wl.shape
    for b in range(s.batch):
        drafts = [t for t in range(wl.x.shape[1]) if wl.view[b, t] == O.VIEW_DRAFT]
        assert len(drafts) >= 2
        for r_, t in enumerate(drafts):
            _, k, v = O.project_qkv(wl.x[b, t:t + 1], wl.w, s.n_heads)
            k = O.rope(k, wl.positions[b, t:t + 1], s.rope_theta)
            np.testing.assert_allclose(cache.K[b, s.max_pos + r_], k[0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(cache.V[b, s.max_pos + r_], v[0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------- drift
def test_cosine_special_cases():
    v = _rng(10).standard_normal(300)
    assert abs(O.cosine(v, v) - 1) < 1e-15
    assert abs(O.cosine(v, -v) + 1) < 1e-15
    assert abs(O.cosine(v, 3.5 * v) - 1) < 1e-15
    e1, e2 = np.eye(2)
    assert O.cosine(e1, e2) == 0.0


def test_topk_brute_force_and_block_exclusion():
    r = _rng(11)
    B, S, k = 3, 64, 7
    mass = r.random((B, S)).astype(np.float32)
    lo = np.array([0, 20, 57])
    blen = 7
    mass[1, 20:27] = 10.0  # block masses are the largest, but excluded
    idx = O.kv_topk(mass, lo, blen, k)
    for b in range(B):
        cand = np.array([p for p in range(S) if not (lo[b] <= p < lo[b] + blen)])
        order = np.lexsort((cand, -mass[b, cand].astype(np.float64)))
        np.testing.assert_array_equal(idx[b], cand[order[:k]])


def test_topk_ties_take_lower_position_and_permutation_equivariance():
    mass = np.zeros((1, 10), np.float32)
    mass[0, [2, 5, 7]] = 0.5
    idx = O.kv_topk(mass, np.array([9]), 1, 4)
    np.testing.assert_array_equal(idx[0], [2, 5, 7, 0])
    r = _rng(12)
    m = r.random((1, 40)).astype(np.float32)
    perm = r.permutation(40)
    a = O.kv_topk(m, np.array([40]), 0, 5)[0]
    b = O.kv_topk(m[:, perm], np.array([40]), 0, 5)[0]
    inv = np.argsort(perm)
    np.testing.assert_array_equal(np.sort(perm[b]), np.sort(a))
    assert set(inv[a]) == set(b)


def test_drift_is_one_when_probe_equals_cached_token():
    wl = W.make("llada8b-b32-drift", batch=2, d_model=256, head_dim=128, max_pos=96, gen_lo=48, block=16, drift_k=5)
    s = wl.shape
    cache = O.OracleCache(s.batch, s.max_pos, 0, s.n_heads, s.head_dim)
    O.write_rows(cache, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    idx = O.kv_topk(wl.mass, wl.block_lo, wl.block_len, 5)
    xp = np.stack([np.stack([wl.prefill_row(b, int(p)) for p in idx[b]]) for b in range(s.batch)])
    _, probe = O.step(cache, wl.w, s.rope_theta, wl.x[:, :0], wl.positions[:, :0], kv_x=xp, kv_pos=idx, probe=True)
    cos = O.kv_drift(cache, idx, probe)
    np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-12)
    # noisy probes drift below one
    _, probe2 = O.step(cache, wl.w, s.rope_theta, wl.x[:, :0], wl.positions[:, :0],
                       kv_x=wl.probe_rows(idx), kv_pos=idx, probe=True)
    c2 = O.kv_drift(cache, idx, probe2)
    assert np.all(c2 < 1.0) and np.all(c2 > 0.9)


def test_drift_closed_form_over_the_whole_token_vector():
    """Flash-dLLM, paragraph 4: the drift of a tracked token is the cosine between its
    cached and recomputed K (and, apart, V) over the token's whole D-vector.  Negating
    head h of the probe K gives 1 - 2|K_h|^2 / |K|^2; a probe V of -V gives -1."""
    r = _rng(13)
    B, S, H, hd = 2, 16, 4, 8
    cache = O.OracleCache(B, S, 0, H, hd)
    cache.K[:] = r.standard_normal(cache.K.shape) * r.uniform(0.5, 2.0, size=(B, S, H, 1))
    cache.V[:] = r.standard_normal(cache.V.shape)
    idx = np.array([[3, 0, 9], [15, 7, 2]])
    k, D = idx.shape[1], H * hd
    probe = np.empty((B, k, 2, D))
    expect = np.empty((B, k, 2))
    for b in range(B):
        for j in range(k):
            Kt = cache.K[b, idx[b, j]]
            h = (b + j) % H
            Kp = Kt.copy()
            Kp[h] *= -1.0
            probe[b, j, 0] = Kp.reshape(D)
            probe[b, j, 1] = -cache.V[b, idx[b, j]].reshape(D)
            expect[b, j, 0] = 1.0 - 2.0 * np.sum(Kt[h] ** 2) / np.sum(Kt ** 2)
            expect[b, j, 1] = -1.0
    np.testing.assert_allclose(O.kv_drift(cache, idx, probe), expect, rtol=0, atol=1e-12)


# ------------------------------------------------------------------------------ FP8
def test_e4m3_named_values():
    for code, val in GOLD["e4m3_named_values"]["codes"].items():
        assert O.e4m3_decode(int(code, 16)) == val


def test_e4m3_table_matches_library_cast():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = O.e4m3_table()
    nan = np.isnan(tab)
    np.testing.assert_array_equal(nan, np.isnan(lib))
    np.testing.assert_array_equal(tab[~nan], lib[~nan])


def test_e4m3_quantize_matches_library_rounding_in_range():
    torch = pytest.importorskip("torch")
    r = _rng(13)
    y = np.concatenate([r.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    y = y[np.abs(y) <= 448]
    # exact midpoints between neighbouring codes decide the tie rule (to even)
    tab = np.unique(O.e4m3_table()[np.isfinite(O.e4m3_table())])
    y = np.concatenate([y, 0.5 * (tab[1:] + tab[:-1])])
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_quantize(y), lib)


def test_e4m3_saturation_roundtrip_and_error_bound():
    np.testing.assert_array_equal(O.e4m3_quantize(np.array([500.0, 1e6, -1000.0, 464.0])), [448, 448, -448, 448])
    tab = O.e4m3_table()
    fin = tab[np.isfinite(tab)]
    np.testing.assert_array_equal(O.e4m3_quantize(fin), fin)
    y = _rng(14).uniform(-448, 448, 100000)
    err = np.abs(O.e4m3_quantize(y) - y)
    normal = np.abs(y) >= 2 ** -6
    assert np.all(err[normal] <= 2 ** -4 * np.abs(y[normal]) + 1e-300)
    assert np.all(err[~normal] <= 2 ** -10)


def test_fp8_group_quantize_scale_and_zero_group():
    v = _rng(15).standard_normal(128)
    deq, scale = O.fp8_group_quantize(v)
    amax = np.max(np.abs(v))
    assert scale == amax / 448.0
    i = np.argmax(np.abs(v))
    assert abs(deq[i] - v[i]) <= 1e-12 * amax
    assert np.max(np.abs(deq - v)) <= 2 ** -4 * amax
    z, s0 = O.fp8_group_quantize(np.zeros(128))
    assert s0 == 1.0 and not np.any(z)


def test_fp8_cache_stores_group_quantised_values():
    # an e4m3 cache keeps, per (token, head) group, exactly the group quantiser's output
    r = _rng(16)
    c = O.OracleCache(1, 4, 0, 2, 8, kv="e4m3")
    w = r.standard_normal((3 * 16, 16))
    x = r.standard_normal((1, 2, 16))
    O.write_rows(c, w, x, np.array([[1, 3]]), 1e4)
    _, k, v = O.project_qkv(x[0], w, 2)
    k = O.rope(k, np.array([1, 3]), 1e4)
    for t, s in enumerate([1, 3]):
        for h in range(2):
            np.testing.assert_array_equal(c.K[0, s, h], O.fp8_group_quantize(k[t, h])[0])
            np.testing.assert_array_equal(c.V[0, s, h], O.fp8_group_quantize(v[t, h])[0])
            # every stored value is an e4m3 value times the group scale
            scale = np.max(np.abs(v[t, h])) / 448.0
            codes = c.V[0, s, h] / scale
            np.testing.assert_allclose(O.e4m3_quantize(codes), codes, rtol=1e-12)


# ------------------------------------------------------------------ attention mass
def test_attention_weights_rows_sum_to_one_and_match_attention():
    r = _rng(20)
    q, K, V = r.standard_normal((5, 2, 8)), r.standard_normal((9, 2, 8)), r.standard_normal((9, 2, 8))
    p = O.attention_weights(q, K)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-13)
    # weights applied to V reproduce the attention output (an independent contraction)
    np.testing.assert_allclose(np.einsum("hqk,khd->qhd", p, V), O.attention(q, K, V), rtol=1e-12)


def test_attention_mass_totals_uniform_keys_and_views():
    r = _rng(21)
    S, H, hd, n = 12, 3, 8, 4
    cache = O.OracleCache(1, S, 0, H, hd)
    cache.K[0] = r.standard_normal((S, H, hd))
    q = r.standard_normal((1, n, H, hd))
    pos = np.array([[2, 5, 7, 9]])
    m = O.attention_mass(cache, q, pos)
    assert m.shape == (1, S)
    np.testing.assert_allclose(m.sum(), H * n, rtol=1e-13)  # every query's weights sum to 1
    cache.K[0] = 1.0  # identical keys: every slot gets the same share
    np.testing.assert_allclose(O.attention_mass(cache, q, pos), np.full((1, S), H * n / S), rtol=1e-12)
    # brute force on one (head, query): a hand-written softmax
    cache.K[0] = r.standard_normal((S, H, hd))
    m = O.attention_mass(cache, q[:, :1], pos[:, :1])
    ref = np.zeros(S)
    for h in range(H):
        sc = [float(np.dot(q[0, 0, h], cache.K[0, j, h])) / math.sqrt(hd) for j in range(S)]
        mx = max(sc)
        e = [math.exp(v - mx) for v in sc]
        ref += np.array(e) / sum(e)
    np.testing.assert_allclose(m[0], ref, rtol=1e-12)
    # a DRAFT query sees the tail slot, whose mass is not a position's: totals drop
    cache2 = O.OracleCache(1, S, 2, H, hd)
    cache2.K[0] = r.standard_normal((S + 2, H, hd))
    view = np.array([[O.VIEW_BASE, O.VIEW_MASK, O.VIEW_BASE, O.VIEW_DRAFT]])
    pos2 = np.array([[2, 5, 7, 5]])
    m2 = O.attention_mass(cache2, q, pos2, view)
    assert m2.sum() < H * n - 1e-9


# -------------------------------------------------------------- partial softmax states
def test_partial_states_merge_to_full_attention():
    r = _rng(30)
    q, K, V = r.standard_normal((4, 2, 16)), r.standard_normal((20, 2, 16)), r.standard_normal((20, 2, 16))
    full = O.attention(q, K, V)
    for cut in (1, 7, 19):
        a = O.attention_partial(q, K[:cut], V[:cut])
        b = O.attention_partial(q, K[cut:], V[cut:])
        np.testing.assert_allclose(O.state_output(O.merge_states(a, b)), full, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(O.state_output(O.merge_states(b, a)), full, rtol=1e-12, atol=1e-14)
    # the same through visibility masks over the whole key set
    va = O.range_visible(4, 20, 0, 11)
    vb = O.range_visible(4, 20, 11, 20)
    st = O.merge_states(O.attention_partial(q, K, V, va), O.attention_partial(q, K, V, vb))
    np.testing.assert_allclose(O.state_output(st), full, rtol=1e-12, atol=1e-14)


def test_partial_state_closed_forms():
    r = _rng(31)
    q, K, V = r.standard_normal((3, 1, 8)), r.standard_normal((5, 1, 8)), r.standard_normal((5, 1, 8))
    O1, m1, l1 = O.attention_partial(q, K[2:3], V[2:3])  # one key: l = 1, O = v, m = its score
    np.testing.assert_allclose(l1, 1.0, rtol=0)
    np.testing.assert_allclose(O1[:, 0], np.broadcast_to(V[2, 0], (3, 8)), rtol=1e-15)
    np.testing.assert_allclose(m1[:, 0], q[:, 0] @ K[2, 0] / math.sqrt(8) / math.log(2.0), rtol=1e-13)
    Oe, me, le = O.attention_partial(q, K, V, O.range_visible(3, 5, 2, 2))  # empty range
    assert np.all(me == -np.inf) and np.all(le == 0) and np.all(Oe == 0)
    # m + log2(l) is the base-2 log-sum-exp of the scores
    _, m, l = O.attention_partial(q, K, V)
    sc = np.einsum("qhd,khd->qhk", q, K) / math.sqrt(8) / math.log(2.0)
    np.testing.assert_allclose(m + np.log2(l), np.logaddexp2.reduce(sc, axis=-1), rtol=1e-12)
    # merging with an empty state changes nothing
    st = O.attention_partial(q, K, V)
    mg = O.merge_states(st, (Oe, me, le))
    for x, y in zip(mg, st):
        np.testing.assert_allclose(x, y, rtol=1e-15)


# -------------------------------------------------------------- depth-wise refresh
def _elastic_setup(sigma, gamma, **kw):
    import workloads as W
    kw = dict(dict(batch=3, d_model=16, head_dim=8, max_pos=24, beta=4, gen_lo=8, k=3, act="f32"), **kw)
    wl = W.make_elastic(np.asarray(sigma, np.float32), seed=5, gamma=gamma, **kw)
    s = wl.shape
    caches = []
    for l in range(wl.n_layers):
        c = O.OracleCache(s.batch, s.max_pos, 0, s.n_heads, s.head_dim)
        O.write_rows(c, wl.w[l], wl.x_prev[l], np.tile(np.arange(s.max_pos, dtype=np.int32), (s.batch, 1)),
                     s.rope_theta)
        caches.append(c)
    return wl, caches


def _prefilled(wl, xs, l):
    """A fresh cache of layer l holding K/V of every slot computed from xs[l]."""
    s = wl.shape
    c = O.OracleCache(s.batch, s.max_pos, 0, s.n_heads, s.head_dim)
    O.write_rows(c, wl.w[l], xs[l], np.tile(np.arange(s.max_pos, dtype=np.int32), (s.batch, 1)), s.rope_theta)
    return c


def _outside_window(wl, b):
    keep = np.ones(wl.shape.max_pos, bool)
    keep[wl.win_lo[b]:wl.win_lo[b] + wl.beta] = False
    return keep


def test_elastic_never_refreshes_when_gamma_below_minus_one():
    wl, caches = _elastic_setup(np.full((3, 3), 2.0), gamma=-2.0)
    out, cos, flags, _ = O.elastic_step(caches, wl.w, wl.shape.rope_theta, wl.x_all, wl.win_lo, wl.beta, wl.mass,
                                        wl.k, wl.gamma)
    assert not flags.any()
    assert np.all(cos >= -1.0 - 1e-12) and np.all(cos <= 1.0 + 1e-12)
    for l in range(3):
        old, new = _prefilled(wl, wl.x_prev, l), _prefilled(wl, wl.x_all, l)
        for b in range(3):
            keep = _outside_window(wl, b)
            np.testing.assert_array_equal(caches[l].K[b][keep], old.K[b][keep])  # untouched
            np.testing.assert_allclose(caches[l].K[b][~keep], new.K[b][~keep], rtol=1e-13, atol=1e-15)  # window rows
            np.testing.assert_allclose(caches[l].V[b][~keep], new.V[b][~keep], rtol=1e-13, atol=1e-15)


def test_elastic_failing_first_layer_recomputes_every_deeper_layer():
    wl, caches = _elastic_setup(np.full((3, 3), 0.3), gamma=2.0)  # cos <= 1 < gamma: every test fails
    out, cos, flags, _ = O.elastic_step(caches, wl.w, wl.shape.rope_theta, wl.x_all, wl.win_lo, wl.beta, wl.mass,
                                        wl.k, wl.gamma)
    assert flags.all()
    old0 = _prefilled(wl, wl.x_prev, 0)
    for b in range(3):  # the failing layer itself keeps its cache outside the window
        keep = _outside_window(wl, b)
        np.testing.assert_array_equal(caches[0].K[b][keep], old0.K[b][keep])
    assert np.all(cos[0] < 0.999)
    for l in (1, 2):  # deeper layers: every slot from this step's states, so the probes match the cache
        new = _prefilled(wl, wl.x_all, l)
        np.testing.assert_allclose(caches[l].K, new.K, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(caches[l].V, new.V, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(cos[l], 1.0, atol=1e-12)


def test_elastic_refresh_starts_after_the_failing_layer_and_only_there():
    # sequence 0 barely drifts; sequence 1 drifts from layer 1 on; sequence 2 from layer 0 on
    sigma = np.array([[0.05, 0.05, 3.0], [0.05, 3.0, 3.0], [0.05, 3.0, 3.0]])
    wl, caches = _elastic_setup(sigma, gamma=0.9)
    out, cos, flags, _ = O.elastic_step(caches, wl.w, wl.shape.rope_theta, wl.x_all, wl.win_lo, wl.beta, wl.mass,
                                        wl.k, wl.gamma)
    # a recomputed layer matches its probes, so only the first failing layer flags
    np.testing.assert_array_equal(flags, [[0, 0, 1], [0, 1, 0], [0, 0, 0]])
    for l in range(3):
        old, new = _prefilled(wl, wl.x_prev, l), _prefilled(wl, wl.x_all, l)
        for b in range(3):
            keep = _outside_window(wl, b)
            refreshed = (b == 2 and l >= 1) or (b == 1 and l >= 2)
            ref = new if refreshed else old
            np.testing.assert_allclose(caches[l].K[b][keep], ref.K[b][keep], rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(caches[l].V[b][keep], ref.V[b][keep], rtol=1e-12, atol=1e-15)
    assert np.all(cos[1, 2] > 1 - 1e-12) and np.all(cos[2, 1:] > 1 - 1e-12)
