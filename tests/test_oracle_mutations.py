"""Planted mistakes in the oracle must each fail at least one pin.

Each case swaps one oracle function for a plausibly wrong variant (on the CPU, for
the duration of the test only) and checks that the named pins reject it.
"""
import math

import numpy as np
import pytest

import oracle as O
import oracle.dllm_oracle as OD
from tests import test_oracle_pins as P


def _rope_adjacent_pairs(v, positions, theta):
    v = np.asarray(v, np.float64)
    hd = v.shape[-1]
    ang = np.asarray(positions, np.float64)[:, None] * O.rope_inv_freq(hd, theta)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    ev, od = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = ev * c - od * s
    out[..., 1::2] = od * c + ev * s
    return out


def _rope_wrong_sign(v, positions, theta):
    v = np.asarray(v, np.float64)
    half = v.shape[-1] // 2
    ang = np.asarray(positions, np.float64)[:, None] * O.rope_inv_freq(v.shape[-1], theta)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    lo, hi = v[..., :half], v[..., half:]
    return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)


def _inv_freq_wrong_exponent(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -i / head_dim)


def _project_kv_swapped(x, w, n_heads):
    q, k, v = _orig_project(x, w, n_heads)
    return q, v, k


def _attention_scale_1_over_d(q, K, V, vis=None):
    q = np.asarray(q, float)
    return _att(q, np.asarray(K, float), np.asarray(V, float), vis, 1.0 / q.shape[-1])


def _att(q, K, V, vis, scale, subtract_max=True):
    s = np.einsum("qhd,khd->hqk", q, K) * scale
    if vis is not None:
        s = np.where(np.asarray(vis, bool)[None], s, -np.inf)
    m = s.max(-1, keepdims=True) if subtract_max else 0.0
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s - m)
        p = e / e.sum(-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, V)


def _attention_no_max(q, K, V, vis=None):
    return _att(np.asarray(q, float), np.asarray(K, float), np.asarray(V, float), vis,
                1.0 / math.sqrt(np.shape(q)[-1]), subtract_max=False)


def _visible_base_blind_to_mask(qview, kview):
    q = np.asarray(qview)[:, None]
    k = np.asarray(kview)[None, :]
    return (k == O.KVIEW_SHARED) | ((q == O.VIEW_MASK) & (k == O.KVIEW_MASK)) | ((q == O.VIEW_DRAFT) & (k == O.KVIEW_DRAFT))


def _topk_ties_high(mass, block_lo, block_len, k):
    B, S = mass.shape
    out = np.empty((B, k), np.int32)
    for b in range(B):
        cand = [p for p in range(S) if not (block_lo[b] <= p < block_lo[b] + block_len)]
        cand.sort(key=lambda p: (-float(mass[b, p]), -p))
        out[b] = cand[:k]
    return out


def _e4m3_round_away(y):
    y = np.asarray(y, np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)
    e = np.clip(ex - 1, -6, 8)
    quantum = np.ldexp(1.0, e - 3)
    q = np.floor(a / quantum + 0.5) * quantum
    return np.sign(y) * np.minimum(q, 448.0)


_orig_project = OD.project_qkv

CASES = [
    ("rope", _rope_adjacent_pairs, [P.test_rope_golden_pairing_and_frequency]),
    ("rope", _rope_wrong_sign, [P.test_rope_golden_hd2]),
    ("rope_inv_freq", _inv_freq_wrong_exponent, [P.test_rope_golden_pairing_and_frequency]),
    ("project_qkv", _project_kv_swapped, [P.test_projection_identity_weights]),
    ("attention", _attention_scale_1_over_d, [P.test_attention_golden_weights]),
    ("attention", _attention_no_max, [P.test_attention_permutation_invariant_and_shift_stable]),
    ("visible", _visible_base_blind_to_mask, [P.test_visibility_truth_table]),
    ("kv_topk", _topk_ties_high, [P.test_topk_ties_take_lower_position_and_permutation_equivariance]),
    ("e4m3_quantize", _e4m3_round_away, [P.test_e4m3_quantize_matches_library_rounding_in_range]),
]


@pytest.mark.parametrize("name,bad,pins", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pins):
    monkeypatch.setattr(OD, name, bad)
    monkeypatch.setattr(O, name, bad)
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError):
            caught += 1
    assert caught == len(pins), f"planted mistake in {name} slipped past {pins}"


def _refresh_due_late(flags, layer):
    flags = np.asarray(flags)
    if layer <= 1:
        return np.zeros(flags.shape[1], bool)
    return flags[:layer - 1].astype(bool).any(axis=0)


def _refresh_due_every_sequence(flags, layer):
    flags = np.asarray(flags)
    any_failed = bool(flags[:layer].any()) if layer > 0 else False
    return np.full(flags.shape[1], any_failed)


REFRESH_CASES = [
    (_refresh_due_late, P.test_elastic_refresh_starts_after_the_failing_layer_and_only_there),
    (_refresh_due_every_sequence, P.test_elastic_refresh_starts_after_the_failing_layer_and_only_there),
    (_refresh_due_late, P.test_elastic_failing_first_layer_recomputes_every_deeper_layer),
]


@pytest.mark.parametrize("bad,pin", REFRESH_CASES, ids=[f"{c[0].__name__}-{c[1].__name__}" for c in REFRESH_CASES])
def test_planted_refresh_mistake_is_caught(monkeypatch, bad, pin):
    monkeypatch.setattr(OD, "refresh_due", bad)
    monkeypatch.setattr(O, "refresh_due", bad)
    with pytest.raises(AssertionError):
        pin()


def _merge_states_natural_base(a, b):
    Oa, ma, la = a
    Ob, mb, lb = b
    M = np.maximum(ma, mb)
    Mu = np.where(np.isfinite(M), M, 0.0)
    wa = np.where(np.isfinite(ma), np.exp(ma - Mu), 0.0)
    wb = np.where(np.isfinite(mb), np.exp(mb - Mu), 0.0)
    return Oa * wa[..., None] + Ob * wb[..., None], M, la * wa + lb * wb


def _merge_states_sums_not_rescaled(a, b):
    Oa, ma, la = a
    Ob, mb, lb = b
    M = np.maximum(ma, mb)
    Mu = np.where(np.isfinite(M), M, 0.0)
    wa = np.where(np.isfinite(ma), np.exp2(ma - Mu), 0.0)
    wb = np.where(np.isfinite(mb), np.exp2(mb - Mu), 0.0)
    return Oa * wa[..., None] + Ob * wb[..., None], M, la + lb


def _attention_partial_natural_units(q, K, V, vis=None):
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    s = np.einsum("qhd,khd->qhk", q, K) / math.sqrt(q.shape[-1])
    if vis is not None:
        s = np.where(np.asarray(vis, bool)[:, None, :], s, -np.inf)
    m = s.max(axis=-1) if s.shape[-1] else np.full(s.shape[:2], -np.inf)
    w = np.where(np.isfinite(m)[..., None], np.exp(s - np.where(np.isfinite(m), m, 0.0)[..., None]), 0.0)
    return np.einsum("qhk,khd->qhd", w, V), m, w.sum(axis=-1)


STATE_CASES = [
    ("merge_states", _merge_states_natural_base, P.test_partial_states_merge_to_full_attention),
    ("merge_states", _merge_states_sums_not_rescaled, P.test_partial_states_merge_to_full_attention),
    ("attention_partial", _attention_partial_natural_units, P.test_partial_state_closed_forms),
]


@pytest.mark.parametrize("name,bad,pin", STATE_CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in STATE_CASES])
def test_planted_state_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(OD, name, bad)
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        pin()


def _row_slots_drafts_reversed(positions, view, max_pos):
    positions = np.asarray(positions, dtype=np.int64)
    slots = positions.copy()
    if view is None:
        return slots
    drafts = [t for t in range(len(positions)) if view[t] == O.VIEW_DRAFT]
    for r, t in enumerate(drafts):
        slots[t] = max_pos + len(drafts) - 1 - r
    return slots


def _drift_per_head_mean(cache, idx, probe_kv):
    B, k = idx.shape
    H, hd = cache.H, cache.hd
    cos = np.empty((B, k, 2))
    for b in range(B):
        for j in range(k):
            s = int(idx[b, j])
            for c, X in enumerate((cache.K, cache.V)):
                pr = np.asarray(probe_kv[b, j, c]).reshape(H, hd)
                cos[b, j, c] = np.mean([O.cosine(X[b, s, h], pr[h]) for h in range(H)])
    return cos


def _drift_kv_swapped(cache, idx, probe_kv):
    return _orig_drift(cache, idx, probe_kv)[..., ::-1]


_orig_drift = OD.kv_drift

SLOT_DRIFT_CASES = [
    ("row_slots", _row_slots_drafts_reversed, P.test_verify_rth_draft_row_writes_tail_slot_r),
    ("kv_drift", _drift_per_head_mean, P.test_drift_closed_form_over_the_whole_token_vector),
    ("kv_drift", _drift_kv_swapped, P.test_drift_closed_form_over_the_whole_token_vector),
]


@pytest.mark.parametrize("name,bad,pin", SLOT_DRIFT_CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in SLOT_DRIFT_CASES])
def test_planted_slot_or_drift_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(OD, name, bad)
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        pin()


def test_reversed_draft_slots_pass_the_written_set_pin(monkeypatch):
    """Why the contents pin is needed: the written-set pin alone cannot see the order."""
    monkeypatch.setattr(OD, "row_slots", _row_slots_drafts_reversed)
    monkeypatch.setattr(O, "row_slots", _row_slots_drafts_reversed)
    P.test_verify_draft_rows_use_tail_slots()


def _mass_mean_over_heads(cache, q, positions, view=None):
    return _orig_mass(cache, q, positions, view) / cache.H


def _group_scale_fnuz_max(v):
    v = np.asarray(v, np.float64)
    amax = float(np.max(np.abs(v)))
    scale = amax / 240.0 if amax > 0 else 1.0
    return O.e4m3_quantize(v / scale) * scale, scale


def _e4m3_decode_bias_8(code):
    code = int(code) & 0xFF
    sgn = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sgn * m * 2.0 ** -10
    return sgn * (1.0 + m / 8.0) * 2.0 ** (e - 8)


_orig_mass = OD.attention_mass

MASS_FP8_CASES = [
    ("attention_mass", _mass_mean_over_heads, P.test_attention_mass_totals_uniform_keys_and_views),
    ("fp8_group_quantize", _group_scale_fnuz_max, P.test_fp8_group_quantize_scale_and_zero_group),
    ("e4m3_decode", _e4m3_decode_bias_8, P.test_e4m3_named_values),
]


@pytest.mark.parametrize("name,bad,pin", MASS_FP8_CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in MASS_FP8_CASES])
def test_planted_mass_or_fp8_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(OD, name, bad)
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        pin()


def _elastic_step_window_early(caches, ws, theta, x_all, win_lo, beta, masses, k, gamma, with_mass=False):
    # the multi-layer step with its window one position early (positions win_lo - 1 ...)
    L = len(caches)
    B = x_all[0].shape[0]
    positions = (np.asarray(win_lo)[:, None] - 1 + np.arange(beta)[None, :]).astype(np.int32)
    flags = np.zeros((L, B), np.int32)
    outs, coss = [], []
    for l in range(L):
        c = caches[l]
        for b in np.nonzero(O.refresh_due(flags, l))[0]:
            O.refresh_sequence(c, ws[l], x_all[l][b], int(b), theta)
        idx = O.kv_topk(masses[l], win_lo, beta, k)
        x_win = np.stack([x_all[l][b][positions[b]] for b in range(B)])
        x_trk = np.stack([x_all[l][b][idx[b]] for b in range(B)])
        out, probe = O.step(c, ws[l], theta, x_win, positions, kv_x=x_trk, kv_pos=idx, probe=True)
        cos = O.kv_drift(c, idx, probe)
        flags[l] = (cos.min(axis=(1, 2)) < gamma).astype(np.int32)
        outs.append(out)
        coss.append(cos)
    return np.stack(outs), np.stack(coss), flags, None


def test_planted_early_window_is_caught(monkeypatch):
    monkeypatch.setattr(OD, "elastic_step", _elastic_step_window_early)
    monkeypatch.setattr(O, "elastic_step", _elastic_step_window_early)
    with pytest.raises(AssertionError):
        P.test_elastic_never_refreshes_when_gamma_below_minus_one()
