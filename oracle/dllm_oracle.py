"""Plain, slow, fp64 definition of one cached-attention denoising step.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline legs; never by the product path.

What is computed, and where the pages state it
----------------------------------------------
Sources (web pages, cited by title and section):

* [Flash-dLLM] "Flash-dLLM: IO-aware KV caching and parallel decoding"
  (skillfed.io news item).  Paragraph 2: the per-layer cache pipeline is QKV
  projection -> rotary embedding -> cache write -> attention.  Paragraph 3:
  Flash-Verify duplicates search-set tokens as a draft view and a mask view that
  cannot see each other.  Paragraph 4: tracking of the top-32 most-attended
  decoded tokens.  Paragraph 5: one flat preallocated cache.
* [LaCache] "LaCache: Exact Caching and Precision-Adaptive Inference for
  Diffusion Large Language Models" (gist.science summary).  Technical summary,
  Problem Statement: within a block the queries use bidirectional attention over
  the full context.  Methodology 1 (RoPECache): the cached per-token state is the
  projected, rotary-embedded K/V.  Methodology 2: per-group FP8 with groups of
  1x128 elements.
* [Elastic-Cache] "Elastic-Cache" (academy.dair.ai).  Core idea: cosine
  similarity between the cached and the recomputed K/V of the previous step's
  most-attended tokens; a value below gamma triggers a refresh.  Algorithm knobs:
  gamma = 0.9.
* [dLLM-Cache] "dLLM-Cache: Accelerating Diffusion Large Language Models with
  Adaptive Caching" (codewithpapers record): lists a ``rotate_half`` routine
  name, taken as evidence for the half-split rotary convention.

Readings where the pages are silent (each is listed in the design notes):

* rotary pairs are ``(i, i + hd/2)`` with angle ``p * theta^(-2i/hd)``;
* ``W_qkv`` is stored ``[3D][D]`` (row ``n`` = output feature ``n``), no bias;
  output columns ``[0,D)`` are Q, ``[D,2D)`` K, ``[2D,3D)`` V, head-major;
* the cache holds post-rotary K and V (not the attention output);
* every one of the ``max_pos`` regular slots is visible to every query, plus
  the draft-view tail slots written in this step (Flash-Verify rule below);
* Flash-Verify visibility: key j is visible to query q iff
  ``kview(j) == SHARED`` or ``kview(j) == qview(q)`` or
  ``(qview(q) == BASE and kview(j) == MASK)``;
  the r-th draft row of a sequence writes tail slot ``max_pos + r``;
* softmax scale ``1/sqrt(hd)``; the softmax is the textbook two-pass form;
* drift cosine is taken over the full ``D``-vector of each tracked token, K and
  V separately; top-k orders by mass descending, then position ascending, over
  positions outside the active block;
* FP8 groups are one (token, head, K|V) vector of ``hd = 128`` elements with
  ``scale = amax / 448`` and round-to-nearest-even, saturating at 448.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

__all__ = [
    "VIEW_BASE", "VIEW_DRAFT", "VIEW_MASK", "KVIEW_SHARED", "KVIEW_MASK", "KVIEW_DRAFT", "KVIEW_NONE",
    "rope_inv_freq", "rope", "project_qkv", "project_head", "row_slots", "key_views", "visible", "attention",
    "OracleCache", "write_rows", "step", "kv_topk", "cosine", "kv_drift", "attention_weights", "attention_mass",
    "attention_partial", "merge_states", "state_output", "range_visible",
    "refresh_due", "refresh_sequence", "elastic_step",
    "e4m3_decode", "e4m3_table", "e4m3_quantize", "fp8_group_quantize",
]

VIEW_BASE, VIEW_DRAFT, VIEW_MASK = 0, 1, 2
KVIEW_SHARED, KVIEW_MASK, KVIEW_DRAFT, KVIEW_NONE = 0, 1, 2, 3


# ------------------------------------------------------------------------------------
# Rotary embedding ([LaCache] Methodology 1 RoPECache: the cached state is taken after
# projection and rotary embedding; [dLLM-Cache] rotate_half -> half-split pairs).
# ------------------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta_i = theta ** (-2 i / hd), i = 0 .. hd/2 - 1, in fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(v: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate ``v[..., n, H, hd]`` at absolute positions ``positions[n]``.

    For each pair (x_i, x_{i+hd/2}) with angle a = p * theta_i:
        x_i'        = x_i cos a - x_{i+hd/2} sin a
        x_{i+hd/2}' = x_{i+hd/2} cos a + x_i sin a
    """
    v = np.asarray(v, dtype=np.float64)
    hd = v.shape[-1]
    half = hd // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]  # [n][1][hd/2], broadcast over heads
    s = np.sin(ang)[:, None, :]
    lo, hi = v[..., :half], v[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


# ------------------------------------------------------------------------------------
# QKV projection ([Flash-dLLM] paragraph 2: first stage of the per-layer pipeline).
# ------------------------------------------------------------------------------------

def project_qkv(x: np.ndarray, w: np.ndarray, n_heads: int):
    """``[q|k|v] = x . W_qkv`` with W stored ``[3D][D]``; returns q, k, v as [n][H][hd]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    D = w.shape[1]
    y = x @ w.T  # library matmul as one step; fp64 sums
    hd = D // n_heads
    q = y[:, 0:D].reshape(-1, n_heads, hd)
    k = y[:, D:2 * D].reshape(-1, n_heads, hd)
    v = y[:, 2 * D:3 * D].reshape(-1, n_heads, hd)
    return q, k, v


def project_head(x: np.ndarray, w: np.ndarray, n_heads: int, h: int):
    """q, k, v of head ``h`` only ([n][hd] each): output features part*D + h*hd + i."""
    x = np.asarray(x, dtype=np.float64)
    D = w.shape[1]
    hd = D // n_heads
    out = []
    for part in range(3):
        rows = np.asarray(w[part * D + h * hd: part * D + (h + 1) * hd], dtype=np.float64)
        out.append(x @ rows.T)
    return tuple(out)


# ------------------------------------------------------------------------------------
# Slots and visibility ([Flash-dLLM] paragraphs 3 and 5).
# ------------------------------------------------------------------------------------

def row_slots(positions: np.ndarray, view: Optional[np.ndarray], max_pos: int) -> np.ndarray:
    """Cache slot of each query row of one sequence.

    BASE and MASK rows write their own position; the r-th DRAFT row (in row order)
    writes tail slot ``max_pos + r``.
    """
    positions = np.asarray(positions, dtype=np.int64)
    slots = positions.copy()
    if view is None:
        return slots
    r = 0
    for t in range(len(positions)):
        if view[t] == VIEW_DRAFT:
            slots[t] = max_pos + r
            r += 1
    return slots


def key_views(positions: np.ndarray, view: Optional[np.ndarray], max_pos: int, n_slots: int) -> np.ndarray:
    """View tag of every cache slot of one sequence for this step.

    Regular slots are SHARED unless a MASK row of this step sits at that position;
    tail slots written by this step's DRAFT rows are DRAFT; other tail slots are NONE.
    """
    kv = np.full(n_slots, KVIEW_NONE, np.int64)
    kv[:max_pos] = KVIEW_SHARED
    if view is None:
        return kv
    slots = row_slots(positions, view, max_pos)
    for t in range(len(positions)):
        if view[t] == VIEW_MASK:
            kv[slots[t]] = KVIEW_MASK
        elif view[t] == VIEW_DRAFT:
            kv[slots[t]] = KVIEW_DRAFT
    return kv


def visible(qview: np.ndarray, kview: np.ndarray) -> np.ndarray:
    """Boolean [nq][nk]: key j visible to query q (reading of the Flash-Verify rule)."""
    q = np.asarray(qview)[:, None]
    k = np.asarray(kview)[None, :]
    same = ((q == VIEW_MASK) & (k == KVIEW_MASK)) | ((q == VIEW_DRAFT) & (k == KVIEW_DRAFT))
    base_sees_mask = (q == VIEW_BASE) & (k == KVIEW_MASK)
    return (k == KVIEW_SHARED) | same | base_sees_mask


# ------------------------------------------------------------------------------------
# Bidirectional attention ([LaCache] Problem Statement: full-context bidirectional
# attention inside a block; [Flash-Cache article] section 3.1: softmax(q k^T / sqrt d) v).
# ------------------------------------------------------------------------------------

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, vis: Optional[np.ndarray] = None) -> np.ndarray:
    """``o = softmax(q K^T / sqrt(hd) masked by vis) V`` per head, two-pass softmax.

    q [nq][H][hd], K/V [nk][H][hd], vis [nq][nk] bool or None (all visible).
    Returns [nq][H][hd] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hd = q.shape[-1]
    s = np.einsum("qhd,khd->hqk", q, K) / math.sqrt(hd)
    if vis is not None:
        s = np.where(np.asarray(vis, bool)[None, :, :], s, -np.inf)
    m = s.max(axis=-1, keepdims=True)  # pass 1: max
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row has no visible key")
    e = np.exp(s - m)  # pass 2: exponentials and their sum
    p = e / e.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, V)


def attention_weights(q: np.ndarray, K: np.ndarray, vis: Optional[np.ndarray] = None) -> np.ndarray:
    """softmax(q K^T / sqrt(hd)) per head, masked by vis: [H][nq][nk] fp64 (rows sum to 1)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    s = np.einsum("qhd,khd->hqk", q, K) / math.sqrt(q.shape[-1])
    if vis is not None:
        s = np.where(np.asarray(vis, bool)[None, :, :], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


# ------------------------------------------------------------------------------------
# Partial softmax states ([LaCache] Methodology 1, FACache: the running maximum m, the
# normaliser l and the unnormalised accumulator O of online softmax, kept for key blocks
# that do not change and combined with the blocks that do).  Base-2 units, as the
# kernels keep them: s = q.k / sqrt(hd) * log2(e).
# ------------------------------------------------------------------------------------

LOG2E = 1.0 / math.log(2.0)


def range_visible(n_q: int, n_keys: int, lo: int, hi: int) -> np.ndarray:
    """Boolean [n_q][n_keys]: keys lo <= j < hi visible to every query."""
    v = np.zeros((n_q, n_keys), bool)
    v[:, max(lo, 0):max(min(hi, n_keys), 0)] = True
    return v


def attention_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray, vis: Optional[np.ndarray] = None):
    """State of q [nq][H][hd] over keys K, V [nk][H][hd] (masked by vis [nq][nk]):
    m = max_j s_j, l = sum_j 2^(s_j - m), O = sum_j 2^(s_j - m) v_j.
    Returns (O [nq][H][hd], m [nq][H], l [nq][H]); m = -inf, l = 0, O = 0 without keys."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    s = np.einsum("qhd,khd->qhk", q, K) / math.sqrt(q.shape[-1]) * LOG2E
    if vis is not None:
        s = np.where(np.asarray(vis, bool)[:, None, :], s, -np.inf)
    m = s.max(axis=-1) if s.shape[-1] else np.full(s.shape[:2], -np.inf)
    w = np.where(np.isfinite(m)[..., None], np.exp2(s - np.where(np.isfinite(m), m, 0.0)[..., None]), 0.0)
    return np.einsum("qhk,khd->qhd", w, V), m, w.sum(axis=-1)


def merge_states(a, b):
    """Combine two states of the same rows over disjoint key sets."""
    Oa, ma, la = a
    Ob, mb, lb = b
    M = np.maximum(ma, mb)
    Mu = np.where(np.isfinite(M), M, 0.0)
    wa = np.where(np.isfinite(ma), np.exp2(ma - Mu), 0.0)
    wb = np.where(np.isfinite(mb), np.exp2(mb - Mu), 0.0)
    return Oa * wa[..., None] + Ob * wb[..., None], M, la * wa + lb * wb


def state_output(st) -> np.ndarray:
    """Normalised attention output O / l (0 where l = 0)."""
    O, _, l = st
    return np.where(l[..., None] > 0, O / np.where(l > 0, l, 1.0)[..., None], 0.0)


# ------------------------------------------------------------------------------------
# The flat per-layer cache and one step ([Flash-dLLM] paragraphs 2 and 5).
# ------------------------------------------------------------------------------------

class OracleCache:
    """K/V of one layer for B sequences, ``max_pos + tail_slots`` slots each, fp64.

    ``kv="e4m3"``: the cache stores FP8 ([LaCache] Methodology 2, per-group FP8): every
    (token, head) vector of K and of V written into it is one quantisation group and
    is kept as its dequantised value ``e4m3(x / s) * s`` with ``s = amax / 448``.
    ``kv="exact"`` keeps the fp64 values.
    """

    def __init__(self, batch: int, max_pos: int, tail_slots: int, n_heads: int, head_dim: int, kv: str = "exact"):
        self.B, self.S, self.T, self.H, self.hd = batch, max_pos, tail_slots, n_heads, head_dim
        if kv not in ("exact", "e4m3"):
            raise ValueError(kv)
        self.kv = kv
        n = max_pos + tail_slots
        self.K = np.zeros((batch, n, n_heads, head_dim))
        self.V = np.zeros((batch, n, n_heads, head_dim))
        self.written = np.zeros((batch, n), bool)

    def stored(self, vec: np.ndarray) -> np.ndarray:
        """What the cache keeps for one (token, head) K or V vector."""
        if self.kv == "e4m3":
            return fp8_group_quantize(vec)[0]
        return vec


def write_rows(cache: OracleCache, w: np.ndarray, x: np.ndarray, positions: np.ndarray, theta: float,
               slots: Optional[np.ndarray] = None):
    """Project rows ``x[B][n][D]`` at ``positions[B][n]``, rotate K, store K/V at ``slots``.

    Returns the rotated q of every row, [B][n][H][hd].
    """
    B = x.shape[0]
    qs = []
    for b in range(B):
        q, k, v = project_qkv(x[b], w, cache.H)
        q = rope(q, positions[b], theta)
        k = rope(k, positions[b], theta)
        sl = positions[b] if slots is None else slots[b]
        for t, s in enumerate(sl):
            if not (0 <= s < cache.S + cache.T):
                raise IndexError("slot out of range")
            for h in range(cache.H):
                cache.K[b, s, h] = cache.stored(k[t, h])
                cache.V[b, s, h] = cache.stored(v[t, h])
            cache.written[b, s] = True
        qs.append(q)
    return np.stack(qs)


def step(cache: OracleCache, w: np.ndarray, theta: float, x: np.ndarray, positions: np.ndarray,
         view: Optional[np.ndarray] = None, kv_x: Optional[np.ndarray] = None,
         kv_pos: Optional[np.ndarray] = None, probe: bool = False):
    """One layer-step: project, rotate, write, then attend.

    * ``kv_x/kv_pos`` (optional): K/V-only rows.  With ``probe=False`` they are written
      to the cache (a refresh); with ``probe=True`` they are returned as probe K/V
      ``[B][n_kv][2][D]`` and the cache is left untouched.
    * ``x/positions/view``: query rows; their K/V go to ``row_slots`` and each row
      attends over all visible slots after all writes of the step.
    Returns ``(out [B][n][D], probe_kv or None)``.
    """
    B, n, D = x.shape
    H, hd = cache.H, cache.hd
    probe_kv = None
    if kv_x is not None and kv_x.shape[1] > 0:
        if probe:
            probe_kv = np.empty((B, kv_x.shape[1], 2, D))
            for b in range(B):
                _, k, v = project_qkv(kv_x[b], w, H)
                k = rope(k, kv_pos[b], theta)
                probe_kv[b, :, 0] = k.reshape(-1, D)
                probe_kv[b, :, 1] = v.reshape(-1, D)
        else:
            write_rows(cache, w, kv_x, kv_pos, theta)
    out = np.zeros((B, n, D))
    if n == 0:
        return out, probe_kv
    slots = np.stack([row_slots(positions[b], None if view is None else view[b], cache.S) for b in range(B)])
    q = write_rows(cache, w, x, positions, theta, slots)
    n_slots = cache.S + cache.T
    for b in range(B):
        vb = None if view is None else view[b]
        kview = key_views(positions[b], vb, cache.S, n_slots)
        qview = np.zeros(n, np.int64) if vb is None else np.asarray(vb, np.int64)
        vis = visible(qview, kview)
        used = vis.any(axis=0)
        if not np.all(cache.written[b][used]):
            raise ValueError("a visible slot was never written")
        out[b] = attention(q[b], cache.K[b], cache.V[b], vis).reshape(n, D)
    return out, probe_kv


def attention_mass(cache: OracleCache, q: np.ndarray, positions: np.ndarray,
                   view: Optional[np.ndarray] = None) -> np.ndarray:
    """Attention mass each cached position receives in this step: for sequence b and
    regular slot j, the sum over heads and query rows of the softmax weight of key j
    ([Flash-dLLM] paragraph 4 and [Elastic-Cache] Core idea track the most-attended
    tokens).  q: rotated queries [B][n][H][hd] (as ``write_rows`` returns them), read
    against the cache after the step's writes.  Returns [B][max_pos] fp64."""
    B, n = positions.shape
    mass = np.zeros((B, cache.S))
    for b in range(B):
        vb = None if view is None else view[b]
        kview = key_views(positions[b], vb, cache.S, cache.S + cache.T)
        qview = np.zeros(n, np.int64) if vb is None else np.asarray(vb, np.int64)
        p = attention_weights(q[b], cache.K[b], visible(qview, kview))
        mass[b] = p.sum(axis=(0, 1))[:cache.S]
    return mass


# ------------------------------------------------------------------------------------
# Tracking and drift ([Flash-dLLM] paragraph 4; [Elastic-Cache] Core idea).
# ------------------------------------------------------------------------------------

def kv_topk(mass: np.ndarray, block_lo: np.ndarray, block_len: int, k: int) -> np.ndarray:
    """Positions of the k largest masses outside the active block, per sequence.

    Order: mass descending, ties broken by the lower position first.  [B][k] int32.
    """
    mass = np.asarray(mass)
    B, S = mass.shape
    out = np.empty((B, k), np.int32)
    for b in range(B):
        cand = [p for p in range(S) if not (block_lo[b] <= p < block_lo[b] + block_len)]
        if len(cand) < k:
            raise ValueError("fewer candidates than k")
        cand.sort(key=lambda p: (-float(mass[b, p]), p))
        out[b] = cand[:k]
    return out


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """<a, b> / (|a| |b|) in fp64."""
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.dot(a, b) / (math.sqrt(np.dot(a, a)) * math.sqrt(np.dot(b, b))))


def kv_drift(cache: OracleCache, idx: np.ndarray, probe_kv: np.ndarray) -> np.ndarray:
    """cos[B][k][2]: cosine of cached vs probe K (index 0) and V (index 1) per token."""
    B, k = idx.shape
    D = cache.H * cache.hd
    cos = np.empty((B, k, 2))
    for b in range(B):
        for j in range(k):
            s = int(idx[b, j])
            cos[b, j, 0] = cosine(cache.K[b, s].reshape(D), probe_kv[b, j, 0])
            cos[b, j, 1] = cosine(cache.V[b, s].reshape(D), probe_kv[b, j, 1])
    return cos


# ------------------------------------------------------------------------------------
# Depth-wise refresh over the layers of one step ([Elastic-Cache] Core idea: when the
# drift test of the most-attended tokens fails at layer l, the layers after l are
# recomputed; shallow layers keep their caches.  Algorithm knobs: threshold gamma,
# sliding window of beta active tokens).
# ------------------------------------------------------------------------------------

def refresh_due(flags: np.ndarray, layer: int) -> np.ndarray:
    """Sequences whose cache of ``layer`` is recomputed this step: those whose drift
    test failed in some layer before it.  flags: [n_layers][B] (rows >= layer unused)."""
    flags = np.asarray(flags)
    if layer == 0:
        return np.zeros(flags.shape[1], bool)
    return flags[:layer].astype(bool).any(axis=0)


def refresh_sequence(cache: OracleCache, w: np.ndarray, x_seq: np.ndarray, b: int, theta: float):
    """Recompute K/V of every regular slot of sequence b from its hidden states
    x_seq [max_pos][D] (the full-sequence recompute of a refreshed layer)."""
    _, k, v = project_qkv(x_seq, w, cache.H)
    pos = np.arange(cache.S)
    k = rope(k, pos, theta)
    for s in range(cache.S):
        for h in range(cache.H):
            cache.K[b, s, h] = cache.stored(k[s, h])
            cache.V[b, s, h] = cache.stored(v[s, h])
        cache.written[b, s] = True


def elastic_step(caches, ws, theta: float, x_all, win_lo: np.ndarray, beta: int, masses, k: int, gamma: float,
                 with_mass: bool = False):
    """One denoising step over the layers in order.  Per layer l:

    1. sequences due for refresh (``refresh_due``) get every regular slot of layer l
       recomputed from ``x_all[l]``;
    2. the tracked tokens are the top-k of ``masses[l]`` outside the window
       ``[win_lo[b], win_lo[b] + beta)``;
    3. the window rows of ``x_all[l]`` are projected, written and attend over the cache
       (``step``); the tracked rows are projected as probes;
    4. the drift test compares the cached and probe K/V of the tracked tokens; the
       sequence's flag is ``min cos < gamma``.

    caches: one OracleCache per layer (modified in place); ws: weights per layer;
    x_all: per layer [B][max_pos][D]; masses: per layer [B][max_pos].
    Returns (out [L][B][beta][D], cos [L][B][k][2], flags [L][B] int32, mass [L][B][max_pos]
    or None): the mass each slot receives from the window's queries after the step's
    writes (``attention_mass``)."""
    L = len(caches)
    B = x_all[0].shape[0]
    positions = (np.asarray(win_lo)[:, None] + np.arange(beta)[None, :]).astype(np.int32)
    flags = np.zeros((L, B), np.int32)
    outs, coss, mass_out = [], [], []
    for l in range(L):
        c = caches[l]
        due = refresh_due(flags, l)
        for b in np.nonzero(due)[0]:
            refresh_sequence(c, ws[l], x_all[l][b], int(b), theta)
        idx = kv_topk(masses[l], win_lo, beta, k)
        x_win = np.stack([x_all[l][b][positions[b]] for b in range(B)])
        x_trk = np.stack([x_all[l][b][idx[b]] for b in range(B)])
        out, probe = step(c, ws[l], theta, x_win, positions, kv_x=x_trk, kv_pos=idx, probe=True)
        if with_mass:
            q = np.stack([rope(project_qkv(x_win[b], ws[l], c.H)[0], positions[b], theta) for b in range(B)])
            mass_out.append(attention_mass(c, q, positions))
        cos = kv_drift(c, idx, probe)
        flags[l] = (cos.min(axis=(1, 2)) < gamma).astype(np.int32)
        outs.append(out)
        coss.append(cos)
    return np.stack(outs), np.stack(coss), flags, (np.stack(mass_out) if with_mass else None)


# ------------------------------------------------------------------------------------
# FP8 E4M3 ([LaCache] Methodology 2: per-group FP8 with 1x128 groups).  Written from
# the OCP 8-bit floating point definition of E4M3: 1 sign, 4 exponent bits with bias
# 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448, smallest
# subnormal 2^-9.
# ------------------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    code = int(code) & 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)])


def e4m3_quantize(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (ties to even mantissa), saturating to +-448; returns fp64 values."""
    y = np.asarray(y, np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)  # a = f * 2**ex with f in [0.5, 1)
    e = np.clip(ex - 1, -6, 8)  # unbiased exponent of the binade, subnormals share -6
    quantum = np.ldexp(1.0, e - 3)  # spacing of values in that binade
    q = np.round(a / quantum) * quantum  # numpy rounds half to even
    q = np.minimum(q, 448.0)
    return np.sign(y) * q


def fp8_group_quantize(v: np.ndarray):
    """Per-group quantisation of a vector group: scale = amax/448 (1 if amax = 0).

    Returns (dequantised values fp64, scale).
    """
    v = np.asarray(v, np.float64)
    amax = float(np.max(np.abs(v)))
    scale = amax / 448.0 if amax > 0 else 1.0
    return e4m3_quantize(v / scale) * scale, scale
