"""Seeded synthetic inputs for the cached-attention denoising step.

This module only draws random numbers and rounds them to the storage type of the
workload (fp32 or bf16).  It holds none of the method's arithmetic: no
projection, rotation, attention, selection or similarity is computed here.  Both
the fp64 oracle (through the tests) and the CUDA path consume exactly the arrays
it returns, so both sides see bit-identical inputs.

Every hidden-state row is drawn from its own counter-keyed generator
``numpy.random.default_rng([seed, stream, b, p])`` so that any single row of a
full-size workload can be regenerated without drawing the rest, which is what the
sampled full-size parity tests rely on.

Workload recipe (shapes are those of a LLaDA-8B attention layer where stated):

* hidden states ``x ~ N(0, 1)``, one row per (sequence, position, stream);
* ``W_qkv ~ N(0, 0.02^2)`` stored as ``[3D][D]`` (row ``n`` = output feature
  ``n``; columns ``[0, D)`` of the mathematical ``[D x 3D]`` matrix are Q,
  ``[D, 2D)`` K and ``[2D, 3D)`` V, head-major inside each);
* active block of ``block`` consecutive positions at ``block_lo[b]`` (fixed or a
  seeded block-aligned offset in the generation region);
* previous-step attention mass over all cache positions ~ Dirichlet(0.1);
* Flash-Verify: a seeded subset of the block is the search set; its draft view
  rows are fresh N(0, 1) rows and its mask view rows all equal one seeded
  N(0, 1) "mask embedding" row;
* drift probes: the current hidden state of a tracked token is its prefill row
  plus ``0.1 * N(0, 1)`` noise.
* multi-layer steps (``make_elastic``): per layer, weights as above, the hidden
  states the cache was built from ``x_prev ~ N(0, 1)`` at every position, and this
  step's states ``x_all = x_prev + sigma[l][b] * N(0, 1)``: ``sigma`` sets how far
  each (layer, sequence) drifts; a window of ``beta`` positions per sequence at a
  seeded block-aligned offset; previous-step mass ~ Dirichlet(0.1) per layer.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Row view tags of the step (shared vocabulary with the C header).
VIEW_BASE = 0
VIEW_DRAFT = 1
VIEW_MASK = 2

# Generator stream ids.
_S_WEIGHT = 1
_S_PREFILL = 2
_S_BLOCK = 3
_S_DRAFT = 4
_S_MASKEMB = 5
_S_NOISE = 6
_S_OFFSET = 7
_S_SEARCH = 8
_S_MASS = 9
_S_LAYER_PREV = 10
_S_LAYER_NOISE = 11


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if not np.all(np.isfinite(a)):
        raise ValueError("round_bf16 expects finite values")
    u = a.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    r = ((u + bias) >> np.uint32(16)) << np.uint32(16)
    return r.view(np.float32).reshape(np.shape(a))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of float32 values that are exactly representable in bf16."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("values are not bf16-representable; round them first")
    return (u >> np.uint32(16)).astype(np.uint16).reshape(np.shape(a))


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), *[int(k) for k in key]])


@dataclasses.dataclass
class Shape:
    batch: int
    d_model: int
    n_heads: int
    head_dim: int
    max_pos: int
    tail_slots: int
    rope_theta: float
    act: str  # "f32" | "bf16"   (activations, weights, Q/out)
    kv: str  # "f32" | "bf16" | "e4m3"   (cache storage)

    @property
    def D(self) -> int:
        return self.n_heads * self.head_dim

    def __post_init__(self):
        if self.n_heads * self.head_dim != self.d_model:
            raise ValueError("d_model must equal n_heads * head_dim")


@dataclasses.dataclass
class Workload:
    """One denoising step of one layer, plus what precedes it.

    ``pre_x/pre_pos``: rows written to the cache before the step (K/V only).
    ``x/positions/view``: the step's query rows (Q, K, V; attend over the cache).
    ``kv_x/kv_pos``: the step's K/V-only rows (full refresh), or None.
    ``mass/block_lo/block_len/drift_k``: drift inputs, or None.
    """

    name: str
    shape: Shape
    seed: int
    w: np.ndarray  # [3D][D] float32 (storage-rounded)
    block_lo: np.ndarray  # int32 [B]
    block_len: int
    pre_x: Optional[np.ndarray]  # [B][n_pre][D]
    pre_pos: Optional[np.ndarray]  # int32 [B][n_pre]
    x: np.ndarray  # [B][n_tok][D]
    positions: np.ndarray  # int32 [B][n_tok]
    view: Optional[np.ndarray]  # uint8 [B][n_tok] or None (all BASE)
    kv_x: Optional[np.ndarray] = None  # [B][n_kv][D]
    kv_pos: Optional[np.ndarray] = None  # int32 [B][n_kv]
    mass: Optional[np.ndarray] = None  # float32 [B][S]
    drift_k: int = 0
    gamma: float = 0.9

    # ---- helpers that draw rows on demand (used by sampled full-size tests) ----
    def prefill_row(self, b: int, p: int) -> np.ndarray:
        return hidden_row(self.seed, _S_PREFILL, b, p, self.shape)

    def probe_rows(self, idx: np.ndarray, b0: int = 0) -> np.ndarray:
        """Current hidden states of tracked tokens: prefill row + 0.1 * N(0,1).

        ``idx`` is ``[n][k]`` positions of sequences ``b0 .. b0+n-1``; returns
        ``[n][k][D]`` storage-rounded.
        """
        B, k = idx.shape
        out = np.empty((B, k, self.shape.D), np.float32)
        for i in range(B):
            b = b0 + i
            for j in range(k):
                p = int(idx[i, j])
                base = _rng(self.seed, _S_PREFILL, b, p).standard_normal(self.shape.D, dtype=np.float32)
                noise = _rng(self.seed, _S_NOISE, b, p).standard_normal(self.shape.D, dtype=np.float32)
                out[i, j] = base + np.float32(0.1) * noise
        return _store(out, self.shape.act)


def _store(a: np.ndarray, act: str) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return round_bf16(a) if act == "bf16" else a


def hidden_row(seed: int, stream: int, b: int, p: int, shape: Shape) -> np.ndarray:
    r = _rng(seed, stream, b, p).standard_normal(shape.D, dtype=np.float32)
    return _store(r, shape.act)


def _rows(seed: int, stream: int, pos: np.ndarray, shape: Shape) -> np.ndarray:
    B, n = pos.shape
    out = np.empty((B, n, shape.D), np.float32)
    for b in range(B):
        for i in range(n):
            out[b, i] = _rng(seed, stream, b, int(pos[b, i])).standard_normal(shape.D, dtype=np.float32)
    return _store(out, shape.act)


def weights(shape: Shape, seed: int) -> np.ndarray:
    w = _rng(seed, _S_WEIGHT).standard_normal((3 * shape.D, shape.D), dtype=np.float32)
    return _store(w * np.float32(0.02), shape.act)


def _block_offsets(seed: int, B: int, lo: int, hi: int, block: int, fixed: Optional[int]) -> np.ndarray:
    if fixed is not None:
        return np.full(B, fixed, np.int32)
    n_choices = (hi - lo) // block
    u = _rng(seed, _S_OFFSET).integers(0, n_choices, size=B)
    return (lo + block * u).astype(np.int32)


def _others(B: int, S: int, block_lo: np.ndarray, block: int) -> np.ndarray:
    rows = []
    for b in range(B):
        p = np.arange(S, dtype=np.int32)
        keep = (p < block_lo[b]) | (p >= block_lo[b] + block)
        rows.append(p[keep])
    return np.stack(rows)


# ----------------------------------------------------------------------------------
# The five workloads.  ``overrides`` shrink a workload for oracle-sized parity cases
# while keeping its structure (e.g. batch=2, d_model=512, max_pos=300).
# ----------------------------------------------------------------------------------

def _shape(d: dict) -> Shape:
    return Shape(
        batch=d["batch"], d_model=d["d_model"], n_heads=d["n_heads"], head_dim=d["head_dim"],
        max_pos=d["max_pos"], tail_slots=d.get("tail_slots", 0), rope_theta=d["rope_theta"],
        act=d["act"], kv=d["kv"],
    )


WORKLOADS = {
    # tiny single layer-step, fp32
    "tiny-f32": dict(name="tiny-f32", batch=1, d_model=256, n_heads=4, head_dim=64, max_pos=128,
            rope_theta=1e4, act="f32", kv="f32", block=16, gen_lo=64, fixed_lo=64, kind="plain"),
    # LLaDA-8B layer, batch 1
    "llada8b-b1": dict(name="llada8b-b1", batch=1, d_model=4096, n_heads=32, head_dim=128, max_pos=768,
            rope_theta=5e5, act="bf16", kv="bf16", block=32, gen_lo=512, fixed_lo=512, kind="plain"),
    # LLaDA-8B layer, batch 32, random block offsets, top-32 drift
    "llada8b-b32-drift": dict(name="llada8b-b32-drift", batch=32, d_model=4096, n_heads=32, head_dim=128, max_pos=1024,
            rope_theta=5e5, act="bf16", kv="bf16", block=32, gen_lo=512, fixed_lo=None, kind="drift",
            drift_k=32),
    # Flash-Verify layout, batch 16: 16 search tokens duplicated as draft + mask views
    "llada8b-b16-verify": dict(name="llada8b-b16-verify", batch=16, d_model=4096, n_heads=32, head_dim=128, max_pos=1024,
            tail_slots=16, rope_theta=5e5, act="bf16", kv="bf16", block=32, gen_lo=512, fixed_lo=None,
            kind="verify", search=16),
    # long-context full refresh into an FP8-e4m3 cache, batch 8
    "llada8b-b8-refresh-fp8": dict(name="llada8b-b8-refresh-fp8", batch=8, d_model=4096, n_heads=32, head_dim=128, max_pos=3072,
            rope_theta=5e5, act="bf16", kv="e4m3", block=32, gen_lo=2048, fixed_lo=None, kind="refresh"),
}


def make(name: str, seed: int = 0, **overrides) -> Workload:
    """Build the workload called ``name`` (a key of WORKLOADS), optionally shrunk by
    ``overrides``."""
    d = dict(WORKLOADS[name])
    d.update(overrides)
    if "d_model" in overrides and "n_heads" not in overrides:
        d["n_heads"] = d["d_model"] // d["head_dim"]
    shape = _shape(d)
    B, S, block = shape.batch, shape.max_pos, d["block"]
    gen_lo = min(d["gen_lo"], S - block)
    fixed = d["fixed_lo"]
    if fixed is not None:
        fixed = min(fixed, S - block)
    block_lo = _block_offsets(seed, B, gen_lo, S, block, fixed)
    w = weights(shape, seed)
    blk_pos = (block_lo[:, None] + np.arange(block, dtype=np.int32)[None, :]).astype(np.int32)
    others = _others(B, S, block_lo, block)
    kind = d["kind"]
    wl = Workload(name=d["name"], shape=shape, seed=seed, w=w, block_lo=block_lo, block_len=block,
                  pre_x=None, pre_pos=None, x=None, positions=None, view=None)

    if kind == "refresh":
        # the step itself rewrites every non-block position (K/V only) ...
        wl.kv_pos = others
        wl.kv_x = _rows(seed, _S_PREFILL, others, shape)
        # ... and the block rows (Q, K, V) attend over the refreshed cache
        wl.positions = blk_pos
        wl.x = _rows(seed, _S_BLOCK, blk_pos, shape)
        return wl

    wl.pre_pos = others
    wl.pre_x = _rows(seed, _S_PREFILL, others, shape)

    if kind in ("plain", "drift"):
        wl.positions = blk_pos
        wl.x = _rows(seed, _S_BLOCK, blk_pos, shape)
        if kind == "drift":
            k = d["drift_k"]
            rng = _rng(seed, _S_MASS)
            wl.mass = rng.dirichlet(np.full(S, 0.1), size=B).astype(np.float32)
            wl.drift_k = k
        return wl

    if kind == "verify":
        n_search = d["search"]
        if shape.tail_slots < n_search:
            raise ValueError("tail_slots must hold the draft view of every search token")
        rng = _rng(seed, _S_SEARCH)
        # rows 0..block-1: the ordinary step (search positions carry the mask view);
        # rows block..block+n_search-1: draft views of the search positions.
        x = np.empty((B, block + n_search, shape.D), np.float32)
        pos = np.empty((B, block + n_search), np.int32)
        view = np.empty((B, block + n_search), np.uint8)
        mask_emb = _store(_rng(seed, _S_MASKEMB).standard_normal(shape.D, dtype=np.float32), shape.act)
        base_rows = _rows(seed, _S_BLOCK, blk_pos, shape)
        draft_rows = _rows(seed, _S_DRAFT, blk_pos, shape)
        for b in range(B):
            search = np.sort(rng.choice(block, size=n_search, replace=False))
            is_search = np.zeros(block, bool)
            is_search[search] = True
            pos[b, :block] = blk_pos[b]
            x[b, :block] = base_rows[b]
            view[b, :block] = VIEW_BASE
            x[b, :block][is_search] = mask_emb
            view[b, :block][is_search] = VIEW_MASK
            pos[b, block:] = blk_pos[b, search]
            x[b, block:] = draft_rows[b, search]
            view[b, block:] = VIEW_DRAFT
        wl.x, wl.positions, wl.view = x, pos, view
        return wl
    raise ValueError(kind)


# ----------------------------------------------------------------------------------
# Multi-layer step with the depth-wise refresh.
# ----------------------------------------------------------------------------------

@dataclasses.dataclass
class ElasticWorkload:
    """One denoising step over ``n_layers`` layers.

    ``x_prev[l]``: hidden states every cache slot of layer l was built from (an earlier
    step); ``x_all[l]``: this step's hidden states of every position; ``w[l]``: weights;
    ``mass[l]``: previous-step attention mass; ``win_lo``/``beta``: the active window.
    """

    name: str
    shape: Shape
    seed: int
    n_layers: int
    w: list  # [3D][D] per layer
    x_prev: list  # [B][S][D] per layer
    x_all: list  # [B][S][D] per layer
    mass: np.ndarray  # float32 [L][B][S]
    win_lo: np.ndarray  # int32 [B]
    beta: int
    k: int
    gamma: float
    sigma: np.ndarray  # [L][B]


def make_elastic(sigma, seed: int = 0, batch: int = 4, d_model: int = 256, head_dim: int = 128,
                 max_pos: int = 384, beta: int = 32, gen_lo: int = 128, k: int = 8, gamma: float = 0.9,
                 rope_theta: float = 5e5, act: str = "bf16", kv: str = "bf16") -> ElasticWorkload:
    """``sigma`` [n_layers][batch]: drift scale of each layer and sequence."""
    sigma = np.asarray(sigma, np.float32)
    L = sigma.shape[0]
    if sigma.shape != (L, batch):
        raise ValueError("sigma must be [n_layers][batch]")
    shape = Shape(batch=batch, d_model=d_model, n_heads=d_model // head_dim, head_dim=head_dim, max_pos=max_pos,
                  tail_slots=0, rope_theta=rope_theta, act=act, kv=kv)
    S, D = max_pos, shape.D
    ws, xp, xa = [], [], []
    for l in range(L):
        w = _rng(seed, _S_WEIGHT, l).standard_normal((3 * D, D), dtype=np.float32) * np.float32(0.02)
        ws.append(_store(w, act))
        prev = np.empty((batch, S, D), np.float32)
        cur = np.empty((batch, S, D), np.float32)
        for b in range(batch):
            prev[b] = _rng(seed, _S_LAYER_PREV, l, b).standard_normal((S, D), dtype=np.float32)
            noise = _rng(seed, _S_LAYER_NOISE, l, b).standard_normal((S, D), dtype=np.float32)
            cur[b] = prev[b] + sigma[l, b] * noise
        xp.append(_store(prev, act))
        xa.append(_store(cur, act))
    mass = np.stack([_rng(seed, _S_MASS, l).dirichlet(np.full(S, 0.1), size=batch) for l in range(L)]).astype(np.float32)
    win_lo = _block_offsets(seed, batch, min(gen_lo, S - beta), S, beta, None)
    return ElasticWorkload(name=f"elastic-L{L}-b{batch}", shape=shape, seed=seed, n_layers=L, w=ws, x_prev=xp,
                           x_all=xa, mass=mass, win_lo=win_lo, beta=beta, k=k, gamma=gamma, sigma=sigma)
