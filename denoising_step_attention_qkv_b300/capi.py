"""Thin ctypes binding of ``include/dllm_cache.h`` (argument marshalling only).

Every function keeps the C name and forwards device pointers, sizes and the current
CUDA stream to ``libdllmcache.so``; all computation happens in the library's kernels.
There is no fallback: if the library is missing or a call fails, an exception is
raised.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_size_t, c_void_p
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdllmcache.so")

DLLM_OK, DLLM_EINVAL, DLLM_EOOM, DLLM_ECUDA, DLLM_EDEVICE, DLLM_EUNSUPPORTED = range(6)
DLLM_F32, DLLM_BF16, DLLM_E4M3 = 0, 1, 2
DLLM_VIEW_BASE, DLLM_VIEW_DRAFT, DLLM_VIEW_MASK = 0, 1, 2
DEV_BAD_POSITION, DEV_BAD_VIEW, DEV_TAIL_FULL, DEV_TIMEOUT, DEV_BAD_INDEX = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTS = ("dllm_cache_bytes", "dllm_cache_alloc", "dllm_cache_free", "dllm_cache_get_layout", "dllm_cache_step",
           "dllm_cache_project", "dllm_cache_project_drift", "dllm_cache_step_drift", "dllm_cache_attend", "dllm_cache_attend_noalloc", "dllm_unfused_workspace_bytes",
           "dllm_cache_step_unfused", "dllm_attention_mass", "dllm_cache_attend_ragged", "dllm_cache_attend_partial",
           "dllm_cache_attend_with_state",
           "dllm_attend_merge", "dllm_kv_topk", "dllm_gather_rows", "dllm_kv_topk_gather", "dllm_kv_drift", "dllm_elastic_workspace_bytes",
           "dllm_elastic_step",
           "dllm_selftest_wait_timeout", "dllm_selftest_fail_alloc",
           "dllm_cache_status", "dllm_strerror", "dllm_host_alloc", "dllm_host_free",
           "dllm_host_stage")


class dllm_cache_desc(ctypes.Structure):
    _fields_ = [("n_layers", c_int), ("batch", c_int), ("max_pos", c_int), ("tail_slots", c_int),
                ("n_heads", c_int), ("head_dim", c_int), ("kv_dtype", c_int), ("rope_theta", c_double),
                ("external_buf", c_void_p), ("external_bytes", c_size_t)]


class dllm_cache_layout(ctypes.Structure):
    _fields_ = [("kv", c_void_p), ("scale", c_void_p), ("kv_bytes", c_size_t), ("scale_bytes", c_size_t),
                ("layer_elems", c_size_t), ("slots", c_int), ("elem_bytes", c_int)]


class DllmError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({dllm_strerror(code)})")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with denoising_step_attention_qkv_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.dllm_cache_bytes.argtypes = [POINTER(dllm_cache_desc)]
        L.dllm_cache_bytes.restype = c_size_t
        L.dllm_cache_alloc.argtypes = [POINTER(dllm_cache_desc), POINTER(c_void_p)]
        L.dllm_cache_free.argtypes = [c_void_p]
        L.dllm_cache_get_layout.argtypes = [c_void_p, POINTER(dllm_cache_layout)]
        L.dllm_cache_step.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                      c_void_p, c_void_p, c_int, c_void_p, c_void_p]
        L.dllm_cache_project.argtypes = L.dllm_cache_step.argtypes
        L.dllm_cache_project_drift.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                               c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p, c_void_p,
                                               c_void_p]
        L.dllm_cache_step_drift.argtypes = L.dllm_cache_project_drift.argtypes
        L.dllm_cache_attend.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p]
        L.dllm_cache_attend_noalloc.argtypes = L.dllm_cache_attend.argtypes
        L.dllm_unfused_workspace_bytes.argtypes = [c_void_p, c_int, c_int]
        L.dllm_unfused_workspace_bytes.restype = c_size_t
        L.dllm_cache_step_unfused.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                              c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]
        L.dllm_kv_topk.argtypes = [c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_void_p, c_void_p]
        L.dllm_gather_rows.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p]
        L.dllm_kv_topk_gather.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                          c_void_p, c_void_p]
        L.dllm_kv_drift.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_float, c_void_p, c_void_p, c_void_p]
        L.dllm_selftest_wait_timeout.argtypes = [c_void_p, c_void_p]
        L.dllm_selftest_fail_alloc.argtypes = [c_int]
        L.dllm_attention_mass.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]
        L.dllm_cache_attend_ragged.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p]
        L.dllm_cache_attend_partial.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_void_p,
                                                c_void_p]
        L.dllm_cache_attend_with_state.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_int,
                                                   c_void_p, c_void_p, c_void_p]
        L.dllm_attend_merge.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]
        L.dllm_elastic_workspace_bytes.argtypes = [c_void_p, c_int, c_int]
        L.dllm_elastic_workspace_bytes.restype = c_size_t
        L.dllm_elastic_step.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int, c_float,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
        L.dllm_cache_status.argtypes = [c_void_p, POINTER(c_int)]
        L.dllm_strerror.argtypes = [c_int]
        L.dllm_strerror.restype = ctypes.c_char_p
        L.dllm_host_alloc.argtypes = [c_size_t, POINTER(c_void_p)]
        L.dllm_host_free.argtypes = [c_void_p]
        L.dllm_host_stage.argtypes = [c_void_p, c_void_p, c_size_t]
        for name in EXPORTS:
            if name not in ("dllm_cache_bytes", "dllm_strerror", "dllm_unfused_workspace_bytes",
                            "dllm_elastic_workspace_bytes"):
                getattr(L, name).restype = c_int
        _lib = L
    return _lib


def _check(fn: str, code: int):
    if code != DLLM_OK:
        raise DllmError(fn, code)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dllm_strerror(code: int) -> str:
    return lib().dllm_strerror(int(code)).decode()


def dllm_cache_bytes(desc: dllm_cache_desc) -> int:
    return int(lib().dllm_cache_bytes(ctypes.byref(desc)))


def dllm_cache_alloc(desc: dllm_cache_desc) -> c_void_p:
    h = c_void_p()
    _check("dllm_cache_alloc", lib().dllm_cache_alloc(ctypes.byref(desc), ctypes.byref(h)))
    return h


def dllm_cache_free(handle) -> None:
    _check("dllm_cache_free", lib().dllm_cache_free(handle))


def dllm_cache_get_layout(handle) -> dllm_cache_layout:
    out = dllm_cache_layout()
    _check("dllm_cache_get_layout", lib().dllm_cache_get_layout(handle, ctypes.byref(out)))
    return out


def dllm_cache_step(handle, layer: int, x: Optional[torch.Tensor], w_qkv: torch.Tensor,
                    positions: Optional[torch.Tensor], view: Optional[torch.Tensor], out: Optional[torch.Tensor],
                    kv_x: Optional[torch.Tensor] = None, kv_positions: Optional[torch.Tensor] = None,
                    probe_kv: Optional[torch.Tensor] = None, stream=None) -> None:
    n_tok = 0 if positions is None else int(positions.shape[-1])
    n_kv = 0 if kv_positions is None else int(kv_positions.shape[-1])
    _check("dllm_cache_step", lib().dllm_cache_step(
        handle, int(layer), _ptr(x), _ptr(w_qkv), _ptr(positions), _ptr(view), n_tok, _ptr(out),
        _ptr(kv_x), _ptr(kv_positions), n_kv, _ptr(probe_kv), _stream(stream)))


def dllm_cache_project(handle, layer: int, x: Optional[torch.Tensor], w_qkv: torch.Tensor,
                       positions: Optional[torch.Tensor], view: Optional[torch.Tensor], out: Optional[torch.Tensor],
                       kv_x: Optional[torch.Tensor] = None, kv_positions: Optional[torch.Tensor] = None,
                       probe_kv: Optional[torch.Tensor] = None, stream=None) -> None:
    n_tok = 0 if positions is None else int(positions.shape[-1])
    n_kv = 0 if kv_positions is None else int(kv_positions.shape[-1])
    _check("dllm_cache_project", lib().dllm_cache_project(
        handle, int(layer), _ptr(x), _ptr(w_qkv), _ptr(positions), _ptr(view), n_tok, _ptr(out),
        _ptr(kv_x), _ptr(kv_positions), n_kv, _ptr(probe_kv), _stream(stream)))


def _drift_call(fn: str, handle, layer, x, w_qkv, positions, view, out, kv_x, idx, gamma, cos, refresh, stream):
    n_tok = 0 if positions is None else int(positions.shape[-1])
    _check(fn, getattr(lib(), fn)(handle, int(layer), _ptr(x), _ptr(w_qkv), _ptr(positions), _ptr(view), n_tok,
                                  _ptr(out), _ptr(kv_x), _ptr(idx), int(idx.shape[-1]), float(gamma), _ptr(cos),
                                  _ptr(refresh), _stream(stream)))


def dllm_cache_project_drift(handle, layer: int, x: Optional[torch.Tensor], w_qkv: torch.Tensor,
                             positions: Optional[torch.Tensor], view: Optional[torch.Tensor],
                             out: Optional[torch.Tensor], kv_x: torch.Tensor, idx: torch.Tensor, gamma: float,
                             cos: torch.Tensor, refresh: Optional[torch.Tensor] = None, stream=None) -> None:
    """Projection with the drift test of the tracked rows fused (no probe buffer)."""
    _drift_call("dllm_cache_project_drift", handle, layer, x, w_qkv, positions, view, out, kv_x, idx, gamma, cos,
                refresh, stream)


def dllm_cache_step_drift(handle, layer: int, x: Optional[torch.Tensor], w_qkv: torch.Tensor,
                          positions: Optional[torch.Tensor], view: Optional[torch.Tensor],
                          out: Optional[torch.Tensor], kv_x: torch.Tensor, idx: torch.Tensor, gamma: float,
                          cos: torch.Tensor, refresh: Optional[torch.Tensor] = None, stream=None) -> None:
    """dllm_cache_project_drift then dllm_cache_attend."""
    _drift_call("dllm_cache_step_drift", handle, layer, x, w_qkv, positions, view, out, kv_x, idx, gamma, cos,
                refresh, stream)


def dllm_cache_attend(handle, layer: int, positions: torch.Tensor, view: Optional[torch.Tensor], out: torch.Tensor,
                      stream=None) -> None:
    _check("dllm_cache_attend", lib().dllm_cache_attend(handle, int(layer), _ptr(positions), _ptr(view),
                                                        int(positions.shape[-1]), _ptr(out), _stream(stream)))


def dllm_cache_attend_noalloc(handle, layer: int, positions: torch.Tensor, view: Optional[torch.Tensor],
                              out: torch.Tensor, stream=None) -> None:
    """dllm_cache_attend with its scratch in a fixed static device array (no allocation)."""
    _check("dllm_cache_attend_noalloc", lib().dllm_cache_attend_noalloc(
        handle, int(layer), _ptr(positions), _ptr(view), int(positions.shape[-1]), _ptr(out), _stream(stream)))


def dllm_attention_mass(handle, layer: int, positions: torch.Tensor, view: Optional[torch.Tensor], q: torch.Tensor,
                        mass: torch.Tensor, stream=None) -> None:
    """Per-position attention mass of the step (needs the rotated Q from dllm_cache_project)."""
    _check("dllm_attention_mass", lib().dllm_attention_mass(handle, int(layer), _ptr(positions), _ptr(view),
                                                            int(positions.shape[-1]), _ptr(q), _ptr(mass),
                                                            _stream(stream)))


def dllm_cache_attend_ragged(handle, layer: int, positions: torch.Tensor, key_len: torch.Tensor, out: torch.Tensor,
                             stream=None) -> None:
    """Attention of sequence b over its first key_len[b] slots only."""
    _check("dllm_cache_attend_ragged", lib().dllm_cache_attend_ragged(
        handle, int(layer), _ptr(positions), int(positions.shape[-1]), _ptr(key_len), _ptr(out), _stream(stream)))


def dllm_cache_attend_partial(handle, layer: int, positions: torch.Tensor, q: torch.Tensor, slot_lo: int,
                              slot_hi: int, state: torch.Tensor, stream=None) -> None:
    """Partial softmax state (O, m, l) of the query rows over slots [slot_lo, slot_hi)."""
    _check("dllm_cache_attend_partial", lib().dllm_cache_attend_partial(
        handle, int(layer), _ptr(positions), int(positions.shape[-1]), _ptr(q), int(slot_lo), int(slot_hi),
        _ptr(state), _stream(stream)))


def dllm_cache_attend_with_state(handle, layer: int, positions: torch.Tensor, q: torch.Tensor, slot_lo: int,
                                 slot_hi: int, state: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Attention over [slot_lo, slot_hi) merged with a cached state of the other keys."""
    _check("dllm_cache_attend_with_state", lib().dllm_cache_attend_with_state(
        handle, int(layer), _ptr(positions), int(positions.shape[-1]), _ptr(q), int(slot_lo), int(slot_hi),
        _ptr(state), _ptr(out), _stream(stream)))


def dllm_attend_merge(state_a: torch.Tensor, state_b: torch.Tensor, out: Optional[torch.Tensor] = None,
                      state_out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Combine two partial states ([B][n][H][hd+2]) into an output and/or a state."""
    B, n, H, w = state_a.shape
    _check("dllm_attend_merge", lib().dllm_attend_merge(_ptr(state_a), _ptr(state_b), int(B), int(n), int(H),
                                                        int(w - 2), _ptr(out), _ptr(state_out), _stream(stream)))


def dllm_unfused_workspace_bytes(handle, n_tok: int, n_kv: int) -> int:
    return int(lib().dllm_unfused_workspace_bytes(handle, int(n_tok), int(n_kv)))


def dllm_cache_step_unfused(handle, layer: int, x: Optional[torch.Tensor], w_qkv: torch.Tensor,
                            positions: Optional[torch.Tensor], view: Optional[torch.Tensor], out: Optional[torch.Tensor],
                            workspace: torch.Tensor, kv_x: Optional[torch.Tensor] = None,
                            kv_positions: Optional[torch.Tensor] = None, probe_kv: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """The four-kernel pipeline (projection, rotary, cache write, attention) for comparison."""
    n_tok = 0 if positions is None else int(positions.shape[-1])
    n_kv = 0 if kv_positions is None else int(kv_positions.shape[-1])
    _check("dllm_cache_step_unfused", lib().dllm_cache_step_unfused(
        handle, int(layer), _ptr(x), _ptr(w_qkv), _ptr(positions), _ptr(view), n_tok, _ptr(out),
        _ptr(kv_x), _ptr(kv_positions), n_kv, _ptr(probe_kv), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def dllm_kv_topk(mass: torch.Tensor, block_lo: torch.Tensor, block_len: int, k: int, idx: torch.Tensor,
                 stream=None) -> None:
    B, n_pos = mass.shape
    _check("dllm_kv_topk", lib().dllm_kv_topk(_ptr(mass), int(B), int(n_pos), _ptr(block_lo), int(block_len),
                                              int(k), _ptr(idx), _stream(stream)))


def dllm_gather_rows(handle, x_all: torch.Tensor, idx: torch.Tensor, x_rows: torch.Tensor, stream=None) -> None:
    """x_rows[b][j] = x_all[b][idx[b][j]] (the tracked tokens' hidden states)."""
    _check("dllm_gather_rows", lib().dllm_gather_rows(handle, _ptr(x_all), int(x_all.shape[1]), _ptr(idx),
                                                      int(idx.shape[-1]), _ptr(x_rows), _stream(stream)))


def dllm_kv_topk_gather(handle, mass: torch.Tensor, block_lo: torch.Tensor, block_len: int, k: int,
                        idx: torch.Tensor, x_all: torch.Tensor, x_rows: torch.Tensor, stream=None) -> None:
    """dllm_kv_topk then dllm_gather_rows of the selected positions (one launch for k <= 32)."""
    n_pos = int(mass.shape[1])
    _check("dllm_kv_topk_gather", lib().dllm_kv_topk_gather(handle, _ptr(mass), n_pos, _ptr(block_lo), int(block_len),
                                                            int(k), _ptr(idx), _ptr(x_all), _ptr(x_rows),
                                                            _stream(stream)))


def dllm_kv_drift(handle, layer: int, idx: torch.Tensor, probe_kv: torch.Tensor, gamma: float, cos: torch.Tensor,
                  refresh: Optional[torch.Tensor] = None, stream=None) -> None:
    k = int(idx.shape[-1])
    _check("dllm_kv_drift", lib().dllm_kv_drift(handle, int(layer), _ptr(idx), k, _ptr(probe_kv), float(gamma),
                                                _ptr(cos), _ptr(refresh), _stream(stream)))


def dllm_elastic_workspace_bytes(handle, beta: int, k: int) -> int:
    return int(lib().dllm_elastic_workspace_bytes(handle, int(beta), int(k)))


def dllm_elastic_step(handle, x_all: Sequence[torch.Tensor], w_qkv: Sequence[torch.Tensor], win_lo: torch.Tensor,
                      beta: int, mass: torch.Tensor, k: int, gamma: float, out: torch.Tensor, cos: torch.Tensor,
                      flags: torch.Tensor, workspace: torch.Tensor, mass_out: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """One denoising step over len(x_all) layers with the depth-wise drift refresh."""
    n = len(x_all)
    if len(w_qkv) != n:
        raise ValueError("x_all and w_qkv must have one entry per layer")
    xs = (c_void_p * n)(*[_ptr(t) for t in x_all])
    ws = (c_void_p * n)(*[_ptr(t) for t in w_qkv])
    _check("dllm_elastic_step", lib().dllm_elastic_step(
        handle, n, xs, ws, _ptr(win_lo), int(beta), _ptr(mass), int(k), float(gamma), _ptr(out), _ptr(cos),
        _ptr(flags), _ptr(mass_out), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream(stream)))


def dllm_selftest_fail_alloc(nth: int) -> None:
    """Make the nth device allocation of the library from now on fail (0 cancels)."""
    _check("dllm_selftest_fail_alloc", lib().dllm_selftest_fail_alloc(int(nth)))


def dllm_selftest_wait_timeout(handle, stream=None) -> None:
    """Launch the bounded-wait self-test (sets DEV_TIMEOUT in the status word after ~1 s)."""
    _check("dllm_selftest_wait_timeout", lib().dllm_selftest_wait_timeout(handle, _stream(stream)))


def dllm_cache_status(handle):
    """Returns (status, device_bits); clears the device status word."""
    bits = c_int(0)
    rc = lib().dllm_cache_status(handle, ctypes.byref(bits))
    if rc not in (DLLM_OK, DLLM_EDEVICE):
        raise DllmError("dllm_cache_status", rc)
    return rc, bits.value


def dllm_host_alloc(nbytes: int) -> Optional[int]:
    """Page-locked host block of nbytes bytes; returns its address (None for 0 bytes)."""
    p = c_void_p()
    _check("dllm_host_alloc", lib().dllm_host_alloc(int(nbytes), ctypes.byref(p)))
    return p.value


def dllm_host_free(ptr: Optional[int]) -> None:
    _check("dllm_host_free", lib().dllm_host_free(ptr))


def dllm_host_stage(dst: torch.Tensor, src: torch.Tensor) -> torch.Tensor:
    """Byte copy of the contiguous CPU tensor src into dst (same byte size) with
    streaming stores; returns dst."""
    if dst.device.type != "cpu" or src.device.type != "cpu":
        raise ValueError("dllm_host_stage copies host tensors")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dllm_host_stage: dst and src differ in size")
    _check("dllm_host_stage", lib().dllm_host_stage(_ptr(dst) if nbytes else None, _ptr(src) if nbytes else None,
                                                   nbytes))
    return dst


class _HostBlock:
    """Owns one dllm_host_alloc block; freed when the last tensor viewing it is gone."""

    def __init__(self, nbytes: int):
        self.ptr = None
        self.ptr = dllm_host_alloc(nbytes)

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.dllm_host_free(self.ptr)
            self.ptr = None


def host_empty(shape, dtype: torch.dtype) -> torch.Tensor:
    """Uninitialised CPU tensor over a dllm_host_alloc block (page-locked, read and
    written by the GPU's copy engines at the link rate).  The block is released when
    the tensor and every view of it are gone."""
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list, torch.Size)) else (shape,)))
    numel = 1
    for s in shape:
        numel *= s
    nbytes = numel * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype)
    blk = _HostBlock(nbytes)
    arr = (ctypes.c_uint8 * nbytes).from_address(blk.ptr)
    arr._owner = blk  # the tensor's storage keeps arr, and arr the block, alive
    return torch.frombuffer(arr, dtype=torch.uint8).view(dtype).reshape(shape)


# ------------------------------------------------------------------------------------
# Convenience owner: a cache whose flat buffer is a torch allocation (so tests and
# callers can view it), released with the object.
# ------------------------------------------------------------------------------------

_DTYPES = {DLLM_F32: torch.float32, DLLM_BF16: torch.bfloat16, DLLM_E4M3: torch.uint8}


class Cache:
    def __init__(self, n_layers: int, batch: int, max_pos: int, n_heads: int, head_dim: int, kv_dtype: int,
                 rope_theta: float, tail_slots: int = 0, device: str = "cuda"):
        if not torch.cuda.is_available():
            raise RuntimeError("a CUDA device is required")
        self.desc = dllm_cache_desc(n_layers, batch, max_pos, tail_slots, n_heads, head_dim, kv_dtype,
                                    float(rope_theta), None, 0)
        nbytes = dllm_cache_bytes(self.desc)
        if nbytes == 0:
            raise ValueError("invalid cache shape")
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.desc.external_buf = self.buf.data_ptr()
        self.desc.external_bytes = nbytes
        self.handle = dllm_cache_alloc(self.desc)
        self.layout = dllm_cache_get_layout(self.handle)
        self.slots = max_pos + tail_slots
        self.shape = (n_layers, batch, self.slots, 2, n_heads, head_dim)

    def kv(self, layer: Optional[int] = None) -> torch.Tensor:
        t = self.buf[: self.layout.kv_bytes].view(_DTYPES[self.desc.kv_dtype]).view(self.shape)
        return t if layer is None else t[layer]

    def scale(self, layer: Optional[int] = None) -> Optional[torch.Tensor]:
        if self.desc.kv_dtype != DLLM_E4M3:
            return None
        t = self.buf[self.layout.kv_bytes: self.layout.kv_bytes + self.layout.scale_bytes].view(torch.float32)
        t = t.view(self.shape[:-1])
        return t if layer is None else t[layer]

    def status(self):
        return dllm_cache_status(self.handle)

    def close(self):
        if getattr(self, "handle", None) is not None:
            dllm_cache_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
