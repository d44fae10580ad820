"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function the header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from denoising_step_attention_qkv_b300 import capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dllm_cache.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dllm_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    L = capi.lib()
    names = _declared()
    assert "dllm_cache_step" in names and "dllm_kv_drift" in names and "dllm_cache_alloc" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in the header but not exported"
    assert set(names) == set(capi.EXPORTS)


def _desc(**kw):
    d = dict(n_layers=1, batch=32, max_pos=1024, tail_slots=0, n_heads=32, head_dim=128,
             kv_dtype=capi.DLLM_BF16, rope_theta=5e5)
    d.update(kw)
    return capi.dllm_cache_desc(d["n_layers"], d["batch"], d["max_pos"], d["tail_slots"], d["n_heads"],
                                d["head_dim"], d["kv_dtype"], d["rope_theta"], None, 0)


def test_cache_bytes_matches_flat_layout():
    assert capi.dllm_cache_bytes(_desc()) == 32 * 1024 * 2 * 32 * 128 * 2
    assert capi.dllm_cache_bytes(_desc(kv_dtype=capi.DLLM_E4M3, batch=8, max_pos=3072)) == 8 * 3072 * (2 * 4096 + 2 * 32 * 4)
    assert capi.dllm_cache_bytes(_desc(kv_dtype=capi.DLLM_F32, n_heads=4, head_dim=64, batch=1, max_pos=128,
                                       tail_slots=16, n_layers=3)) == 3 * 144 * 2 * 256 * 4


@pytest.mark.parametrize("bad", [dict(n_layers=0), dict(batch=0), dict(max_pos=0), dict(tail_slots=-1),
                                 dict(kv_dtype=7), dict(rope_theta=0.0), dict(rope_theta=float("nan")),
                                 dict(head_dim=64), dict(kv_dtype=capi.DLLM_F32, head_dim=6)])
def test_bad_descriptors_rejected_on_host(bad):
    d = _desc(**bad)
    assert capi.dllm_cache_bytes(d) == 0
    h = ctypes.c_void_p()
    rc = capi.lib().dllm_cache_alloc(ctypes.byref(d), ctypes.byref(h))
    assert rc in (capi.DLLM_EINVAL, capi.DLLM_EUNSUPPORTED) and not h.value


def test_null_handles_rejected():
    L = capi.lib()
    assert L.dllm_cache_step(None, 0, None, None, None, None, 0, None, None, None, 0, None, None) == capi.DLLM_EINVAL
    assert L.dllm_cache_attend(None, 0, None, None, 1, None, None) == capi.DLLM_EINVAL
    assert L.dllm_kv_drift(None, 0, None, 1, None, 0.9, None, None, None) == capi.DLLM_EINVAL
    assert L.dllm_kv_topk(None, 1, 10, None, 0, 1, None, None) == capi.DLLM_EINVAL
    assert L.dllm_cache_status(None, None) == capi.DLLM_EINVAL
    assert L.dllm_cache_free(None) == capi.DLLM_OK
    assert capi.dllm_strerror(capi.DLLM_EUNSUPPORTED) == "unsupported configuration"


def test_merge_and_multilayer_arguments_rejected_on_host():
    L = capi.lib()
    a, b, o = 0x10000, 0x20000, 0x30000  # never dereferenced: every call below fails its checks
    assert L.dllm_attend_merge(None, b, 1, 1, 1, 128, o, None, None) == capi.DLLM_EINVAL
    assert L.dllm_attend_merge(a, b, 1, 1, 1, 128, None, None, None) == capi.DLLM_EINVAL  # no output
    assert L.dllm_attend_merge(a + 8, b, 1, 1, 1, 128, o, None, None) == capi.DLLM_EINVAL  # misaligned state
    assert L.dllm_attend_merge(a, b, 1, 1, 1, 128, o + 4, None, None) == capi.DLLM_EINVAL  # misaligned out
    assert L.dllm_attend_merge(a, b, 1 << 20, 1 << 10, 4, 128, o, None, None) == capi.DLLM_EINVAL  # rows overflow
    assert L.dllm_attend_merge(a, b, 1, 1, 1, 64, o, None, None) == capi.DLLM_EUNSUPPORTED
    assert L.dllm_attend_merge(a, b, 1, 0, 1, 128, o, None, None) == capi.DLLM_OK  # nothing to do
    assert L.dllm_elastic_workspace_bytes(None, 32, 8) == 0
    xs = (ctypes.c_void_p * 1)(a)
    assert L.dllm_elastic_step(None, 1, xs, xs, a, 32, a, 8, 0.9, o, a, a, None, a, 1 << 20, None) == capi.DLLM_EINVAL
    assert L.dllm_cache_attend_ragged(None, 0, a, 1, a, o, None) == capi.DLLM_EINVAL
    assert L.dllm_cache_attend_partial(None, 0, a, 1, o, 0, 1, a, None) == capi.DLLM_EINVAL
