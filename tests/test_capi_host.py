"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function the header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from denoising_step_attention_qkv_b300 import capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dllm_cache.h")


def _declared():
    with open(HEADER) as f:
        text = f.read()
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
    assert L.dllm_gather_rows(None, None, 10, None, 1, None, None) == capi.DLLM_EINVAL
    assert L.dllm_kv_topk_gather(None, None, 10, None, 0, 1, None, None, None, None) == capi.DLLM_EINVAL
    assert L.dllm_selftest_fail_alloc(-1) == capi.DLLM_EINVAL
    assert L.dllm_selftest_fail_alloc(3) == capi.DLLM_OK and L.dllm_selftest_fail_alloc(0) == capi.DLLM_OK
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


def test_host_alloc_arguments():
    """Page-locked host blocks: a zero-byte request and a NULL free are no-ops, a NULL
    out-pointer is rejected, and without a usable device the call fails cleanly."""
    L = capi.lib()
    p = ctypes.c_void_p(1234)
    assert L.dllm_host_alloc(0, ctypes.byref(p)) == capi.DLLM_OK and p.value is None
    assert L.dllm_host_alloc(16, None) == capi.DLLM_EINVAL
    assert L.dllm_host_free(None) == capi.DLLM_OK
    assert capi.host_empty((0, 3), capi.torch.bfloat16).shape == (0, 3)
    import torch
    if not torch.cuda.is_available():
        p = ctypes.c_void_p()
        assert L.dllm_host_alloc(64, ctypes.byref(p)) == capi.DLLM_ECUDA and p.value is None


@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 63, 64, 65, 1000, 4096 + 7, (1 << 20) + 3])
@pytest.mark.parametrize("dst_off,src_off", [(0, 0), (1, 0), (0, 5), (7, 3), (15, 15)])
def test_host_stage_is_a_byte_copy(nbytes, dst_off, src_off):
    """The streaming-store copy writes exactly the bytes of src into dst, whatever the
    alignment of either side and the length of the unaligned head and tail, and
    touches nothing around the destination range."""
    import numpy as np
    rng = np.random.default_rng(nbytes * 31 + dst_off * 7 + src_off)
    src = np.frombuffer(rng.bytes(nbytes + 32), dtype=np.uint8).copy()
    dst = np.full(nbytes + 32, 0xA5, dtype=np.uint8)
    rc = capi.lib().dllm_host_stage(dst.ctypes.data + dst_off, src.ctypes.data + src_off, nbytes)
    assert rc == capi.DLLM_OK
    assert np.array_equal(dst[dst_off:dst_off + nbytes], src[src_off:src_off + nbytes])
    assert (dst[:dst_off] == 0xA5).all() and (dst[dst_off + nbytes:] == 0xA5).all()


def test_host_stage_arguments():
    import numpy as np
    import torch
    L = capi.lib()
    buf = np.zeros(256, dtype=np.uint8)
    p = buf.ctypes.data
    assert L.dllm_host_stage(None, None, 0) == capi.DLLM_OK
    assert L.dllm_host_stage(None, p, 16) == capi.DLLM_EINVAL
    assert L.dllm_host_stage(p, None, 16) == capi.DLLM_EINVAL
    assert L.dllm_host_stage(p, p + 64, 65) == capi.DLLM_EINVAL  # overlapping ranges
    assert L.dllm_host_stage(p + 64, p, 65) == capi.DLLM_EINVAL
    assert L.dllm_host_stage(p, p + 64, 64) == capi.DLLM_OK  # adjacent is fine
    a, b = torch.arange(100, dtype=torch.int32), torch.empty(100, dtype=torch.int32)
    assert torch.equal(capi.dllm_host_stage(b, a), a)
    with pytest.raises(ValueError):
        capi.dllm_host_stage(b[:50], a)


def test_host_empty_fails_loudly_without_a_device():
    """No silent fallback to ordinary host memory: without a usable device the binding
    raises with the library's status."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    with pytest.raises(capi.DllmError) as e:
        capi.host_empty((4, 8), torch.bfloat16)
    assert e.value.code == capi.DLLM_ECUDA


def test_binding_declares_every_signature():
    """Every exported function has ctypes argument and result types, so no pointer or
    size is ever passed through ctypes' default int conversion; and the argument count
    matches the header's declaration."""
    L = capi.lib()
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    for name in capi.EXPORTS:
        fn = getattr(L, name)
        assert fn.argtypes is not None and fn.restype is not None, name
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
        assert m, f"{name} not declared in the header"
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))
        for decl, ct in zip(params, fn.argtypes):
            if "*" in decl:  # any pointer: an address-sized ctypes type
                assert ct is ctypes.c_void_p or ct is ctypes.c_char_p or hasattr(ct, "_type_") and \
                    issubclass(ct, ctypes._Pointer), (name, decl, ct)
            else:
                ctype = decl.split()[-2] if len(decl.split()) > 1 else decl.split()[0]
                want = {"int": ctypes.c_int, "float": ctypes.c_float, "double": ctypes.c_double,
                        "size_t": ctypes.c_size_t}[ctype]
                assert ct is want, (name, decl, ct)
