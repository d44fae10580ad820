"""The Python wrappers of the binding, on the CPU: each one is called against a stand-in
for the library that records what it receives, and must pass exactly the arguments the
header declares for its C function (count, and the sizes taken from the tensors), and
turn a non-zero status into DllmError."""
import os
import re

import pytest
import torch

from denoising_step_attention_qkv_b300 import capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dllm_cache.h")


def _param_counts():
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for name in capi.EXPORTS:
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
        out[name] = len([p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"])
    return out


class _FakeLib:
    def __init__(self, status=0):
        self.calls = []
        self.status = status

    def __getattr__(self, name):
        if not name.startswith("dllm_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append((name, args))
            if name.endswith("_bytes"):
                return 4096
            if name == "dllm_strerror":
                return b"fake"
            return self.status
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = _FakeLib()
    monkeypatch.setattr(capi, "_lib", lib)
    return lib


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _calls(h):
    """One call of every launching wrapper, with small CPU tensors (B=2, n=3, D=8, k=4)."""
    B, n, D, k = 2, 3, 8, 4
    x, w, out = _t(B, n, D), _t(3 * D, D), _t(B, n, D)
    pos = _t(B, n, dtype=torch.int32)
    view = _t(B, n, dtype=torch.uint8)
    kvx, idx = _t(B, k, D), _t(B, k, dtype=torch.int32)
    probe = _t(B, k, 2, D)
    cos, refresh = _t(B, k, 2, dtype=torch.float32), _t(B, dtype=torch.int32)
    state = _t(B, n, 2, 130, dtype=torch.float32)
    mass = _t(B, 16, dtype=torch.float32)
    return [
        ("dllm_cache_step", lambda: capi.dllm_cache_step(h, 0, x, w, pos, view, out, kvx, idx, probe, stream=0)),
        ("dllm_cache_project", lambda: capi.dllm_cache_project(h, 0, x, w, pos, view, out, kvx, idx, probe, stream=0)),
        ("dllm_cache_project_drift",
         lambda: capi.dllm_cache_project_drift(h, 0, x, w, pos, view, out, kvx, idx, 0.9, cos, refresh, stream=0)),
        ("dllm_cache_step_drift",
         lambda: capi.dllm_cache_step_drift(h, 0, x, w, pos, view, out, kvx, idx, 0.9, cos, refresh, stream=0)),
        ("dllm_cache_attend", lambda: capi.dllm_cache_attend(h, 0, pos, view, out, stream=0)),
        ("dllm_cache_attend_noalloc", lambda: capi.dllm_cache_attend_noalloc(h, 0, pos, view, out, stream=0)),
        ("dllm_attention_mass", lambda: capi.dllm_attention_mass(h, 0, pos, view, out, mass, stream=0)),
        ("dllm_cache_attend_ragged", lambda: capi.dllm_cache_attend_ragged(h, 0, pos, refresh, out, stream=0)),
        ("dllm_cache_attend_partial", lambda: capi.dllm_cache_attend_partial(h, 0, pos, out, 0, 8, state, stream=0)),
        ("dllm_cache_attend_with_state",
         lambda: capi.dllm_cache_attend_with_state(h, 0, pos, out, 4, 8, state, x, stream=0)),
        ("dllm_attend_merge", lambda: capi.dllm_attend_merge(state, state, out=out, stream=0)),
        ("dllm_cache_step_unfused",
         lambda: capi.dllm_cache_step_unfused(h, 0, x, w, pos, view, out, _t(64, dtype=torch.uint8), kvx, idx, probe,
                                              stream=0)),
        ("dllm_kv_topk", lambda: capi.dllm_kv_topk(mass, refresh, 3, k, idx, stream=0)),
        ("dllm_gather_rows", lambda: capi.dllm_gather_rows(h, _t(B, 16, D), idx, kvx, stream=0)),
        ("dllm_kv_topk_gather",
         lambda: capi.dllm_kv_topk_gather(h, mass, refresh, 3, k, idx, _t(B, 16, D), kvx, stream=0)),
        ("dllm_kv_drift", lambda: capi.dllm_kv_drift(h, 0, idx, probe, 0.9, cos, refresh, stream=0)),
        ("dllm_elastic_step",
         lambda: capi.dllm_elastic_step(h, [_t(B, 16, D)] * 2, [w] * 2, refresh, 3, mass, k, 0.9, out, cos, refresh,
                                        _t(64, dtype=torch.uint8), stream=0)),
        ("dllm_selftest_wait_timeout", lambda: capi.dllm_selftest_wait_timeout(h, stream=0)),
        ("dllm_selftest_fail_alloc", lambda: capi.dllm_selftest_fail_alloc(2)),
    ]


def test_every_wrapper_passes_the_declared_arguments(fake):
    counts = _param_counts()
    seen = set()
    for name, call in _calls(h=0x1234):
        fake.calls.clear()
        call()
        assert [c[0] for c in fake.calls] == [name], (name, fake.calls)
        args = fake.calls[0][1]
        assert len(args) == counts[name], (name, len(args), counts[name])
        seen.add(name)
    launching = {n for n in capi.EXPORTS if not n.startswith(("dllm_cache_bytes", "dllm_cache_alloc", "dllm_cache_free",
                                                              "dllm_cache_get_layout", "dllm_strerror", "dllm_host_",
                                                              "dllm_cache_status", "dllm_unfused_workspace",
                                                              "dllm_elastic_workspace"))}
    assert launching <= seen, launching - seen


def test_sizes_come_from_the_tensors(fake):
    B, n, D = 2, 3, 8
    x = _t(B, n, D)
    capi.dllm_cache_project_drift(7, 1, x, _t(3 * D, D), _t(B, n, dtype=torch.int32), None, x, _t(B, 5, D),
                                  _t(B, 5, dtype=torch.int32), 0.75, _t(B, 5, 2, dtype=torch.float32), None, stream=0)
    args = fake.calls[-1][1]
    # handle, layer, x, w, positions, view, n_tok, out, kv_x, idx, k, gamma, cos, refresh, stream
    assert args[0] == 7 and args[1] == 1 and args[6] == n and args[10] == 5 and args[11] == pytest.approx(0.75)
    assert args[5] is None and args[13] is None and args[14] == 0
    st = _t(B, n, 2, 130, dtype=torch.float32)
    capi.dllm_cache_attend_with_state(7, 0, _t(B, n, dtype=torch.int32), x, 100, 300, st, x, stream=0)
    args = fake.calls[-1][1]
    # handle, layer, positions, n_tok, q, slot_lo, slot_hi, state, out, stream
    assert args[3] == n and args[5] == 100 and args[6] == 300 and args[7] == st.data_ptr()


def test_a_failing_status_raises(monkeypatch):
    monkeypatch.setattr(capi, "_lib", _FakeLib(status=capi.DLLM_EINVAL))
    with pytest.raises(capi.DllmError) as e:
        capi.dllm_gather_rows(1, _t(2, 4, 8), _t(2, 2, dtype=torch.int32), _t(2, 2, 8), stream=0)
    assert e.value.code == capi.DLLM_EINVAL
