"""Attention in isolation: the GPU attention reads a cache and rotated queries that the
oracle wrote (rounded to the storage types), so the comparison sees the attention
kernel's own error, without the projection's.  Cases: a ragged last key tile with
split keys (32 queries), the 48-query kernel, and an e4m3 cache (codes and scales
taken from the oracle's quantised groups)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu

CASES = [
    ("bf16-ragged-split", dict(batch=2, d_model=512, head_dim=128, max_pos=300, block=32, gen_lo=128, kv="bf16")),
    ("bf16-48-queries", dict(batch=3, d_model=512, head_dim=128, max_pos=700, block=48, gen_lo=256, kv="bf16")),
    ("e4m3", dict(batch=2, d_model=512, head_dim=128, max_pos=300, block=32, gen_lo=128, kv="e4m3")),
]


def oracle_inputs(wl, model_fp8=True):
    """The oracle's cache after the step's writes (for an e4m3 workload its model of the
    encoding unless model_fp8 is False) and the step's rotated Q."""
    s = wl.shape
    oc = O.OracleCache(s.batch, s.max_pos, 0, s.n_heads, s.head_dim,
                       kv="e4m3" if (s.kv == "e4m3" and model_fp8) else "exact")
    O.write_rows(oc, wl.w, wl.pre_x, wl.pre_pos, s.rope_theta)
    O.write_rows(oc, wl.w, wl.x, wl.positions, s.rope_theta)
    q = np.stack([O.rope(O.project_qkv(wl.x[b], wl.w, s.n_heads)[0], wl.positions[b], s.rope_theta)
                  for b in range(s.batch)])
    return oc, q


def bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(torch.bfloat16)


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_attention_on_an_oracle_written_cache(name, kw):
    wl = W.make("llada8b-b1", **kw)
    s = wl.shape
    B, S, H, hd, n = s.batch, s.max_pos, s.n_heads, s.head_dim, wl.x.shape[1]
    oc, q = oracle_inputs(wl)
    assert oc.written[:, :S].all()
    qb = bf16_round(q)  # [B][n][H][hd]
    cache = G.make_cache(wl)
    kv = cache.kv(0)  # [B][slots][2][H][hd]
    if s.kv == "e4m3":
        groups = np.stack([oc.K[:, :S], oc.V[:, :S]], axis=2)  # dequantised values [B][S][2][H][hd]
        sc = np.max(np.abs(groups), axis=-1) / 448.0  # each group's scale (its max is 448 * scale)
        sc = np.where(sc > 0, sc, 1.0)
        c8 = torch.from_numpy(groups / sc[..., None]).to(torch.float8_e4m3fn)
        np.testing.assert_allclose(c8.double().numpy() * sc[..., None], groups, rtol=1e-12)  # codes recovered
        sc32 = sc.astype(np.float32)
        kv[:, :S].copy_(c8.view(torch.uint8).cuda())
        cache.scale(0)[:, :S].copy_(torch.from_numpy(sc32).cuda())
        deq = c8.double().numpy() * sc32[..., None]  # exactly what the kernel reads
        Kr, Vr = deq[:, :, 0], deq[:, :, 1]
    else:
        kb, vb = bf16_round(oc.K[:, :S]), bf16_round(oc.V[:, :S])
        kv[:, :S, 0].copy_(kb.cuda())
        kv[:, :S, 1].copy_(vb.cuda())
        Kr, Vr = kb.double().numpy(), vb.double().numpy()
    out = qb.reshape(B, n, H * hd).cuda().contiguous()
    capi.dllm_cache_attend(cache.handle, 0, G.idev(wl.positions), None, out)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    qr = qb.double().numpy()
    got = out.double().cpu().numpy()
    # exactly the values the kernel reads: its own error, at the bf16 bound for both caches
    ref = np.stack([O.attention(qr[b], Kr[b], Vr[b]).reshape(n, H * hd) for b in range(B)])
    G.assert_close(got, ref, G.TOL["bf16"], f"isolated attention ({name})")
    if s.kv == "e4m3":  # and against the unquantised oracle, at the FP8 bound
        oe, qe = oracle_inputs(wl, model_fp8=False)
        ref_e = np.stack([O.attention(qe[b], oe.K[b, :S], oe.V[b, :S]).reshape(n, H * hd) for b in range(B)])
        G.assert_close(got, ref_e, G.TOL["e4m3"], f"isolated attention vs the unquantised oracle ({name})")
