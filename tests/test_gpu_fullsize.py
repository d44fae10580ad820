"""Full-size workloads through the C ABI, in the launch configuration the bench times,
against the fp64 oracle: the written-slot set of every sequence and the top-k indices
bit-exactly, then every head of three sequences per workload (cache K/V, attention
output, probes and drift cosines).

The attention runs one persistent CTA per SM (148 on a B300) over units numbered
(sequence, head) in order, in waves of one unit per CTA (where the last wave is
partial, it may be cut into pieces that all CTAs share), so the checked sequences are
the first one (first wave), one that straddles the last two waves and the last one
(every unit in the last wave)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import gpu_harness as G
from denoising_step_attention_qkv_b300 import capi

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _round_seqs(wl, n_queries):
    """First sequence, the sequence holding the first unit of the last round, last sequence."""
    s = wl.shape
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    units = s.batch * s.n_heads * -(-n_queries // 64)
    last_round = (units - 1) // sm * sm
    mid = last_round // (s.n_heads * -(-n_queries // 64))
    return sorted({0, min(mid, s.batch - 1), s.batch - 1})


def _topk(wl):
    idx = torch.empty((wl.shape.batch, wl.drift_k), dtype=torch.int32, device="cuda")
    capi.dllm_kv_topk(torch.from_numpy(wl.mass).cuda(), torch.from_numpy(wl.block_lo).cuda(), wl.block_len,
                      wl.drift_k, idx)
    return idx


def test_config3_batch32_drift_fullsize():
    wl = W.make("llada8b-b32-drift")
    idx = _topk(wl)
    idx_np = idx.cpu().numpy()
    np.testing.assert_array_equal(idx_np, O.kv_topk(wl.mass, wl.block_lo, wl.block_len, wl.drift_k))
    cache = G.make_cache(wl)
    out, probe = G.run_gpu(wl, cache, probe_idx=idx_np)
    seqs = _round_seqs(wl, wl.x.shape[1])
    assert len(seqs) == 3
    _, oracles = G.check_sequences(wl, cache, out, seqs, probe_gpu=probe, probe_idx=idx_np)
    # drift of the same sequences (the cosine spans all heads of a token)
    cos = torch.empty((wl.shape.batch, wl.drift_k, 2), dtype=torch.float32, device="cuda")
    refresh = torch.empty(wl.shape.batch, dtype=torch.int32, device="cuda")
    pk = torch.from_numpy(probe).to(torch.bfloat16).cuda()
    capi.dllm_kv_drift(cache.handle, 0, idx, pk, wl.gamma, cos, refresh)
    g_cos = cos.double().cpu().numpy()
    g_ref = refresh.cpu().numpy()
    o_coss = {}
    for b in seqs:
        _, oc, pr = oracles[b]
        o_coss[b] = O.kv_drift(oc, idx_np[b:b + 1], pr[None])[0]
        G.assert_close(g_cos[b], o_coss[b], G.TOL["bf16"], f"drift cos b={b}")
        assert g_ref[b] == int(g_cos[b].min() < np.float32(wl.gamma))
    assert set(np.unique(g_ref)) <= {0, 1}
    # the drift test fused into the projection (the bench's step): same tracked rows, the
    # same cache afterwards, cosines against the oracle and flags from its own cosines
    fcos = torch.full_like(cos, 7.0)
    fref = torch.full_like(refresh, 7)
    w = G.tdev(wl.w, "bf16")
    out2 = torch.empty((wl.shape.batch, wl.x.shape[1], wl.shape.D), dtype=torch.bfloat16, device="cuda")
    capi.dllm_cache_step_drift(cache.handle, 0, G.tdev(wl.x, "bf16"), w, G.idev(wl.positions), None, out2,
                               G.tdev(wl.probe_rows(idx_np), "bf16"), idx, wl.gamma, fcos, fref)
    torch.cuda.synchronize()
    assert cache.status() == (capi.DLLM_OK, 0)
    f_cos = fcos.double().cpu().numpy()
    for b in seqs:
        G.assert_close(f_cos[b], o_coss[b], G.TOL["bf16"], f"fused drift cos b={b}")
    np.testing.assert_array_equal(fref.cpu().numpy(), (fcos.cpu().numpy().reshape(wl.shape.batch, -1).min(1)
                                                        < np.float32(wl.gamma)).astype(np.int32))
    np.testing.assert_array_equal(out2.double().cpu().numpy(), out)  # same step, same output


def test_config4_verify_fullsize():
    wl = W.make("llada8b-b16-verify")
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    seqs = _round_seqs(wl, wl.x.shape[1])
    assert len(seqs) == 3
    G.check_sequences(wl, cache, out, seqs)


def test_config5_refresh_fp8_fullsize():
    # The e4m3 encoding alone (the oracle's own model of it against the unquantised
    # oracle, no GPU) moves this workload's output by 4.3-10.2% of a sequence's
    # max|out| and by 4.9% of the whole output's, so the output is checked as the bound
    # states it: over the whole output tensor, every sequence computed by the oracle.
    wl = W.make("llada8b-b8-refresh-fp8")
    cache = G.make_cache(wl)
    out, _ = G.run_gpu(wl, cache)
    seqs = _round_seqs(wl, wl.x.shape[1])
    assert len(seqs) == 3
    G.check_sequences(wl, cache, out, seqs, whole_output=True)
