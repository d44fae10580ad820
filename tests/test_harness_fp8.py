"""The e4m3 code check of the GPU tests (tests/gpu_harness.fp8_code_check), on the CPU.

It must accept what a correct e4m3 cache holds (each group quantised from fp32 values
with an fp32 scale, including codes that fp32 rounding moves across a rounding tie) and
reject plausible mistakes: a code two steps away, a flip away from any tie, a scale
that is not amax/448, codes rounded by truncation."""
import numpy as np
import pytest
import torch

import oracle as O
from tests import gpu_harness as G


def _groups(seed=0, n=64, hd=128):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, hd)) * rng.uniform(0.1, 5.0, (n, 1))


def _encode_fp32(exact):
    """What a correct kernel stores: fp32 values and scale, then RNE e4m3 codes."""
    x = exact.astype(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    t = torch.from_numpy(x / scale[:, None])
    codes = t.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, scale.astype(np.float64)


def test_accepts_a_correct_fp32_encoding():
    exact = _groups()
    codes, scale = _encode_fp32(exact)
    G.fp8_code_check(codes, scale, exact, "fp32 encoding")


def test_accepts_a_flip_at_a_rounding_tie():
    exact = _groups(1)
    codes, scale = _encode_fp32(exact)
    # put one value exactly on the midpoint of two codes (in units of its scale): either
    # neighbour is a correct code
    so = np.max(np.abs(exact), axis=-1) / 448.0
    exact[3, 5] = (1.0 + 1.0 / 16.0) * so[3]  # midway between 1.0 and 1.125
    codes[3, 5] = 1.125 if O.e4m3_quantize(np.array([1.0625]))[0] == 1.0 else 1.0
    assert G.fp8_code_check(codes, scale, exact, "tie") == 1


@pytest.mark.parametrize("mistake", ["two_steps", "off_tie", "scale_240", "truncate"])
def test_rejects_planted_mistakes(mistake):
    exact = _groups(2)
    codes, scale = _encode_fp32(exact)
    if mistake == "two_steps":
        i = np.unravel_index(np.argmax(np.abs(codes) * (np.abs(codes) < 200)), codes.shape)
        c = codes[i]
        codes[i] = O.e4m3_quantize(np.array([c * 1.3]))[0]  # skips a neighbour
    elif mistake == "off_tie":
        so = np.max(np.abs(exact), axis=-1) / 448.0
        exact[4, 7] = 1.02 * so[4]  # far from the tie between 1.0 and 1.125
        codes[4, 7] = 1.125
    elif mistake == "scale_240":
        amax = np.max(np.abs(exact), axis=-1)
        scale = amax / 240.0
    elif mistake == "truncate":
        so = np.max(np.abs(exact), axis=-1) / 448.0
        t = exact / so[:, None]
        _, ex = np.frexp(np.abs(t))
        quantum = np.ldexp(1.0, np.clip(ex - 1, -6, 8) - 3)
        codes = np.sign(t) * np.minimum(np.floor(np.abs(t) / quantum) * quantum, 448.0)
    with pytest.raises(AssertionError):
        G.fp8_code_check(codes, scale, exact, mistake)
