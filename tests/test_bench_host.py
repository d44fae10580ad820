"""Host-side logic of bench.py that decides the numbers it reports, checked on CPU:
the algorithmic work behind the roofline fractions, the DRAM traffic read back from
the committed ncu record (withdrawn once a kernel's sources change), and the peaks."""
import json
import os
import shutil

import pytest

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_work_of_the_batch32_step():
    # projection: 1024 block rows x 3D features + 1024 probe rows x 2D features, 2*D FLOP
    # each; attention: K and V of every slot once per (sequence, head) + Q in and O out
    wl = bench._with_drift_inputs(W.make("llada8b-b32-drift"))
    a = bench.algorithmic(wl)
    D, B, n, k, S, H, hd = 4096, 32, 32, 32, 1024, 32, 128
    assert a["proj_flops"] == 2 * D * (B * n * 3 * D + B * k * 2 * D) == 171_798_691_840
    assert a["attn_bytes"] == B * H * (S * hd * 2 * 2 + 2 * n * hd * 2) == 553_648_128
    assert a["drift_bytes"] == B * k * 2 * 16384 == 33_554_432  # cache row + probe row, K and V


def _fake_root(tmp_path):
    """A copy of the kernel sources the bench hashes, and a traffic record made for them
    (sha256 over each kernel's files in order, first 16 hex digits)."""
    import hashlib
    csrc = tmp_path / "denoising_step_attention_qkv_b300" / "csrc"
    os.makedirs(csrc, exist_ok=True)
    os.makedirs(tmp_path / "profiles", exist_ok=True)
    for fn in ("proj_rope_store.cu", "attn_cache.cu", "ptx.cuh", "internal.h"):
        shutil.copy(os.path.join(ROOT, "denoising_step_attention_qkv_b300", "csrc", fn), csrc)

    def digest(files):
        h = hashlib.sha256()
        for fn in files:
            h.update((csrc / fn).read_bytes())
        return h.hexdigest()[:16]

    rec = {"kernels": {
        "project": {"traffic_bytes": 1.25e8, "sources_sha256_16": digest(["proj_rope_store.cu", "ptx.cuh", "internal.h"])},
        "attend": {"traffic_bytes": 5.5e8, "sources_sha256_16": digest(["attn_cache.cu", "ptx.cuh", "internal.h"])}}}
    (tmp_path / "profiles" / "traffic_llada8b_b32.json").write_text(json.dumps(rec))
    return tmp_path


def test_measured_traffic_is_withdrawn_when_a_kernel_changes(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    csrc = root / "denoising_step_attention_qkv_b300" / "csrc"
    assert bench.measured_traffic("project") == 1.25e8
    assert bench.measured_traffic("attend") == 5.5e8
    with open(csrc / "attn_cache.cu", "a") as f:
        f.write("\n")
    assert bench.measured_traffic("attend") is None  # attention sources changed
    assert bench.measured_traffic("project") == 1.25e8  # not a projection source
    with open(csrc / "ptx.cuh", "a") as f:
        f.write("\n")
    assert bench.measured_traffic("project") is None  # shared header changed
    os.remove(root / "profiles" / "traffic_llada8b_b32.json")
    assert bench.measured_traffic("project") is None


def test_committed_traffic_record_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic_llada8b_b32.json")) as f:
        rec = json.load(f)
    assert rec["capture"].startswith("ncu ") and "--clock-control none" in rec["capture"]
    for key in ("project", "attend"):
        k = rec["kernels"][key]
        assert k["traffic_bytes"] > 0 and len(k["sources_sha256_16"]) == 16


def test_peaks_measured_file_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6400.0 and p["bf16_tflops"] == 1800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6459.6, "bf16_tflops": 1781.2,
                                                               "bf16_tflops_sustained": 1400.0}))
    p = bench.peaks()
    assert p == {"hbm_gbs": 6459.6, "bf16_tflops": 1781.2, "bf16_tflops_sustained": 1400.0, "source": "measured"}


@pytest.mark.parametrize("bits,names", [(0x4, ["sw_power_cap"]), (0x8 | 0x40, ["hw_slowdown", "hw_thermal_slowdown"]),
                                        (0x1, [])])
def test_clock_reason_bits(bits, names):
    # NVML clock-event reason bits: 0x4 software power cap, 0x8 hardware slowdown,
    # 0x20 software thermal, 0x40 hardware thermal, 0x80 power brake; 0x1 (GPU idle) is not reported
    assert sorted(v for k, v in bench.Clocks.REASONS.items() if bits & k) == names


def test_roofline_entry_takes_the_slower_bound():
    pk = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    D = 4096
    # batch-1 projection: 32 rows x 3D features; W's 100.7 MB at the copy rate (16.8 us)
    # outlasts its 0.8 TFLOP at the tensor rate (0.4 us), so it is HBM-bound
    flops, nbytes = 2.0 * 32 * 3 * D * D, 3 * D * D * 2 + 32 * D * 2 * 2 + 32 * 2 * D * 2
    e = bench.roofline_entry("project", 28.8, flops, nbytes, pk)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert abs(e["frac"] - nbytes / 28.8e-6 / 6000e9) < 1e-12
    assert e["frac"] > e["other_bound_frac"]
    # batch-32 step projection: 171.8 GFLOP (85.9 us at the tensor rate) against 134 MB
    wl = bench._with_drift_inputs(W.make("llada8b-b32-drift"))
    a = bench.algorithmic(wl)
    e = bench.roofline_entry("project", 120.0, a["proj_flops"], a["proj_bytes"], pk)
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s"
    assert abs(e["achieved"] - a["proj_flops"] / 120e-6 / 1e12) < 1e-9
    # a pure copy has no FLOPs: always HBM-bound
    assert bench.roofline_entry("gather", 5.0, 0.0, 16_777_216, pk)["bound"] == "hbm"
