"""Host-side arithmetic of bench.py, on CPU: the algorithmic FLOP counts that
every TFLOP/s figure divides by, the clock record that decides whether a run
counts, the peak lookup, and the DRAM-traffic records keyed by a hash of the
kernel's source."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from diffusion_transformer_image_gb300 import synth  # noqa: E402


# ------------------------------------------------------------ FLOP counts
def test_ernie_shaped_flops():
    # dense GEMMs 2MNK, non-causal attention 4 S^2 d per head
    wl = synth.WORKLOADS["ernie_full"]
    per_block, step = bench.workload_flops(wl, wl.n_layers)
    n, H, F, d, nh = 4096 + 256, 4096, 12288, 128, 32
    assert per_block["qkv"] == 2 * n * H * (3 * nh * d)
    assert per_block["attention"] == 4 * n * n * d * nh
    assert per_block["out"] == 2 * n * (nh * d) * H
    assert per_block["gate_up"] == 2 * n * H * (2 * F)
    assert per_block["down"] == 2 * n * F * H
    assert per_block["qkv"] == pytest.approx(4.381e11, rel=1e-3)
    assert per_block["attention"] == pytest.approx(3.103e11, rel=1e-3)
    assert sum(per_block.values()) == pytest.approx(2.209e12, rel=1e-3)
    # 36 blocks plus the head and tail (patch embedding, output projection in
    # two passes each, time MLP and modulation GEMVs): 7.95e13 per step
    assert step == pytest.approx(7.95e13, rel=2e-3)
    assert step > 36 * sum(per_block.values())


def test_krea_shaped_flops_use_the_kv_heads():
    wl = synth.WORKLOADS["krea_gqa"]
    per_block, _ = bench.workload_flops(wl, wl.n_layers)
    n, H = 1024 + 256, 6144
    assert per_block["qkv"] == 2 * n * H * ((48 + 2 * 8) * 128)
    assert per_block["attention"] == 4 * n * n * 128 * 48
    assert sum(per_block.values()) == pytest.approx(1.039e12, rel=1e-3)


def test_vit_flops_attend_within_each_image_and_have_no_head_tail():
    # 4 images x 1029 tokens: attention is 4 x 1029^2 x 64 x 16 x 4, not
    # (4 x 1029)^2; the pre-norm backbone has no patch embedding, time MLP or
    # output projection in its count
    wl = synth.WORKLOADS["vit_backbone"]
    per_block, fwd = bench.workload_flops(wl, wl.n_layers)
    n, S, H, d, nh, F = 4 * 1029, 1029, 1024, 64, 16, 4096
    assert per_block["attention"] == 4 * (4 * S * S * d * nh)
    assert per_block["qkv"] == 2 * n * H * 3 * nh * d
    assert per_block["gate_up"] == 2 * n * H * 2 * F
    assert fwd == 24 * sum(per_block.values())
    assert sum(per_block.values()) == pytest.approx(1.55e11, rel=1e-2)


# ------------------------------------------------------------ clock record
class _FakeSmi:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _sampler(lines):
    cs = bench.ClockSampler(0)
    cs.proc = _FakeSmi("\n".join(lines))
    return cs.stop()


def test_clock_record_median_and_power_cap():
    r = _sampler([
        "0, 1900, 2070, 1100.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1950, 2070, 1210.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2000, 2070, 1300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "not a sample",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    assert r["sm_mhz"] == 1950.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3


def test_clock_record_reports_thermal_and_hw_slowdown():
    r = _sampler([
        "0, 1500, 2070, 900, 0x0, Active, Not Active, Not Active, Not Active",
        "0, 1400, 2070, 900, 0x0, Not Active, Active, Active, Not Active",
    ])
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_record_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    cs.proc = None
    r = cs.stop()
    assert r["sm_mhz"] is None and r["reasons"] == ["nvidia-smi unavailable"]


# ------------------------------------------------------------ peaks
def test_peaks_fall_back_and_read_measured_files(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and bench.peak_value(peaks, "hbm_gbs") == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": {"value": 7100.5}, "bf16_tflops_sustained": 1650}))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert bench.peak_value(peaks, "hbm_gbs") == 7100.5
    assert bench.peak_value(peaks, "bf16_tflops_sustained") == 1650.0
    assert bench.peak_value(peaks, "bf16_tflops") == 1900.0   # absent key: fallback


# ------------------------------------------------------------ traffic records
def test_traffic_record_follows_the_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "diffusion_transformer_image_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(b"kernel v1")
    h = hashlib.sha256(b"kernel v1").hexdigest()[:12]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(
        f"# kernel-key bytes file hash\nkern 12345 k.cu {h}\nold 5 k.cu 000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("kern") == 12345.0
    assert bench.traffic_for("old") is None        # measured on another version
    assert bench.traffic_for("absent") is None
    (csrc / "k.cu").write_bytes(b"kernel v2")
    assert bench.traffic_for("kern") is None       # the kernel changed since


def test_committed_traffic_records_name_existing_sources():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    keys = []
    for line in open(path):
        f = line.split()
        if not f or line.startswith("#"):
            continue
        assert len(f) == 4 and int(f[1]) > 0 and len(f[3]) == 12
        assert os.path.exists(os.path.join(ROOT, "diffusion_transformer_image_gb300", "csrc", f[2]))
        keys.append(f[0])
    assert len(keys) == len(set(keys))
