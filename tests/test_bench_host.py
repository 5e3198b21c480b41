"""Host-side logic of bench.py (no GPU): the algorithmic byte count of attention, the choice of
the roofline that binds attention, the staleness check of a committed DRAM-traffic record,
and the clock sampler's aggregation."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import dflash_inputs as di  # noqa: E402


def test_attention_cache_bytes_count_readable_positions():
    w = di.WORKLOADS["decode_8b_b8_ctx4096"]
    anchors, valid, _ = di.inference_block_layout(w)
    mask = di.gen_mask(w)
    work = bench.algorithmic_work(w, {"anchors": anchors, "block_valid": valid}, mask)
    s = w.shape
    # every row reads, per layer, K and V (fp16) of its positions below its largest anchor
    # whose mask is 1
    readable = 0
    for b in range(w.batch):
        a = max(int(x) for x in anchors[b] if x >= 0)
        readable += int(mask[b, :min(a, w.seq_len)].sum())
    assert work["ctx_positions"] == readable
    assert work["attn_cache_bytes"] == readable * 2 * s.kv_width * 2 * s.num_layers


def test_attention_roofline_picks_the_binding_side():
    work = {"attn_flops": 1e12, "attn_cache_bytes": 1e9}
    # 1e9 bytes at 100 GB/s = 10 ms > 1e12 FLOP at 1000 TFLOP/s = 1 ms: HBM binds; the step
    # measured 4 ms over 2 steps = 2 ms per step
    r = bench.attention_roofline(work, 4.0, 2, peak_tflops=1000.0, hbm_gbs=100.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(10e-3 / 2e-3)
    assert r["achieved"] == pytest.approx(1e9 / 2e-3 / 1e9)
    assert r["frac_tensor"] == pytest.approx(1e-3 / 2e-3)
    r = bench.attention_roofline(work, 4.0, 2, peak_tflops=100.0, hbm_gbs=1e6)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(10e-3 / 2e-3)
    assert bench.attention_roofline(work, 0.0, 2, 1.0, 1.0)["frac"] is None


def test_traffic_record_is_dropped_once_its_sources_change(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"kernel as profiled")
    (tmp_path / "profiles").mkdir()
    rec = {"sources": ["kernel.cu"], "dram_bytes_per_launch": 123.0,
           "source_sha256": hashlib.sha256(b"kernel as profiled").hexdigest()}
    (tmp_path / "profiles" / "gemm_traffic_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("w") == 123.0
    src.write_bytes(b"kernel changed since")
    assert bench.profiled_traffic("w") is None
    assert bench.profiled_traffic("no_such_workload") is None


class _FakeNvml:
    def __init__(self, samples):
        self.samples = samples

    def start(self):
        pass

    def stop(self):
        return self.samples


def _no_popen(*a, **k):
    raise OSError("no nvidia-smi")


def test_clock_sampler_aggregates_nvml_samples(monkeypatch):
    monkeypatch.setattr(subprocess, "Popen", _no_popen)
    c = bench.ClockSampler(0)
    # (SM MHz, max SM MHz, event-reason bits): 0x4 software power cap, 0x20 software thermal
    c.nvml = _FakeNvml([(2070, 2070, 0), (1900, 2070, 0x4), (2000, 2070, 0x20)])
    c.start()
    out = c.stop()
    assert out["sm_mhz"] == 2000 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert out["samples"] == 3 and out["samples_nvml"] == 3


def test_clock_sampler_without_any_source(monkeypatch):
    monkeypatch.setattr(subprocess, "Popen", _no_popen)
    c = bench.ClockSampler(0)
    c.nvml = None
    c.start()
    out = c.stop()
    assert out["sm_mhz"] is None and out["reasons"]


def test_gemm_roofline_uses_burst_peak_and_picks_the_binding_side():
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 8000.0,
             "source": "test"}
    # 1e12 FLOP over 1e9 weight bytes: 1000 FLOP/B, above the ridge (250): tensor-bound
    work = {"gemm_flops": 1e12, "layer_weight_bytes": 1e9, "ctx_weight_bytes": 0.0}
    r = bench.gemm_roofline(work, False, 10.0, 10, 2, peaks)   # 1 ms per launch
    assert r["bound"] == "tensor" and r["peak"] == 2000.0
    assert r["algorithmic_per_launch"] == pytest.approx(2e11)
    assert r["achieved"] == pytest.approx(2e11 / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / 1600.0)
    # a decode step: 32 FLOP per weight byte, below the ridge: weight-read bound
    work = {"gemm_flops": 3.2e10, "layer_weight_bytes": 1e9, "ctx_weight_bytes": 5e8}
    r = bench.gemm_roofline(work, True, 10.0, 10, 2, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_per_launch"] == pytest.approx(1e9 * 2 / 10)


def test_oracle_sample_prefix_is_bounded():
    assert bench.oracle_prefix(di.WORKLOADS["train_8b_b16_l4096"]) == 1024
    assert bench.oracle_prefix(di.WORKLOADS["longctx_8b_l32768"]) == 8192
    assert bench.oracle_prefix(di.WORKLOADS["tiny_f32"]) == 128
    assert bench.valid_rows(di.WORKLOADS["train_8b_b4_l2048"]) == [0, 1, 2]
