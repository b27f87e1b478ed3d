"""Host-side logic of bench.py that its JSON line rests on (no GPU): the algorithmic
work behind the roofline entry, the choice of the binding resource and of the peak,
the L2 flush rule, the DRAM-traffic record's source check, and the clock summaries
(NVML reason bits, the busy-window filter, the nvidia-smi fallback's parser).

Expected values come from elsewhere than the formulas under test: byte counts from
arrays of the shapes the path moves, reason bits from NVML's own Python bindings."""

import json
import os
import sys
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import Workload  # noqa: E402


def _bytes_moved(w, counts, m_rows):
    """The bytes one fused launch and one combine touch, summed over arrays of the
    shapes the path reads and writes (A, the weights of experts with rows, the rows
    sent; the received rows, the gates and the combined output)."""
    fp8 = w.dtype == "fp8_1d2d"
    el = np.uint8 if fp8 else np.uint16
    nonempty = int((counts.sum(axis=1) > 0).sum())
    arrays = [np.zeros((m_rows, w.K), el), np.zeros((nonempty, w.N, w.K), el),
              np.zeros((m_rows, w.N), np.uint16)]
    if fp8:
        arrays += [np.zeros((m_rows, w.K // 128), np.float32),
                   np.zeros((nonempty, w.N // 128, w.K // 128), np.float32)]
    send = sum(a.nbytes for a in arrays)
    comb = (np.zeros((w.tokens, w.top_k, w.N), np.uint16).nbytes
            + np.zeros((w.tokens, w.N), np.uint16).nbytes
            + np.zeros((w.tokens, w.top_k), np.float32).nbytes)
    return send, comb


@pytest.mark.parametrize("dtype", ["bf16", "fp8_1d2d"])
def test_algorithmic_work_counts_what_the_path_moves(dtype):
    w = Workload("wk", 2, 3, 2, 40, 256, 384, dtype, "uniform", "softmax_sel", 1)
    counts = np.array([[5, 2], [0, 0], [1, 0]])  # expert 1 receives nothing
    m_rows = int(counts.sum())
    flops, send, comb = bench.algorithmic_work(w, counts, m_rows)
    exp_send, exp_comb = _bytes_moved(w, counts, m_rows)
    assert send == exp_send and comb == exp_comb
    # one multiply and one add per (row, k, n)
    assert flops == 2 * np.ones((m_rows, w.K)).dot(np.ones((w.K, w.N))).sum()


def test_roofline_names_the_binding_resource_and_its_peak():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0}
    bf16 = Workload("b", 1, 1, 1, 1, 128, 128, "bf16", "uniform", "softmax_sel", 1)
    fp8 = Workload("f", 1, 1, 1, 1, 128, 128, "fp8_1d2d", "uniform", "softmax_sel", 1)
    # 2 TFLOP over 1 GB: compute takes 2 ms at 1 PFLOP/s, memory 0.2 ms at 5 TB/s
    r = bench.roofline(bf16, 2e12, 1e9, 4e-3, peaks, "measured", traffic=123)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 123
    assert r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)
    # fp8 doubles the tensor peak (the nominal fp8 / bf16 ratio) and says so
    r = bench.roofline(fp8, 2e12, 1e9, 4e-3, peaks, "measured")
    assert r["peak"] == 2000.0 and r["frac"] == pytest.approx(0.25)
    assert "x2" in r["peak_source"]
    # 1 GFLOP over 1 GB: memory-bound; frac against the copy bandwidth
    r = bench.roofline(bf16, 1e9, 1e9, 0.4e-3, peaks, "fallback")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(2500.0) and r["frac"] == pytest.approx(0.5)
    assert r["peak_source"].startswith("fallback")


def test_l2_flush_only_for_working_sets_under_twice_the_l2():
    small = Workload("s", 2, 2, 2, 64, 256, 128, "bf16", "uniform", "softmax_sel", 1)
    flush, text = bench.l2_policy(small, 100)
    assert flush and text == bench.FLUSH_TEXT
    big = Workload("g", 8, 1, 2, 4096, 14336, 4096, "bf16", "uniform", "softmax_sel", 1)
    flush, text = bench.l2_policy(big, 8192)
    assert not flush and "> L2" in text
    # the boundary: operand bytes exactly at twice the L2 are no longer flushed
    K = N = 1024
    w = Workload("e", 1, 1, 1, 1, K, N, "bf16", "uniform", "softmax_sel", 1)
    rows = -(-(2 * bench.L2_BYTES - N * K * 2) // (K * 2))  # first row count at or past it
    assert bench.l2_policy(w, rows - 1)[0] and not bench.l2_policy(w, rows)[0]


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    rec = {"mixtral_prefill": {"grouped_gemm_combine_send": {
        "bytes_per_launch": 4242, "source_sha": "feedface00000000"}}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "feedface00000000")
    assert bench.measured_traffic("mixtral_prefill", "grouped_gemm_combine_send") == 4242
    assert bench.measured_traffic("qwen3_skew", "grouped_gemm_combine_send") is None
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0123456789abcdef")
    assert bench.measured_traffic("mixtral_prefill", "grouped_gemm_combine_send") is None


def test_source_digest_ignores_comments_only():
    a = "int f() {\n  return 1; // one\n}\n/* a\n   block */\n\n"
    b = "// header\nint f() {\n  return 1;\n}\n"
    assert bench._code_only(a) == bench._code_only(b) == "int f() {\n  return 1;\n}"
    assert bench._code_only("int f() { return 2; }") != bench._code_only(b)
    assert len(bench.kernel_source_sha()) == 16


def test_nvml_reason_bits_match_nvml():
    pynvml = pytest.importorskip("pynvml")
    names = {"sw_power_cap": "SwPowerCap", "hw_slowdown": "HwSlowdown",
             "sw_thermal_slowdown": "SwThermalSlowdown",
             "hw_thermal_slowdown": "HwThermalSlowdown",
             "hw_power_brake_slowdown": "HwPowerBrakeSlowdown"}
    for bit, name in bench.NvmlClocks.REASONS.items():
        assert getattr(pynvml, "nvmlClocksThrottleReason" + names[name]) == bit


def test_nvml_summary_keeps_the_busy_window():
    s = object.__new__(bench.NvmlClocks)
    s.lib = object()
    s.thread = types.SimpleNamespace(join=lambda: None)
    s.max_sm_mhz = lambda: 2070
    # (time, SM MHz, reason bits, watts): idle before and after, loaded in between
    s.samples = [(0.0, 2070, 0x1, 90.0), (1.0, 1800, 0x4, 1300.0), (1.1, 1700, 0x4, 1350.0),
                 (1.2, 1750, 0x0, 1200.0), (3.0, 2070, 0x1, 95.0)]
    out = s.stop(busy=(0.5, 2.0))
    assert out["samples"] == 3 and out["sm_mhz"] == 1750 and out["sm_mhz_min"] == 1700
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_max"] == 1350.0
    assert out["sm_max_mhz"] == 2070
    # a window that holds no sample keeps them all rather than reporting nothing
    s.thread = types.SimpleNamespace(join=lambda: None)
    assert s.stop(busy=(5.0, 6.0))["samples"] == 5


def test_nvidia_smi_fallback_parses_its_csv(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1980, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 1965, 2070, 1120.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 2070, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "garbled line\n")
    c = bench.ClockSampler(0)
    c.proc = types.SimpleNamespace(terminate=lambda: None, wait=lambda timeout=None: 0,
                                   kill=lambda: None)
    c.fh = open(tmp_path / "sink.txt", "w")
    c.path = str(path)
    out = c.stop()
    assert out["samples"] == 3 and out["sm_mhz"] == 1980 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert not path.exists()  # the sampler removes its file


def test_clock_sampler_falls_back_without_nvml(monkeypatch):
    import ctypes

    def no_lib(*a, **k):
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")
    monkeypatch.setattr(ctypes, "CDLL", no_lib)
    assert isinstance(bench.clock_sampler(0), bench.ClockSampler)
