"""Host-side logic of bench.py (CPU only): the clock record of the timed region
and the gate on the committed DRAM-traffic figure.

* ClockSampler.summary keeps only the samples taken inside the timed region,
  reports the median SM clock and every throttle reason seen there as active
  (a run with a hardware or thermal slowdown must be recognisable as such), and
  skips lines it cannot parse.
* _read_traffic reports the committed per-launch DRAM bytes only while the
  Hessian kernel's sources hash to the value recorded with the capture, and only
  for the workload it was taken on: a changed kernel has no traffic figure.
"""
import datetime
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(ts, sm, mx=2032, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return (f"{ts.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {sm}, {mx}, 900.00, 0x0000000000000000, "
            f"{hw}, {hwt}, {swt}, {cap}")


def _sampler(lines, start, stop):
    s = bench.ClockSampler(0)
    s.lines = list(lines)
    s.start, s.stop = start, stop
    return s


def test_clock_summary_uses_only_the_timed_region():
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    step = datetime.timedelta(milliseconds=100)
    lines = [_line(t0 + i * step, sm) for i, sm in enumerate([1200, 2032, 2017, 2032, 1100])]
    s = _sampler(lines, t0 + step, t0 + 3 * step)
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2032
    assert out["sm_max_mhz"] == 2032
    assert out["reasons"] == []


def test_clock_summary_reports_active_throttle_reasons():
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    step = datetime.timedelta(milliseconds=100)
    lines = [_line(t0, 2032),
             _line(t0 + step, 1800, hw="Active"),
             _line(t0 + 2 * step, 1900, cap="Active"),
             _line(t0 + 3 * step, 1700, swt="Active"),
             _line(t0 + 10 * step, 900, hwt="Active")]  # outside the window: ignored
    out = _sampler(lines, t0, t0 + 3 * step).summary()
    assert out["samples"] == 4
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == (1800 + 1900) / 2


def test_clock_summary_without_samples_and_with_garbage():
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    lines = ["not a csv line", "a, b, c", _line(t0, "[N/A]")]
    out = _sampler(lines, t0, t0 + datetime.timedelta(seconds=1)).summary()
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def _write_record(root, workload, sha):
    os.makedirs(os.path.join(root, "profiles"))
    csrc = os.path.join(root, "post_weight_quantization_30_b300", "csrc")
    os.makedirs(csrc)
    for n, body in (("hessian_tc.cu", b"kernel A"), ("tc_common.cuh", b"helpers")):
        with open(os.path.join(csrc, n), "wb") as f:
            f.write(body)
    rec = {"workload": workload, "dram_bytes_per_launch": 123456789,
           "kernel_source_sha256": sha if sha else hashlib.sha256(b"kernel Ahelpers").hexdigest()}
    with open(os.path.join(root, "profiles", "hessian_traffic.json"), "w") as f:
        json.dump(rec, f)


def test_traffic_is_reported_only_for_the_captured_kernel_and_workload(tmp_path, monkeypatch):
    _write_record(str(tmp_path), "llama7b_q_proj_4096x4096 (X 262144x4096 bf16)", None)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._read_traffic("llama7b_q_proj_4096x4096") == 123456789
    assert bench._read_traffic("qwen32b_5120x5120") is None
    # the kernel changed since the capture: no figure
    with open(os.path.join(str(tmp_path), "post_weight_quantization_30_b300", "csrc", "hessian_tc.cu"), "ab") as f:
        f.write(b" edited")
    assert bench._read_traffic("llama7b_q_proj_4096x4096") is None


def test_traffic_with_a_stale_hash_or_no_record(tmp_path, monkeypatch):
    _write_record(str(tmp_path), "llama7b_q_proj_4096x4096", "0" * 64)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._read_traffic("llama7b_q_proj_4096x4096") is None
    os.remove(os.path.join(str(tmp_path), "profiles", "hessian_traffic.json"))
    assert bench._read_traffic("llama7b_q_proj_4096x4096") is None



class _KT:
    """A stand-in for the library's per-class timing record."""

    def __init__(self, ms, flops, count):
        self.ms, self.flops, self.count = ms, flops, count


def test_phase_rooflines_arithmetic():
    """Each phase's roofline from its time and algorithmic work: the factor as cols^3/3 flops against
    the 3xTF32 rate (measured bf16 burst x 1.1/2.25 / 3), sweep + pack as bytes against the HBM copy
    rate with the chain floor cols x (block-kernel time per column step: the kernels' time over the
    cols columns they sweep, one or two blocks per launch), the GEMM class as its
    declared useful flops over its summed time."""
    from synthetic import LAYERS

    spec = LAYERS["llama7b_down_proj_4096x11008"]
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0}
    kt = _KT(ms={"hessian": 20.0, "gemm3": 8.0, "sweep": 2.0, "diag": 4.0, "gemm_tf32": 0.0},
             flops={"hessian": 3.2e13, "gemm3": 9.6e11, "sweep": 0.0, "diag": 0.0, "gemm_tf32": 0.0},
             count={"hessian": 1, "gemm3": 250, "sweep": 86, "diag": 86, "gemm_tf32": 0})
    phase = {"hessian": 20.0, "factor": 8.0, "sweep": 6.0}
    out = bench.phase_rooflines(spec, phase, kt, peaks, "measured", codes=False, w_hat=False)
    tf32x3 = 1800.0 * 1.1 / 2.25 / 3
    assert out["factor"]["peak"] == round(tf32x3, 1)
    assert out["factor"]["achieved"] == round(11008 ** 3 / 3 / 8e-3 / 1e12, 2)
    byt = 4096 * 11008 * 2 + 4096 * 11008 * 3 / 8 + (11008 // 128) * 4096 * (4 + 3 / 8) + 11008 * 4
    assert bench.sweep_pack_bytes(spec, False, False) == byt
    assert out["sweep_pack"]["achieved"] == round(byt / 6e-3 / 1e9, 1)
    assert out["sweep_pack"]["column_step_ns"] == round(2.0e6 / 11008, 2)
    assert out["sweep_pack"]["chain_floor_ms"] == round(11008 * (2.0e6 / 11008) / 1e6, 4)
    assert out["gemm3"]["achieved"] == round(9.6e11 / 8e-3 / 1e12, 2)
    assert out["gemm3"]["frac"] == round(out["gemm3"]["achieved"] / tf32x3, 4)
    assert out["hessian"]["frac"] == round(3.2e13 / 20e-3 / 1e12 / 1800.0, 4)
    # optional outputs add their bytes
    assert bench.sweep_pack_bytes(spec, True, True) == byt + 4096 * 11008 * 5
