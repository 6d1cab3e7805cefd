"""The benchmark's JSON line keeps the keys its readers need: the headline
line built from a measurement (no GPU needed to build it), and the
reference arm (the CPU oracle) run end to end on the tiny workload."""
import argparse
import json
import os
import subprocess
import sys

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _head():
    wl = synth.workloads()["siso_b8_l4096"]
    return {"value": 7.1e7, "unit": "tokens/s", "ms_per_step": 0.46, "dtype": "f16x2",
            "config": bench.config_of(wl),
            "roofline": {"bound": "hbm", "achieved": 2368.0, "peak": 6486.1, "unit": "GB/s", "frac": 0.365,
                         "traffic": 1.08e9, "algorithmic_bytes_per_launch": 1094909952},
            "e2e": {"value": 1.6e6, "unit": "tokens/s", "h2d_bytes_per_step": 809500672,
                    "d2h_bytes_per_step": 268435456},
            "gpu_launches": 20, "device_status": 0,
            "clocks": {"sm_mhz": 2032.0, "sm_max_mhz": 2032, "reasons": []}, "parity": {"units": [0, 255]}}


def test_headline_line_has_the_contract_keys():
    args = argparse.Namespace(steps=20, warmup=3, algo="auto")
    cpu = {"value": 1.1e4, "unit": "tokens/s", "cores": 16, "kind": "oracle", "sample": "16 of 256 units"}
    line = json.loads(json.dumps(bench.contract_line(_head(), cpu, [], args, 1)))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
              "clocks"):
        assert k in line, k
    assert line["config"]["workload"] == "siso_b8_l4096" and "l2" in line["config"]
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert set(line["cpu_baseline"]) >= {"value", "unit", "cores", "kind", "sample"}
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_f32",
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["cpu_baseline"]) >= {"value", "cores", "kind", "sample"}


class _FakeNvml:
    """Stands in for the NVML library (reading only): a scripted SM clock
    and throttle-reason word per query."""

    def __init__(self, script):
        self.script, self.calls = list(script), 0

    def _next(self):
        i = min(self.calls, len(self.script) - 1)
        return self.script[i]

    def nvmlDeviceGetClockInfo(self, h, kind, ref):
        ref._obj.value = self._next()[0]
        return 0

    def reasons(self, h, ref):
        ref._obj.value = self._next()[1]
        self.calls += 1
        return 0


def test_clock_sampler_keeps_only_the_timed_region():
    """The sampler drops what it saw before restart() (the warm-up), takes a
    sample at the region's start, decodes the throttle-reason bits and stops
    its thread on exit; a box without NVML reports the error, no samples."""
    import ctypes
    import time

    fake = _FakeNvml([(1500, 0x8)] * 3 + [(2032, 0x4)])  # warm-up: hw_slowdown; region: sw_power_cap
    clk = bench.ClockSampler(0, period_s=0.001)

    def fake_open():
        clk.lib, clk.h, clk.ct, clk.max_mhz = fake, ctypes.c_void_p(), ctypes, 2032
        clk.get_reasons = fake.reasons

    clk._open = fake_open
    with clk:
        while fake.calls < 4:  # the warm-up's three samples are all in (the thread samples in turn)
            time.sleep(0.001)
        clk.restart()
        time.sleep(0.01)
    s = clk.summary()
    assert not clk.th.is_alive()
    assert s["sm_mhz"] == 2032 and s["sm_max_mhz"] == 2032 and s["samples"] >= 1
    assert s["reasons"] == ["sw_power_cap"], s

    bad = bench.ClockSampler(0)

    def no_nvml():
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")

    bad._open = no_nvml
    with bad:
        bad.restart()
    assert bad.summary()["sm_mhz"] is None and "no samples" not in bad.summary()["reasons"][0]
