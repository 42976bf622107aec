"""Host logic of bench.py that decides whether a bench line is valid (CPU).

- the DRAM traffic record is used only while the GEMM source it was taken on
  is unchanged (null otherwise);
- the nvidia-smi clock sampler reports the median SM clock and every throttle
  reason that was active in any sample;
- the whole-job rate counts every rank's work over the slowest rank's time.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_record_matches_the_committed_gemm_source():
    t = bench._traffic_for_current_gemm()
    assert t is not None, "profiles/ traffic record does not match gemm_pair.cu"
    # the record is read + write bytes of one launch
    kv = dict(line.split("=", 1) for line in open(bench.TRAFFIC_FILE).read().split() if "=" in line)
    assert t == float(kv["dram_bytes_read"]) + float(kv["dram_bytes_write"])
    # reads cover at least the operand codes of prefill MLP-up (x_q and W); the
    # writes need not reach the bf16 output's size, since part of it can still
    # sit in the L2 when the kernel ends
    M, N, K = 4096, 14336, 4096
    assert float(kv["dram_bytes_read"]) >= M * K + N * K


def test_traffic_is_null_once_the_gemm_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "gemm_pair.cu"
    src.write_bytes(open(bench.GEMM_SOURCE, "rb").read() + b"\n// edited\n")
    monkeypatch.setattr(bench, "GEMM_SOURCE", str(src))
    assert bench._traffic_for_current_gemm() is None


def test_traffic_is_null_without_a_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench._traffic_for_current_gemm() is None


class _FakeSmi:
    """Stands in for the nvidia-smi child process: returns canned CSV rows."""

    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _row(sm, reasons=("Not Active",) * 4, smax=2070, power=900.0):
    return ", ".join(["0", str(sm), str(smax), str(power), "0x0000000000000000", *reasons])


def _sampled(rows):
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("\n".join(rows) + "\n")
    return s.stop()


def test_clock_sampler_median_and_no_reasons():
    c = _sampled([_row(2070), _row(2055), _row(2070), "garbage line", _row(2040)])
    assert c["sm_mhz"] == pytest.approx(2062.5)
    assert c["sm_max_mhz"] == 2070
    assert c["samples"] == 4
    assert c["reasons"] == []


@pytest.mark.parametrize("which,name", [(0, "hw_slowdown"), (1, "hw_thermal_slowdown"),
                                        (2, "sw_thermal_slowdown"), (3, "sw_power_cap")])
def test_clock_sampler_reports_each_active_reason(which, name):
    active = ["Not Active"] * 4
    active[which] = "Active"
    c = _sampled([_row(2070), _row(1800, tuple(active)), _row(2070)])
    assert c["reasons"] == [name]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    c = s.stop()
    assert c["sm_mhz"] is None and c["reasons"] == ["nvidia-smi unavailable"]


def test_job_rate_counts_all_ranks_over_the_slowest():
    flops = 2.0 * 4096 * 14336 * 4096
    one = bench.job_tflops(flops, steps=10, world=1, max_total_ms=2.0)
    assert one == pytest.approx(flops * 10 / 2e-3 / 1e12)
    # two replicas doing the same work in the same (slowest-rank) time: twice the rate
    assert bench.job_tflops(flops, steps=10, world=2, max_total_ms=2.0) == pytest.approx(2 * one)
    assert bench.max_over_ranks(3.5) == 3.5  # no process group: this rank's own time
