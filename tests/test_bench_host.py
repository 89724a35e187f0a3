"""Host-side pieces of bench.py: the CPU baseline leg (the oracle timed on a
bounded sample, with the step time it implies) and the per-workload FLOP and
byte models behind the roofline."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_cpu_baseline_tiny_keys_and_single_core():
    w = synth.WORKLOADS["tiny"]
    cb = bench.cpu_baseline(w)
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT and cb["cores"] >= 1
    assert cb["value"] > 0 and cb["step_s"] > 0 and cb["step_s_kind"] == "measured"
    assert "whole step" in cb["sample"]
    one = cb.get("single_core")
    if one is not None:  # the child process may be unavailable in odd sandboxes
        assert one["cores"] == 1 and one["value"] > 0


@pytest.mark.parametrize("name", ["gpt", "swiglu", "sp", "narrow", "attn_proj"])
def test_kernel_flops_add_up_to_the_step(name):
    """The per-GEMM FLOP model sums to the workload's algorithmic FLOP."""
    w = synth.WORKLOADS[name]
    kf = bench.kernel_flops(w)
    names = (["col_fwd", "row_fwd", "col_dgrad", "wgrad_col", "row_dgrad", "wgrad_row"] if w.kind == "attn_proj"
             else ["col_fwd", "row_fwd", "row_dgrad_act", "wgrad_row", "wgrad_col", "col_dgrad"])
    assert sum(kf[n] for n in names) == pytest.approx(w.flops(), rel=1e-12)
    gb = bench.gemm_bytes(w)
    for n in names:
        assert gb[n] > 0
        if name != "narrow":  # the wide workloads' GEMMs sit far above the ridge point
            assert kf[n] / gb[n] > 300
    if name == "narrow":  # H = 256: the act' dgrad is below it (HBM bound)
        assert kf["row_dgrad_act"] / gb["row_dgrad_act"] < 300


def test_step_bytes_counts_each_tensor_once():
    w = synth.WORKLOADS["gpt"]
    M, H, F = w.M, w.H, w.F
    expect = 2 * (4 * M * H + 2 * M * F + 2 * F * H) + 4 * 2 * F * H
    assert bench.step_bytes(w) == expect


def test_peak_follows_the_timed_region():
    """A timed region shorter than the sustained measurement's 4 s is
    compared against the burst peak, a longer one against the sustained
    peak; FP8 takes twice the bf16 figure."""
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "measured"}
    p, kind = bench.pick_peak(peaks, 0.074, "bf16")
    assert p == 1900.0 and "burst" in kind and "0.07 s" in kind
    p, kind = bench.pick_peak(peaks, 12.0, "bf16")
    assert p == 1700.0 and "sustained" in kind
    p, kind = bench.pick_peak(peaks, 1.0, "fp8")
    assert p == 3800.0 and kind.startswith("fp8")


def test_fp32_engine_peak_from_unit_counts():
    """The fp32 engine's roof: SMs x 128 FP32 lanes x 2 FLOP x the maximum
    SM clock (GB300: 152 SMs at 2070 MHz, 80.6 TFLOP/s)."""
    import bench
    peak, kind = bench.fp32_alu_peak(152, {"sm_max_mhz": 2070.0})
    assert abs(peak - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
    assert abs(peak - 80.55) < 0.01 and "FFMA" in kind
