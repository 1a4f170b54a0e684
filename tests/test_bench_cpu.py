"""The bench's reporting arithmetic, on the CPU: the protocol's launch counts,
the per-arm record (µs per call, GB/s of algorithmic bytes, the fraction of
the measured peak, TFLOP/s for the prefill GEMM) and the rejection rule."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6785.2, "bf16_tflops": 1905.0}


class FakeArm:
    name = "bf16 x bf16 GEMV M=1 K=4096 N=12288"
    bytes_per_call = 100720640
    R = 11
    launches_per_call = 1
    route = "lanes_per_row_rows"


def timing(us_per_call, spread=0.004, repeats=10, per_repeat=200):
    calls = repeats * per_repeat
    return {"repeats": repeats, "launches_per_repeat": per_repeat, "seconds": us_per_call * 1e-6 * calls,
            "spread": spread, "spread_ok": spread < bench.MAX_SPREAD}


@pytest.mark.parametrize("steps,per_repeat", [(1, 200), (20, 200), (2000, 200), (2001, 201), (5000, 500)])
def test_protocol_is_ten_repeats_of_at_least_200_launches(steps, per_repeat):
    assert bench.protocol_launches(steps) == (10, per_repeat)


def test_gemv_record():
    rec = bench.arm_record(FakeArm(), timing(15.41), PEAKS)
    assert rec["timed_calls"] == 2000 and rec["launches"] == 2000
    assert rec["us_per_call"] == pytest.approx(15.41)
    assert rec["GB_per_s"] == pytest.approx(100720640 / 15.41e-6 / 1e9, abs=0.05)
    assert rec["frac_of_peak"] == pytest.approx(100720640 / 15.41e-6 / 1e9 / 6785.2, abs=1e-4)
    assert rec["working_set_bytes"] == 11 * 100720640 and rec["route"] == "lanes_per_row_rows"


def test_gemm_record_reports_the_tensor_peak():
    arm = FakeArm()
    arm.name, arm.bytes_per_call, arm.flops = "q4_0 x bf16 prefill GEMM", 66584576, 2.0 * 512 * 14336 * 4096
    rec = bench.arm_record(arm, timing(62.94), PEAKS)
    assert rec["bound"] == "tensor" and "frac_of_peak" not in rec
    assert rec["TFLOP_per_s"] == pytest.approx(60129542144 / 62.94e-6 / 1e12, abs=0.05)
    assert rec["frac_of_tensor_peak"] == pytest.approx(60129542144 / 62.94e-6 / 1e12 / 1905.0, abs=1e-4)


def test_a_rejected_measurement_carries_no_rate():
    t = timing(15.41, spread=0.08)
    t["rejected"] = True
    rec = bench.arm_record(FakeArm(), t, PEAKS)
    assert rec["rejected"] and not rec["spread_ok"]
    assert not any(k in rec for k in ("us_per_call", "GB_per_s", "frac_of_peak"))
