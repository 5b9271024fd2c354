"""Host-side helpers of bench.py on the CPU: the byte counts behind the GB/s figures
and the oracle samples that the CPU baselines time (small samples, short minimum
times, so the suite stays fast)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = {"value", "unit", "cores", "kind", "sample", "seconds"}


def test_bytes_io_counts_every_output():
    # 32 x 48: x 2 bytes each, codes half a byte per element in each direction,
    # one scale byte per 16 elements in each direction, one float amax per line
    assert bench.bytes_io(32, 48) == 2 * 32 * 48 + (32 * 24 + 48 * 16) + (32 * 3 + 48 * 2) \
        + 4 * (32 + 48)
    # odd sizes round the packed codes and the partial blocks up
    assert bench.bytes_io(17, 33) == 2 * 17 * 33 + (17 * 17 + 33 * 9) + (17 * 3 + 33 * 2) \
        + 4 * (17 + 33)


def test_quant_bytes_by_dtype_and_mode():
    assert bench.quant_bytes(32, 48) == bench.bytes_io(32, 48)
    # FP32 input reads 4 bytes per value; per-tensor writes one amax per direction
    assert bench.quant_bytes(32, 48, 4, True) == bench.bytes_io(32, 48) + 2 * 32 * 48
    assert bench.quant_bytes(32, 48, 2, False) == bench.bytes_io(32, 48) - 4 * 80 + 8


@pytest.mark.parametrize("w", ["rht", "rht-both", "dequant", "moe-col", "weights16x16", "moe", "outliers",
                               "edge", "tiny"])
@pytest.mark.parametrize("threads", [1, 2])
def test_supplementary_oracle_samples_repeat_to_the_minimum_time(w, threads):
    r = bench.supplementary_oracle_sample(w, 16, min_seconds=0.2, threads=threads)
    assert KEYS <= set(r) and r["kind"] == "oracle" and r["cores"] == threads
    assert r["seconds"] >= 0.2 and r["value"] > 0 and r["unit"] == "GB/s"
    assert r["sample"].endswith("round(s)") and r["sample"].startswith(f"{threads} strip")


def test_headline_oracle_sample_strips():
    jobs, nbytes, what = bench.prepare_oracle_sample(8, threads=3)
    assert len(jobs) == 3
    assert nbytes == 3 * (bench.bytes_io(8, bench.K_X) + bench.bytes_io(8, bench.K_DY))
    dt, rounds = bench.timed_strips(jobs, 3, 0.1)
    assert dt >= 0.1 and rounds >= 1
    r = bench.oracle_sample(8, threads=2, min_seconds=0.1)
    assert KEYS <= set(r) and r["cores"] == 2


def test_host_cores_is_positive():
    assert bench.host_cores() >= 1


def test_gemm_oracle_sample_counts_its_flops():
    r = bench.gemm_oracle_sample(8, 64)
    assert KEYS <= set(r) and r["unit"] == "TFLOP/s"
    assert abs(r["value"] - 2 * 8 * 8 * 64 / r["seconds"] / 1e12) <= 1e-9 * r["value"]


def test_job_throughput_single_rank():
    t, rate = bench.job_throughput(2.0, 1, 100.0, 4)
    assert t == 2.0 and rate == 200.0  # 100 units x 4 steps in 2 s
