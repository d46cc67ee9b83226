"""Host-side arithmetic of the benchmark (no GPU): algorithmic bytes and FLOPs of the
attention launch, the L2 labelling of a workload, the whole-job aggregate."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import mla_inputs  # noqa: E402


def test_v3_batch64_roofline_figures():
    """262,208 rows of 1,152 B (512 + 64 bf16) and 2*128*(576 + 512) FLOP per row."""
    wl = mla_inputs.WORKLOADS["v3_b64_l4096"]
    lens = mla_inputs.context_lengths(wl)
    rows, nbytes, flops = bench.workload_facts(wl, lens)
    assert rows == 64 * 4097
    assert nbytes == rows * 1152 == 302_063_616
    assert flops == rows * 278_528
    assert bench.step_footprint(wl, lens) > bench.L2_BYTES
    assert bench.l2_note(wl, lens).startswith("inputs larger than L2")


def test_small_sweep_point_is_labelled_l2_resident():
    wl = [w for w in mla_inputs.sweep_workloads() if w.batch == 1 and w.prefill == 512][0]
    lens = mla_inputs.context_lengths(wl)
    assert bench.step_footprint(wl, lens) < bench.L2_BYTES
    assert bench.l2_note(wl, lens).startswith("inputs fit in L2")


def test_fp32_rows_count_four_bytes():
    wl = mla_inputs.WORKLOADS["tiny_f32"]
    lens = mla_inputs.context_lengths(wl)
    rows, nbytes, _ = bench.workload_facts(wl, lens)
    assert nbytes == rows * (wl.d_c + wl.d_r) * 4


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(64, 8, 1000, 150.0) == pytest.approx(64 * 8 * 1000 / 0.150)


def test_clock_summary_keeps_only_samples_inside_the_windows():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.period, cs.error, cs.source = 0.002, None, "nvml"
    cs.rows = [(1.0, 1000.0, 2032.0, 0), (2.0, 2032.0, 2032.0, 0x4), (2.5, 1900.0, 2032.0, 0),
               (3.0, 500.0, 2032.0, 0x40 | 0x8)]
    s = cs.summary([(1.9, 2.6)])
    assert s["samples"] == 2 and s["sm_mhz"] == 1966.0 and s["reasons"] == ["sw_power_cap"]
    s = cs.summary([(0.5, 1.5), (2.9, 3.1)])
    assert s["samples"] == 2 and s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    s = cs.summary([(5.0, 6.0)])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["error"]


def test_named_workloads_cover_configs_and_sweep_points():
    named = bench.named_workloads()
    for name in ("tiny_f32", "small_bf16", "v3_b64_l4096", "v3_ragged_b16", "v3_sweep_b128_l8192"):
        assert name in named
    sweep = [n for n in named if n.startswith("v3_sweep_")]
    assert len(sweep) == len(mla_inputs.SWEEP_BATCHES) * len(mla_inputs.SWEEP_CONTEXTS)
    w = named["v3_sweep_b256_l32768"]
    assert (w.batch, w.prefill, w.seed) == (256, 32768, 4)
