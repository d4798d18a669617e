"""Host-side arithmetic of the benchmark report (no GPU): the algorithmic work per direction equals the
figures derived from the workload shapes, and the per-direction report divides them correctly."""

import pytest

import bench
from gated_delta_rule_38_gb300.inputs import WORKLOADS


def test_dense_workload_bytes_and_flops():
    wk = bench.work(WORKLOADS["dense"])
    tok, H, K = 2 * 4096, 32, 128
    # forward-only: q, k, v, g, beta in and o out, 16-bit
    assert wk["fwd_only_bytes"] == tok * H * (2 * K * 2 + K * 2 + 2 * 2 + K * 2)
    # the training forward adds A (64 16-bit values) and g_cumsum (fp32) per token and head
    assert wk["train_fwd_bytes"] - wk["fwd_only_bytes"] == tok * H * (64 * 2 + 4)
    assert round(wk["fwd_only_bytes"] / 1e6, 1) == 269.5
    assert round(wk["train_fwd_bytes"] / 1e6, 1) == 304.1
    assert round(wk["bwd_bytes"] / 1e6, 1) == 505.9
    assert wk["fwd_flops"] == tok * H * 180224
    assert wk["bwd_flops"] == tok * H * 376832


def test_states_enter_the_bytes():
    w = WORKLOADS["varlen"]          # initial and final states of 5 sequences
    wk = bench.work(w)
    st = 5 * 32 * 128 * 128 * 4
    assert wk["parts"]["state"] == st
    assert wk["bwd_bytes"] - bench.work(WORKLOADS["varlen"].__class__(**{**w.__dict__, "has_h0": False,
                                                                          "final_state": False}))["bwd_bytes"] == 3 * st


def test_direction_report():
    r = bench.direction_report(ms=0.5, flops=1e11, nbytes=3.4e9, tokens=8192, hbm=6800.0, tflops=1700.0)
    assert r["roofline_us"] == pytest.approx(max(3.4e9 / 6.8e12, 1e11 / 1.7e15) * 1e6, rel=1e-3)
    assert r["roofline_frac"] == pytest.approx(500.0 / 500.0, rel=1e-3)
    assert r["tokens_per_s"] == pytest.approx(8192 / 5e-4, rel=1e-6)
    assert "us_median" not in r
    m = bench.direction_report(ms=0.5, flops=1e11, nbytes=3.4e9, tokens=8192, hbm=6800.0, tflops=1700.0,
                               median_ms=0.45)
    assert m["us_median"] == 450.0 and m["us"] == 500.0 and m["roofline_frac"] == r["roofline_frac"]


def test_kernel_bytes_cover_only_the_kernel_io():
    w = WORKLOADS["dense"]
    wk = bench.work(w)
    assert bench.kernel_bytes("bwd_chunk", w, wk) == wk["bwd_bytes"]
    assert bench.kernel_bytes("wy_fwd", w, wk) < wk["train_fwd_bytes"]
    assert bench.kernel_bytes("no_such_kernel", w, wk) is None
