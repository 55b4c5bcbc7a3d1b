"""Host arithmetic of bench.py, checked without a GPU: the visible-pair
count behind the masked-FLOP metric against the oracle's band mask (brute
force), the per-head pair counts and FLOPs per step of the benchmark
configurations, the layer schedules, and the projection FLOPs of the block
workload against the list of GEMMs the block runs."""

import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("T,W", [(1, -1), (7, 0), (10, 3), (10, 9), (10, 40), (33, -1),
                                 (130, 64), (257, 128)])
def test_pairs_count_the_oracle_band(T, W):
    mask = oracle.band_mask(np.arange(T), T, W, True)
    assert bench.pairs(T, W) == int(mask.sum())


def test_pairs_and_flops_of_the_benchmark_configurations():
    # visible pairs per (b, h) head
    assert bench.pairs(256, 128) == 24_768
    assert bench.pairs(2048, 1024) == 1_574_400
    assert bench.pairs(2048, -1) == 2_098_176
    assert bench.pairs(16384, 8192) == 100_675_584
    assert bench.pairs(16384, -1) == 134_225_920
    # S layer: 4 d P B Hq forward, 10 d P B Hq backward
    fwd, bwd = bench.flops(16, 2048, 6, 128, 1024)
    assert fwd == 4 * 128 * 1_574_400 * 16 * 6 == 77_384_908_800
    assert bwd == 10 * 128 * 1_574_400 * 16 * 6
    # the 8-layer stack: 6 S layers and 2 L layers per step
    sched = bench.layer_schedule(oracle.sssl_window, oracle.has_ve)
    assert [w for w, _ in sched] == [1024, 1024, 1024, -1, 1024, 1024, 1024, -1]
    assert [ve for _, ve in sched] == [False, True, False, True, False, True, False, True]
    total = sum(sum(bench.flops(16, 2048, 6, 128, w)) for w, _ in sched)
    assert total == 2_346_989_912_064


def test_long_context_schedule_and_shape():
    assert bench.shape_for("long") == (2, 16384, 16, 4)
    assert bench.schedule_for("long", oracle.sssl_window, oracle.has_ve) == [(8192, False),
                                                                              (-1, False)]
    assert bench.shape_for("stack_mha") == (16, 2048, 6, 6)


def test_block_projection_flops_match_the_gemms_the_block_runs():
    rows, C, nq, nkv = 16 * 2048, 768, 6 * 128, 3 * 128
    # (m, n, k) of every GEMM of one layer, forward then backward
    gemms = [(rows, nq, C), (rows, nkv, C), (rows, nkv, C), (rows, C, nq),     # q, k, v, out
             (C, nq, rows), (rows, nq, C),                                     # dwo, dO
             (nq, C, rows), (nkv, C, rows), (nkv, C, rows),                    # dwq, dwk, dwv
             (rows, C, nq), (rows, C, nkv), (rows, C, nkv)]                    # dxn
    assert bench.block_gemm_flops(rows, C, nq, nkv) == sum(2 * m * n * k for m, n, k in gemms)


def test_tiny_workload_shape_schedule_and_flops():
    assert bench.shape_for("tiny") == (1, 256, 2, 1)
    assert bench.head_dim_for("tiny") == (64, None)
    assert bench.schedule_for("tiny", oracle.sssl_window, oracle.has_ve) == [(128, False)]
    fwd, bwd = bench.flops(1, 256, 2, 64, 128)
    assert (fwd, bwd) == (12_681_216, 31_703_040)


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference: the oracle timed on the host cores on a
    bounded sample, one JSON object with the keys the driver reads."""
    import argparse
    args = argparse.Namespace(steps=1, warmup=1, gpus=1, impl="reference", workload="stack")
    out = bench.run_reference(args, 0, 1)
    assert out["impl"] == "reference" and out["metric"] == bench.METRIC
    assert out["unit"] == "TFLOP/s" and out["higher_is_better"] is True and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"] == {"value": out["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
