"""Host logic of bench.py (no GPU): the byte counts behind the headline, the
job value's weak scaling, the bootstrap interval, and the committed DRAM
traffic record that the bench reports beside its roofline figure."""
import json
import os

import numpy as np

import bench
import s3d8_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_bytes_match_the_pages_bits_per_parameter():
    """One byte per 3 weights at one input column, a bf16 scale per output
    channel and a 96-byte table per matrix: 2.68 bits per parameter for the whole
    model in the format-comparison table of the blog "11 billion parameters on a
    phone" (section "Additional QAT results"); the
    11B layer's seven matrices come to 8/3 bits plus the scale overhead, 16 bits
    per output channel over K columns, plus one zero-scale padding row per matrix
    whose N is not a multiple of 3."""
    params = sum(K * N for _, K, N in si.LLAMA_11B_LAYER)
    bpp = bench.LAYER_WEIGHT_BYTES * 8 / params
    assert 8 / 3 < bpp < 2.69
    overhead = sum(16 * N + 8 * 96 for _, K, N in si.LLAMA_11B_LAYER) / params
    padding = sum(8 * K * (si.groups(N) * 3 - N) / 3 for _, K, N in si.LLAMA_11B_LAYER) / params
    assert abs(bpp - (8 / 3 + overhead + padding)) < 1e-9
    assert bench.LAYER_WEIGHT_BYTES == bench.CONFIG["weight_bytes_per_step"] == 72_811_168


def test_group_bytes_read_each_activation_once():
    """The grouped launch reads each of the four distinct bf16 activations once
    (q, k and v share one; gate and up share one) and writes every output."""
    names = [n for n, _, _ in si.LLAMA_11B_LAYER]
    shapes = {n: (K, N) for n, K, N in si.LLAMA_11B_LAYER}
    outputs = sum(2 * N for _, N in shapes.values())
    acts = sum(2 * K + 4 for K in bench.ACT_K.values())
    assert len({si.LLAMA_11B_INPUT_OF[n] for n in names}) == 4
    assert bench.group_bytes(names) == bench.LAYER_WEIGHT_BYTES + outputs + acts
    assert bench.linear_bytes(1, 4096, 14336) == bench.weight_bytes(4096, 14336) + 4096 + 4 + 2 * 14336


def test_job_value_scales_weakly_with_ranks():
    one = bench.job_value(1, 0.02)
    assert abs(one - bench.LAYER_WEIGHT_BYTES / 20e-6 / 1e9) < 1e-6
    assert abs(bench.job_value(4, 0.02) - 4 * one) < 1e-6


def test_bootstrap_interval_brackets_the_median():
    rng = np.random.default_rng(3)
    samples = 0.0196 + 0.0002 * rng.standard_normal(60)
    r = bench.bootstrap_median(samples)
    lo, hi = r["ci95_ms_per_step"]
    assert r["samples"] == 60
    assert lo <= r["median_ms_per_step"] <= hi
    assert hi - lo < 0.001


def test_committed_dram_traffic_matches_the_gemv_source():
    """The ncu record of the headline kernel's DRAM bytes belongs to the current
    GEMV source (the bench prints null otherwise), and the bytes it counts are
    within 0.1% of the launch's algorithmic bytes: each packed byte read once."""
    with open(os.path.join(ROOT, "profiles", "gemv_traffic.json")) as f:
        rec = json.load(f)
    assert rec["source_sha"] == bench.gemv_source_sha()
    traffic = bench.traffic_per_launch()
    assert traffic == rec["dram_bytes_per_launch"]
    names = [n for n, _, _ in si.LLAMA_11B_LAYER]
    algorithmic = bench.group_bytes(names)
    assert rec["algorithmic_bytes_per_launch"] == algorithmic
    assert 1.0 <= traffic / algorithmic < 1.001
