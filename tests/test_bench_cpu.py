"""bench.py's work model (the numerators of every roofline it reports), checked
against the per-head-token counts written out by hand for the benchmark
workloads."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from kernelized_linear_attention_03_b300 import inputs  # noqa: E402

W = {w.name.split("_")[0]: w for w in inputs.WORKLOADS}


def test_forward_flops_per_head_token():
    # F = 4 n (dv+1) + (C+1)(p+dv): c4 n = 2080 -> 4*2080*65 + 129*128 = 557,312
    per_token = {"c1": 4 * 136 * 17 + 33 * 32, "c2": 4 * 528 * 65 + 65 * 96,
                 "c3": 4 * 2080 * 65 + 65 * 128, "c4": 557_312, "c5": 4 * 528 * 33 + 65 * 64}
    for key, f in per_token.items():
        w = W[key]
        assert bench.flops_forward(w) == w.B * w.H * w.T * f
    assert abs(bench.flops_forward(W["c4"]) / 1e9 - 584.4) < 0.1


def test_kernel_work_split_and_bytes():
    w = W["c4"]
    bht = w.B * w.H * w.T
    kind, tiles = bench.kernel_work("chunked_tc", w)
    assert kind == "flop" and tiles == bht * 4 * 2080 * 65
    kind, intra = bench.kernel_work("intra_tc", w)
    assert kind == "flop" and intra == bht * 129 * 128
    kind, scan = bench.kernel_work("scan_tree", w)
    assert kind == "byte" and scan == 2 * 8 * 1024 * 2080 * 65 * 4
    kind, states = bench.kernel_work("states_tc", w, "chunk_state_scan")
    assert kind == "byte" and states == 8 * 1024 * 2080 * 65 * 4 + bht * 128 * 2
    kind, quad = bench.kernel_work("quadratic_tc", W["c2"], "quadratic")
    assert kind == "flop" and quad == 2 * 8 * 2048 * 2049 * 96
    # the segment-state prepass of the forward does no algorithmic work of its own
    assert bench.kernel_work("states_tc", w) == ("flop", 0)
    # the gated form's chunk states are its own work; its decays one read and one write a token
    c3 = W["c3"]
    bht3 = c3.B * c3.H * c3.T
    assert bench.kernel_work("states_tc", c3, "gated") == ("flop", bht3 * 2 * 2080 * 65)
    assert bench.kernel_work("gate_decay", c3, "gated") == ("byte", bht3 * 8)


def test_block_lift_work_model():
    # KATA-Sigma-2 at p = 64: n = 528, m = 32, 4 block pairs per score; KATA-M-2: n = 1056, 2 pairs
    w = W["c4"]
    bht = w.B * w.H * w.T
    sig, mul = (bench.LIFTS["sigma"], 2), (bench.LIFTS["multi"], 2)
    assert bench.lift_dim(sig[0], 64, 2) == 528 and bench.lift_dim(mul[0], 64, 2) == 1056
    assert bench.kernel_work("block_states_simt", w, "chunked_block", sig) == ("flop", bht * 2 * 528 * 65)
    assert bench.kernel_work("block_output_simt", w, "chunked_block", sig) == (
        "flop", bht * (2 * 528 * 65 + 129 * (4 * 32 + 64)))
    assert bench.kernel_work("block_output_simt", w, "chunked_block", mul) == (
        "flop", bht * (2 * 1056 * 65 + 129 * (2 * 32 + 64)))
    assert bench.kernel_work("scan_tree", w, "chunked_block", sig) == ("byte", 2 * 8 * 1024 * 528 * 65 * 4)
    c2 = W["c2"]
    assert bench.kernel_work("block_quadratic_simt", c2, "quadratic_block", sig) == (
        "flop", 2 * 8 * 2048 * 2049 * (4 * 16 + 64))
