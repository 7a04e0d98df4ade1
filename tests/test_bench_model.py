"""The measurement model of bench.py, on CPU: the algorithmic bytes and flops the roofline
fractions divide by, checked against values worked out by hand from the workloads' shapes (an
accidental change to the model would otherwise move every reported fraction silently)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from linear_latent_routing_gb300 import inputs as W  # noqa: E402


def test_path_bytes_by_hand():
    # benchmark workload: 16 heads x 65536 tokens, bf16, Q_X and K_X (64 wide), V and O (128 wide)
    assert W.LONG_CAUSAL.token_heads == 1_048_576
    assert bench.path_bytes(W.LONG_CAUSAL) == 1_048_576 * 2 * (64 + 64 + 128 + 128)
    # classification-shaped workload: 256 slices x 4096 tokens, d_r = 32, d_v = 64
    assert bench.path_bytes(W.LRA_BIDIR) == 1_048_576 * 2 * (32 + 32 + 64 + 64)
    # fp32 inputs count four bytes an element
    w = W.TINY_BIDIR_F32
    assert bench.path_bytes(w) == w.B * w.H * w.N * 4 * (2 * w.d_r + 2 * w.d_v)


def test_path_flops_by_hand():
    # per token-head: the [x^2, x] logits on both sides (2 x 2 d_r K multiply-adds) and the write
    # and read contractions with the normaliser (2 x K (d_v + 1) multiply-adds), two flops each
    w = W.K_SWEEP[2]   # K = 256, B = 2, H = 16, N = 16384
    per = 2 * (2 * 2 * 64 * 256) + 2 * (2 * 256 * 129)
    assert bench.path_flops(w) == w.B * w.H * w.N * per
    assert bench.path_flops(w) == 137_975_824_384


def test_roofline_step_of_the_benchmark():
    # 805 MB at the measured copy bandwidth, against 72 us of bf16 tensor time: HBM-bound
    pk = {"hbm_gbs": 6784.5, "bf16_tflops": 1927.9}
    w = W.LONG_CAUSAL
    t_mem = bench.path_bytes(w) / (pk["hbm_gbs"] * 1e9)
    t_mma = bench.path_flops(w) / (pk["bf16_tflops"] * 1e12)
    assert abs(t_mem * 1e6 - 118.70) < 0.01
    assert t_mma < t_mem


def test_output_pass_bytes():
    # the causal output pass is credited Q_X + V + O only (its stored Gamma_K is not algorithmic)
    bound, amount, unit = bench.kernel_work(W.LONG_CAUSAL, "tc_causal_chunked")
    assert (bound, unit) == ("hbm", "GB/s")
    assert amount == 1_048_576 * 2 * (64 + 2 * 128)
