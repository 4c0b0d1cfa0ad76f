"""The FLOP accounting of the block metric (dit_inputs.BlockShape.flops: 2R(3H^2 + H^2 + 2HF + FH)
for the four linears plus 4R^2 H for the two attention products) checked against the figures the
klein page prints for its own workload (tests/golden/klein_flop_counts.txt): its attention FLOP
and time per call, its score-matrix size, its single-block linear1 shape (which fixes its MLP
width) and its whole-DiT FLOP per scan (100 block calls), which the blocks' FLOP must account for
up to the small layers outside the blocks."""

import os

import pytest

import dit_inputs as DI

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "klein_flop_counts.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def _klein_shape(g):
    R, H = int(g["rows"]), int(g["hidden"])
    # linear1 of the single-stream block is [qkv | gate/up]: N = 3H + 2F
    F = (int(g["linear1_n"]) - 3 * H) // 2
    # 512 text rows + a 64 x 64 image grid
    return DI.BlockShape("klein", H, int(g["heads"]), int(g["head_dim"]), F, R - 4096, 64, 64, seed=0)


def test_shape_figures_are_consistent():
    g = _golden()
    sh = _klein_shape(g)
    assert sh.R == g["rows"] == g["linear1_m"] and sh.hidden == g["linear1_k"]
    assert sh.heads * sh.head_dim == sh.hidden
    assert sh.ffn == 3 * sh.hidden  # the MLP width the linear1 shape implies
    # fp32 scores, one [R, R] matrix per head
    assert sh.heads * sh.R * sh.R * 4 == pytest.approx(g["score_bytes_per_call"], rel=5e-3)


def test_attention_flop_per_call():
    g = _golden()
    sh = _klein_shape(g)
    attn = sh.flops() - 2.0 * sh.R * (4 * sh.hidden ** 2 + 3 * sh.hidden * sh.ffn)
    assert attn == 4.0 * sh.R * sh.R * sh.hidden
    assert attn / 1e12 == pytest.approx(g["attention_tflop_per_call"], rel=1e-2)
    # and the page's time and rate for it agree with that count
    assert attn / (g["attention_ms_per_call"] * 1e-3) / 1e12 == pytest.approx(g["attention_tflops"], rel=5e-3)


def test_dit_flop_per_scan_is_the_blocks_plus_small_layers():
    g = _golden()
    sh = _klein_shape(g)
    blocks = g["attention_calls_per_image"] * sh.flops()
    # the blocks carry all but a fraction of a percent (time embedding, modulation projections,
    # patch in/out and final layer are thin GEMMs)
    assert blocks <= g["dit_flop_per_scan"]
    assert blocks / g["dit_flop_per_scan"] > 0.99
