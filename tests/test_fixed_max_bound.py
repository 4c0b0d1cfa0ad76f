"""The bound behind the attention's fixed-maximum softmax, checked on the CPU.

For rows that the QKV epilogue has QK-normed (per head x_j / sqrt(mean(x^2) + eps) * w_j, then
rotated and rounded to bf16), every scaled score s = q . k * log2(e) / sqrt(d) satisfies
|s| <= B = (1 + 2^-6)^2 d max|w_q| max|w_k| log2(e) / sqrt(d): the normed vector has Euclidean norm
at most sqrt(d) max|w| (the eps only shrinks it), a rotation keeps the norm, and bf16 rounding
grows each element by at most 2^-8 relative. With B < 60 the softmax can subtract B instead of a
running row maximum: every exponent s - B lies in [-2B, 0], so every weight exp2(s - B) is a normal
fp32 (and bf16) number no larger than 1, and no row sum can vanish or overflow. The attention
kernels take that path exactly when B < 60 (unit norm weights: B = 16.8 at d = 128)."""

import math

import numpy as np
import pytest

import oracle as O

LOG2E = 1.0 / math.log(2.0)


def _bound(d, mq, mk):
    return (1 + 2 ** -6) ** 2 * d * mq * mk * LOG2E / math.sqrt(d)


def _bf16(x):
    return O.bf16_to_f64(O.bf16_rne_bits(np.asarray(x, np.float32)))


def _qk_rows(x, w, ang, eps=1e-6):
    # per-head RMS norm with weight, adjacent-pair rotation, bf16 rounding (the epilogue's steps)
    x = np.asarray(x, np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w
    a, b = y[..., 0::2], y[..., 1::2]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(y)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return _bf16(out)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("wscale", [1.0, 1.02, 1.5])
def test_scores_stay_within_the_bound(d, wscale):
    g = np.random.default_rng(d + int(wscale * 100))
    wq = wscale * (1 + 0.02 * g.standard_normal(d))
    wk = wscale * (1 + 0.02 * g.standard_normal(d))
    B = _bound(d, np.abs(wq).max(), np.abs(wk).max())
    n = 512
    # random rows, and the worst case: all of a row's mass on one component, q and k aligned
    xq = g.standard_normal((n, d))
    xk = g.standard_normal((n, d))
    j = np.argmax(np.abs(wq) * np.abs(wk))
    xq[:8] = 0.0
    xk[:8] = 0.0
    xq[:8, j] = g.uniform(0.5, 3.0, 8)
    xk[:8, j] = g.uniform(0.5, 3.0, 8)
    ang = np.zeros((n, d // 2))
    ang[8:] = g.uniform(-math.pi, math.pi, (n - 8, d // 2))
    q, k = _qk_rows(xq, wq, ang), _qk_rows(xk, wk, ang)
    s = (q @ k.T) * LOG2E / math.sqrt(d)
    assert np.abs(s).max() <= B
    # the aligned rows reach d |w_q[j] w_k[j]| (in log2 units): the bound is tight up to its margin
    assert np.abs(s).max() >= 0.99 * d * abs(wq[j] * wk[j]) * LOG2E / math.sqrt(d)


def test_unit_weights_take_the_fixed_path_and_weights_stay_normal():
    for d in (64, 128):
        B = _bound(d, 1.0, 1.0)
        assert B < 60
        # the smallest weight exp2(-2B) is a normal fp32 value
        assert 2.0 ** (-2 * B) > np.finfo(np.float32).tiny
    assert _bound(128, 1.0, 1.0) == pytest.approx(16.84, abs=0.01)
    assert _bound(64, 1.0, 1.0) == pytest.approx(11.91, abs=0.01)
    # large norm weights leave the fixed path (running maximum instead)
    assert _bound(128, 2.0, 2.0) > 60
