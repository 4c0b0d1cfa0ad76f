"""Pins of the oracle's pieces: modulated norm, QK norm, rotary tables and rotation, attention."""

import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- modulated RMSNorm

def test_modnorm_unit_modulation_rms_closed_form():
    g = np.random.default_rng(0)
    x = g.standard_normal((5, 32)) * g.uniform(0.1, 3, size=(5, 1))
    eps = 0.5  # large so that a dropped eps fails
    y = O.modulated_rmsnorm(x, None, np.zeros_like(x), np.zeros_like(x), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), (1 + eps / ms) ** -0.5, rtol=1e-13)


def test_modnorm_constant_row():
    c = np.array([-2.0, 0.25, 3.0])
    x = np.repeat(c[:, None], 16, axis=1)
    eps = 0.1
    y = O.modulated_rmsnorm(x, None, 0 * x, 0 * x, eps)
    expect = np.sign(c) * (1 + eps / c ** 2) ** -0.5
    np.testing.assert_allclose(y, np.repeat(expect[:, None], 16, axis=1), rtol=1e-14)


def test_modnorm_scale_is_one_plus_scale_and_shift_adds():
    x = np.ones((1, 8))  # RMS 1, with eps = 0 the normalised row is exactly ones
    scale = np.full((1, 8), 0.25)
    shift = np.full((1, 8), -0.5)
    y = O.modulated_rmsnorm(x, None, shift, scale, 0.0)
    np.testing.assert_array_equal(y, np.full((1, 8), 1.25 - 0.5))


def test_modnorm_affine_weight():
    x = np.array([[3.0, -4.0]])  # mean(x^2) = 12.5
    w = np.array([2.0, 0.5])
    y = O.modulated_rmsnorm(x, w, np.zeros((1, 2)), np.zeros((1, 2)), 0.0)
    r = 1 / math.sqrt(12.5)
    np.testing.assert_allclose(y, [[3 * r * 2.0, -4 * r * 0.5]], rtol=1e-15)


def test_qk_norm_unit_rms_per_head():
    g = np.random.default_rng(1)
    t = g.standard_normal((7, 3, 16)) * 5
    y = O.qk_rmsnorm(t, None, 1e-12)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-10)


# ---------------------------------------------------------------- positions and tables

def _golden_grid():
    kv = {}
    for line in open(os.path.join(GOLDEN, "host_contract_grid.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        kv[k] = [int(s) for s in v]
    return kv


def test_positions_centred_grid_golden():
    kv = _golden_grid()
    h = kv["grid_h"][0]
    L = 5
    pos = O.positions(L, h, 3)
    img = pos[L:].reshape(h, 3, 3)
    assert list(img[:, 0, 1]) == kv["height_positions"]   # "for h = 16, rows go -8..7"
    assert np.all(img[:, :, 0] == L)                      # frame axis of image tokens is L
    assert list(img[0, :, 2]) == [-2, -1, 0]              # w = 3: x - (w - w//2) = x - 2
    for i in range(L):
        assert tuple(pos[i]) == (i, i, i)


def test_axis_tables_golden_layout():
    kv = _golden_grid()
    assert list(O.axis_widths(128)) == kv["axis_widths"]
    tabs = [O.rope_axis_table(w) for w in kv["axis_widths"]]
    for (c, s), cols in zip(tabs, kv["axis_columns"]):
        assert c.shape == (kv["table_rows"][0], cols) and s.shape == c.shape
    # axes 1 and 2 have the same width, so their tables are byte-identical
    assert tabs[1][0].tobytes() == tabs[2][0].tobytes() and tabs[1][1].tobytes() == tabs[2][1].tobytes()
    # row of position p is p + 1024: position 0 has angle 0
    first = kv["table_first_position"][0]
    assert np.all(tabs[0][0][0 - first] == 1.0) and np.all(tabs[0][1][0 - first] == 0.0)


def test_token_rows_are_axis_rows_concatenated():
    # cos[token] = axis0[f + 1024] ++ axis1[h + 1024] ++ axis2[w + 1024]   (host contract, section 4)
    L, h, w = 6, 4, 5
    pos = O.positions(L, h, w)
    cos, sin = O.rope_tables(pos, 128)
    tabs = [O.rope_axis_table(wd) for wd in O.axis_widths(128)]
    for r in [0, 3, L, L + 7, L + h * w - 1]:
        rc = np.concatenate([tabs[a][0][pos[r, a] + 1024] for a in range(3)])
        rs = np.concatenate([tabs[a][1][pos[r, a] + 1024] for a in range(3)])
        assert np.array_equal(cos[r], rc) and np.array_equal(sin[r], rs)


def test_tables_match_polar_construction():
    # The page's construction: torch.polar(1, outer(pos, 1 / 10000^(arange(0, d, 2) / d))) per axis,
    # here evaluated in float64 and rounded to float32 like the oracle's tables.
    L, h, w = 9, 6, 7
    pos = O.positions(L, h, w)
    cos, sin = O.rope_tables(pos, 128)
    parts = []
    for a, d in enumerate((16, 56, 56)):
        p = torch.tensor(pos[:, a], dtype=torch.float64)
        f = 1.0 / torch.pow(torch.tensor(10000.0, dtype=torch.float64),
                            torch.arange(0, d, 2, dtype=torch.float64) / d)
        parts.append(torch.polar(torch.ones(len(p), d // 2, dtype=torch.float64), torch.outer(p, f)))
    z = torch.cat(parts, dim=1)
    np.testing.assert_allclose(cos, z.real.float().numpy(), rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(sin, z.imag.float().numpy(), rtol=0, atol=1.2e-7)


def test_tables_head64_widths():
    assert O.axis_widths(64) == (8, 28, 28)
    cos, sin = O.rope_tables(O.positions(8, 8, 8), 64)
    assert cos.shape == (72, 32)


# ---------------------------------------------------------------- rotation

def test_rope_zero_angle_identity_bitwise():
    g = np.random.default_rng(2)
    t = g.standard_normal((4, 2, 8))
    y = O.rope_apply(t, np.ones((4, 4)), np.zeros((4, 4)))
    assert np.array_equal(y, t)


def test_rope_matches_complex_pairs():
    # adjacent pairs as complex numbers times e^{i angle} (torch.polar complex pairs)
    g = np.random.default_rng(3)
    t = g.standard_normal((5, 3, 8))
    ang = g.uniform(-7, 7, size=(5, 4))
    y = O.rope_apply(t, np.cos(ang), np.sin(ang))
    z = (t[..., 0::2] + 1j * t[..., 1::2]) * np.exp(1j * ang)[:, None, :]
    np.testing.assert_allclose(y[..., 0::2], z.real, atol=1e-14)
    np.testing.assert_allclose(y[..., 1::2], z.imag, atol=1e-14)


def test_rope_inverse_and_norm():
    g = np.random.default_rng(4)
    t = g.standard_normal((5, 2, 8))
    ang = g.uniform(-7, 7, size=(5, 4))
    y = O.rope_apply(t, np.cos(ang), np.sin(ang))
    back = O.rope_apply(y, np.cos(-ang), np.sin(-ang))
    np.testing.assert_allclose(back, t, atol=1e-14)
    np.testing.assert_allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2, t[..., 0::2] ** 2 + t[..., 1::2] ** 2, rtol=1e-13)


# ---------------------------------------------------------------- attention

def test_attention_q_zero_gives_mean_of_values():
    g = np.random.default_rng(5)
    R, nh, d = 6, 2, 4
    k, v = g.standard_normal((R, nh, d)), g.standard_normal((R, nh, d))
    o = O.attention(np.zeros((R, nh, d)), k, v).reshape(R, nh, d)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), (R, nh, d)), atol=1e-15)


def test_attention_rows_sum_to_one():
    # with every value row equal to ones, o = sum_j P_ij = 1
    g = np.random.default_rng(6)
    R, nh, d = 9, 3, 8
    q, k = 4 * g.standard_normal((R, nh, d)), 4 * g.standard_normal((R, nh, d))
    o = O.attention(q, k, np.ones((R, nh, d)))
    np.testing.assert_allclose(o, 1.0, rtol=1e-14)


def test_attention_dominant_key():
    R, nh, d = 5, 1, 4
    q = np.zeros((R, nh, d))
    q[:, 0, 0] = 1.0
    k = np.zeros((R, nh, d))
    k[3, 0, 0] = 60.0 * math.sqrt(d)  # score 60 above the others
    v = np.arange(R * d, dtype=float).reshape(R, nh, d)
    o = O.attention(q, k, v).reshape(R, nh, d)
    np.testing.assert_allclose(o, np.broadcast_to(v[3], (R, nh, d)), rtol=1e-12)


def test_attention_brute_force_loops():
    g = np.random.default_rng(7)
    R, nh, d = 5, 2, 4
    q, k, v = (g.standard_normal((R, nh, d)) for _ in range(3))
    o = O.attention(q, k, v)
    for r in range(R):
        for n in range(nh):
            sc = [sum(q[r, n, j] * k[c, n, j] for j in range(d)) / math.sqrt(d) for c in range(R)]
            e = [math.exp(s) for s in sc]
            for j in range(d):
                ref = sum(e[c] * v[c, n, j] for c in range(R)) / sum(e)
                assert abs(o[r, n * d + j] - ref) < 1e-13


def test_attention_row_subset():
    g = np.random.default_rng(8)
    q, k, v = (g.standard_normal((7, 2, 4)) for _ in range(3))
    full = O.attention(q, k, v)
    np.testing.assert_array_equal(O.attention(q, k, v, rows=np.array([6, 1])), full[[6, 1]])
