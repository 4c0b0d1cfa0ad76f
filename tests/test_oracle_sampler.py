"""Pins of the oracle's int8lin dequantisation, Euler step, sigma grid, sinusoids, packing and denoise."""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import dit_inputs as DI
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- int8lin

def _bf16_rne_fraction(v: Fraction) -> Fraction:
    """Round an exact rational to the nearest bfloat16 (8 significant bits), ties to even."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    n = a / ulp
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * lo * ulp


def test_bf16_rne_matches_exact_rational_rounding():
    g = np.random.default_rng(0)
    x = (g.standard_normal(4000) * np.exp(g.uniform(-20, 20, 4000))).astype(np.float32)
    # include exact ties: 8 significant bits plus a half ulp
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(3 + 2 ** -6), 2 ** -20 * (1 + 2 ** -8)], np.float32)
    x = np.concatenate([x, ties])
    got = O.bf16_to_f64(O.bf16_rne_bits(x))
    for xi, gi in zip(x, got):
        assert Fraction(float(gi)) == _bf16_rne_fraction(Fraction(float(xi)))


def test_dequant_definition_and_block_index():
    g = np.random.default_rng(1)
    q = g.integers(-127, 128, size=(3, 96), dtype=np.int8)
    s = DI.bf16_bits_from_f32(g.uniform(0.001, 0.01, size=(3, 3)).astype(np.float32))
    W = O.bf16_to_f64(O.dequant_int8(q, s))
    sv = O.bf16_to_f64(s)
    for o in range(3):
        for i in range(96):
            exact = Fraction(int(q[o, i])) * Fraction(float(sv[o, i // 32]))
            assert Fraction(float(W[o, i])) == _bf16_rne_fraction(exact)


def test_dequant_exact_for_power_of_two_scales():
    q = np.arange(-127, 128, dtype=np.int8).reshape(1, -1)[:, :224]
    s = DI.bf16_bits_from_f32(np.full((1, 7), 2.0 ** -9, np.float32))
    W = O.bf16_to_f64(O.dequant_int8(q, s))
    np.testing.assert_array_equal(W, q.astype(np.float64) * 2.0 ** -9)


def test_dequant_round_trip():
    # |W - q s| <= half a bf16 ulp of 127 s < s / 2, so round(W / s) recovers q exactly
    g = np.random.default_rng(2)
    q = g.integers(-127, 128, size=(16, 256), dtype=np.int8)
    s = DI.bf16_bits_from_f32((DI.INT8_S0 * (0.75 + 0.5 * g.random((16, 8)))).astype(np.float32))
    W = O.bf16_to_f64(O.dequant_int8(q, s))
    back = np.rint(W / np.repeat(O.bf16_to_f64(s), 32, axis=1))
    np.testing.assert_array_equal(back, q.astype(np.float64))


def test_absmax_quantisation_error_bound():
    # the klein article's int8 round-trip figure: relative error up to 0.5/127 of the block absmax
    g = np.random.default_rng(3)
    w = g.standard_normal((8, 128))
    amax = np.abs(w.reshape(8, 4, 32)).max(axis=2)
    s = DI.bf16_bits_from_f32((amax / 127).astype(np.float32))
    sv = O.bf16_to_f64(s)
    q = np.clip(np.rint(w / np.repeat(sv, 32, axis=1)), -127, 127).astype(np.int8)
    W = O.bf16_to_f64(O.dequant_int8(q, s))
    err = np.abs(W - w).reshape(8, 4, 32).max(axis=2) / amax
    assert np.all(err <= 0.5 / 127 * 1.02 + 2 ** -8)


# ---------------------------------------------------------------- Euler step and sigmas

def _golden_sigmas():
    vals = [float(l) for l in open(os.path.join(GOLDEN, "host_contract_sigmas.txt"))
            if l.strip() and not l.startswith("#")]
    return np.array(vals, dtype=np.float32)


def test_sigma_grid_golden_claims():
    s = _golden_sigmas()
    assert len(s) == 8
    # shift 1.0: unchanged bit for bit
    assert np.array_equal(O.shift_sigmas(s, 1.0).view(np.uint32), s.view(np.uint32))
    # t = timesteps[i] / 1000 equals sigma[i] bit for bit
    t = ((s * np.float32(1000)).astype(np.float32) / np.float32(1000)).astype(np.float32)
    assert np.array_equal(t.view(np.uint32), s.view(np.uint32))
    # a shift above 1 moves every sigma except the end point 1.0 upward
    s3 = O.shift_sigmas(s, 3.0)
    assert s3[0] == 1.0 and np.all(s3[1:] > s[1:])


def test_euler_is_float32_separately_rounded():
    g = np.random.default_rng(4)
    s = np.append(_golden_sigmas(), np.float32(0))
    x = g.standard_normal(20000).astype(np.float32)
    v = g.standard_normal(20000).astype(np.float32)
    differs_from_fma = False
    for i in range(8):
        got = O.euler_step(x, v, s[i], s[i + 1])
        dt = np.float32(np.float64(s[i + 1]) - np.float64(s[i]))   # exact difference, one rounding
        prod = np.float32(np.float64(dt) * v.astype(np.float64))   # exact product, one rounding
        ref = (x.astype(np.float64) + prod.astype(np.float64)).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        fused = (x.astype(np.float64) + np.float64(dt) * v.astype(np.float64)).astype(np.float32)
        differs_from_fma |= not np.array_equal(fused, ref)
        x = got
    assert differs_from_fma  # the check above separates the two roundings


def test_euler_constant_velocity_closed_form():
    s = np.array([1.0, 0.75, 0.5, 0.25, 0.0], np.float32)
    assert float(np.sum(np.diff(s.astype(np.float64)))) == -1.0
    x = (np.arange(-64, 64) / 8.0).astype(np.float32)   # dyadic values: every step exact
    v = (np.arange(128) / 16.0 - 3).astype(np.float32)
    x0 = x.copy()
    for i in range(4):
        x0 = O.euler_step(x0, v, s[i], s[i + 1])
    np.testing.assert_array_equal(x0, x - v)


def test_euler_tiny_velocity_vanishes_in_float32():
    x = np.ones(1, np.float32)
    v = np.array([2.0 ** -25], np.float32)
    assert O.euler_step(x, v, 1.0, 0.75)[0] == 1.0   # 1 - 2^-27 rounds back to 1 in float32


# ---------------------------------------------------------------- sinusoids, packing

def test_sinusoids_t0_and_order():
    e = O.timestep_sinusoids([0.0], 256)
    assert np.all(e[0, :128] == 1.0) and np.all(e[0, 128:] == 0.0)   # [cos | sin]
    t = 0.001  # 1000 t = 1
    e = O.timestep_sinusoids([t], 256)[0]
    assert abs(e[0] - math.cos(1.0)) < 1e-15 and abs(e[128] - math.sin(1.0)) < 1e-15
    assert abs(e[64] - math.cos(10000 ** -0.5)) < 1e-15               # frequency 10000^(-64/128)
    assert abs(e[127 + 128] - math.sin(10000 ** (-127 / 128))) < 1e-15


def test_pack_latents_matches_view_transpose():
    g = np.random.default_rng(5)
    z = g.standard_normal((64, 3, 5)).astype(np.float32)
    x = O.pack_latents(z)
    # x = z.view(1, 64, h*w).transpose(1, 2)   (host contract, section 5)
    np.testing.assert_array_equal(x, z.reshape(64, 15).T)
    assert x[1 * 5 + 2, 7] == z[7, 1, 2]


# ---------------------------------------------------------------- denoise loop

def _small_denoise(blocks=2):
    sh = DI.BlockShape("t", 64, 2, 32, 96, 4, 2, 3, seed=11)
    return DI.denoise_inputs(sh, blocks=blocks, latent_channels=8)


def test_denoise_zero_projection_keeps_noise_bitwise():
    inp = _small_denoise()
    inp.w_out[:] = 0
    x = O.denoise(inp)
    assert np.array_equal(x, inp.latents)


def test_denoise_zero_gates_reduce_to_patch_path():
    # zero gate rows in every block's modulation weights: blocks are the identity, so each step's
    # velocity is the final modulated norm of the patched-in image rows, projected out.
    inp = _small_denoise()
    H = inp.shape.hidden
    for b in range(inp.blocks):
        inp.w_ada[b][2 * H:3 * H] = 0
        inp.w_ada[b][5 * H:6 * H] = 0
    trace = []
    x = O.denoise(inp, trace=trace)
    xr = inp.latents.copy()
    s = inp.steps_sigmas
    for i in range(4):
        e = np.array([[math.cos(1000 * float(s[i]) * 10000 ** (-k / 128)) for k in range(128)] +
                      [math.sin(1000 * float(s[i]) * 10000 ** (-k / 128)) for k in range(128)]])
        h = e @ O.bf16_to_f64(inp.w_t1).T
        temb = (h / (1 + np.exp(-h))) @ O.bf16_to_f64(inp.w_t2).T
        st = temb / (1 + np.exp(-temb))
        fin = (O.bf16_to_f64(inp.w_ada_f) @ st[0])
        X = xr.astype(np.float64) @ O.bf16_to_f64(inp.w_in).T
        ms = np.mean(X * X, axis=1, keepdims=True)
        hn = X / np.sqrt(ms + 1e-6) * (1 + fin[H:]) + fin[:H]
        vel = hn @ O.bf16_to_f64(inp.w_out).T
        np.testing.assert_allclose(trace[i], vel, rtol=1e-12, atol=1e-12)
        xr = O.euler_step(xr, vel.astype(np.float32), s[i], s[i + 1])
    assert np.array_equal(x, xr)


def test_denoise_blocks_match_block_oracle_composition():
    inp = _small_denoise(blocks=2)
    trace = []
    O.denoise(inp, steps=1, trace=trace)
    sh = inp.shape
    H, L = sh.hidden, sh.L
    t = float(inp.steps_sigmas[0])
    st = O.silu(O.time_embedding([t], inp.w_t1, inp.w_t2)[0])
    rows = np.concatenate([inp.txt_feats, inp.latents.astype(np.float64) @ O.bf16_to_f64(inp.w_in).T])
    cos, sin = O.rope_tables(O.positions(L, sh.grid_h, sh.grid_w), sh.head_dim)
    for b in range(2):
        mod = (O.bf16_to_f64(inp.w_ada[b]) @ st).reshape(1, 6, H)
        rows = O.block_forward_rows(rows, O.block_weights_f64(inp.block_w[b]), mod,
                                    np.zeros(len(rows), np.int32), cos, sin, sh.heads, sh.head_dim)
    fin = O.bf16_to_f64(inp.w_ada_f) @ st
    vel = O.modulated_rmsnorm(rows[L:], None, fin[:H], fin[H:], 1e-6) @ O.bf16_to_f64(inp.w_out).T
    np.testing.assert_array_equal(trace[0], vel)
