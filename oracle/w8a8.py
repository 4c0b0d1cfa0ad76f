"""W8A8 linears: per-token int8 activations times per-output-channel int8 weights, with the optional
SmoothQuant fold, and the block forward whose four linears take that form (test oracle).

Source: [klein] "944 -> 346 ms: optimizing FLUX.2 klein-4B on one TPU v6e chip", section 5 (int8
detail) and its D4 / D5 log entries: an int8 weight holds int8 values and one float32 scale per
output channel (symmetric absmax / 127, per output channel, at load time); activations are
quantised per token on every call (dynamic absmax / 127 per row); the linear is an int8 x int8 ->
int32 dot product, a float32 dequantisation and one cast to the activation's dtype. SmoothQuant
divides the activation by a per-input-channel divisor before its quantisation and folds the same
divisor into the weight (diag(s) W in float32) before the weight's quantisation; the divisor comes
from calibration statistics through a smoothing formula with exponent alpha.

Readings where the pages are silent (the pages give the scheme, not these details):
* the scale is absmax / 127 in float32; a code is clip(rint(v / scale), -127, 127) with the float32
  division and round-half-to-even (the rounding of jnp.round); a row or channel of zeros has scale
  0 and codes 0;
* the smoothing formula is SmoothQuant's s_j = max|X_j|^alpha / max|W_j|^(1 - alpha); a channel
  whose statistics are zero gets s_j = 1;
* the activation entering a W8A8 linear is its bfloat16 value (the pages' activations are bf16);
* the dequantised output is the exact integer dot product times both scales, formed in float64 here
  (float32 on the pages and the GPU: the comparison allows float32 rounding).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from .dit import (attention, bf16_rne_bits, bf16_to_f64, modulated_layernorm, modulated_rmsnorm, qk_rmsnorm,
                  rotate, swiglu_interleaved, _mod_rows)

__all__ = ["quantize_codes", "quantize_rows", "quantize_weight", "smooth_scales", "w8a8_linear",
           "w8a8_linear_f", "block_forward_w8a8_rows", "parallel_block_forward_w8a8_rows",
           "double_block_forward_w8a8_rows"]


def quantize_codes(v32: np.ndarray, scale32: np.ndarray) -> np.ndarray:
    """int8 codes clip(rint(v / scale), -127, 127) of float32 values v with float32 scales broadcast
    along the last axis's rows (scale 0: code 0). The division is the float32 one."""
    v = np.asarray(v32, dtype=np.float32)
    s = np.asarray(scale32, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(v / s)  # float32 division, round half to even
    r = np.where(s == 0, np.float32(0), r)
    return np.clip(r, -127, 127).astype(np.int8)


def quantize_rows(x32: np.ndarray, smooth: Optional[np.ndarray] = None):
    """Per-token quantisation of activations x [R, K] (float32 values), after the division by the
    SmoothQuant divisor when given: returns (codes int8 [R, K], scale float32 [R]),
    scale = max_j |x_j / s_j| / 127.  [klein, D4 quantize_rows; D5 quantize_rows(x / smooth)]"""
    x = np.asarray(x32, dtype=np.float32)
    if smooth is not None:
        x = (x / np.asarray(smooth, dtype=np.float32)[None, :]).astype(np.float32)
    amax = np.max(np.abs(x), axis=1).astype(np.float32)
    scale = (amax / np.float32(127)).astype(np.float32)
    return quantize_codes(x, scale[:, None]), scale


def quantize_weight(w32: np.ndarray, smooth: Optional[np.ndarray] = None):
    """Per-output-channel quantisation of a weight W [N, K] (float32 values; rows are output
    channels), after folding the SmoothQuant divisor into its input channels, W'[o, j] =
    float32(W[o, j] s_j): returns (codes int8 [N, K], scale float32 [N]).
    [klein, D4 quantize_weight; D5 quantize_weight_smooth]"""
    w = np.asarray(w32, dtype=np.float32)
    if smooth is not None:
        w = (w * np.asarray(smooth, dtype=np.float32)[None, :]).astype(np.float32)
    amax = np.max(np.abs(w), axis=1).astype(np.float32)
    scale = (amax / np.float32(127)).astype(np.float32)
    return quantize_codes(w, scale[:, None]), scale


def smooth_scales(x_absmax: np.ndarray, w_absmax: np.ndarray, alpha: float) -> np.ndarray:
    """SmoothQuant divisors s_j = max|X_j|^alpha / max|W_j|^(1 - alpha) from per-input-channel
    statistics of the activation (calibration) and of the weight; 1 where either is zero. Float32.
    [klein, D5 smooth_scales]"""
    xa = np.asarray(x_absmax, dtype=np.float64)
    wa = np.asarray(w_absmax, dtype=np.float64)
    ok = (xa > 0) & (wa > 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(ok, xa ** alpha / wa ** (1.0 - alpha), 1.0)
    return s.astype(np.float32)


def w8a8_linear(qx: np.ndarray, sx: np.ndarray, qw: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """out[r, o] = (sum_j qx[r, j] qw[o, j]) sx[r] sw[o]: the exact integer dot product (int64),
    then both scales (float64).  [klein, D4 linear_int8]"""
    acc = np.asarray(qx, dtype=np.int64) @ np.asarray(qw, dtype=np.int64).T
    return acc.astype(np.float64) * np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :]


def w8a8_linear_f(x: np.ndarray, qw: np.ndarray, sw: np.ndarray, smooth: Optional[np.ndarray] = None) -> np.ndarray:
    """The W8A8 linear of an activation x (any float values): x is taken at its bfloat16 value,
    quantised per token (after the smoothing division) and multiplied with the quantised weight."""
    xb = bf16_to_f64(bf16_rne_bits(np.asarray(x, dtype=np.float64).astype(np.float32))).astype(np.float32)
    qx, sx = quantize_rows(xb, smooth)
    return w8a8_linear(qx, sx, qw, sw)


def block_forward_w8a8_rows(x, qweights, mod, mod_map, cos, sin, heads, head_dim,
                            rows: Optional[np.ndarray] = None, norm1=None, norm2=None,
                            q_norm=None, k_norm=None, eps=1e-6, qk_eps=1e-6, smooth=None):
    """The AdaLN block (see oracle.dit.block_forward_rows for its nine steps) with its four linears
    (qkv, out, up, down) in W8A8 form. qweights: four (codes int8 [out, in], scale float32 [out])
    pairs, quantised with the same ``smooth`` divisors (four [in] arrays or None). Each linear's
    activation (h, o, h2, a) enters at its bfloat16 value and is quantised per token.
    Float64 otherwise; rows as in block_forward_rows."""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    sm = smooth if smooth is not None else (None, None, None, None)
    lin = lambda i, a: w8a8_linear_f(a, qweights[i][0], qweights[i][1], sm[i])
    all_rows = np.arange(R)
    rows = all_rows if rows is None else np.asarray(rows)
    sa, ca, _, _, _, _ = _mod_rows(mod, mod_map, all_rows)
    h = modulated_rmsnorm(x, norm1, sa, ca, eps)
    qkv = lin(0, h)
    q = qkv[:, 0:H].reshape(R, nh, d)
    k = qkv[:, H:2 * H].reshape(R, nh, d)
    v = qkv[:, 2 * H:3 * H].reshape(R, nh, d)
    q = rotate(qk_rmsnorm(q, q_norm, qk_eps), cos, sin)
    k = rotate(qk_rmsnorm(k, k_norm, qk_eps), cos, sin)
    o = attention(q, k, v, rows)
    _, _, ga_r, sm_r, cm_r, gm_r = _mod_rows(mod, mod_map, rows)
    xr = x[rows] + ga_r * lin(1, o)
    h2 = modulated_rmsnorm(xr, norm2, sm_r, cm_r, eps)
    a = swiglu_interleaved(lin(2, h2))
    return xr + gm_r * lin(3, a)


def parallel_block_forward_w8a8_rows(x, linear1, linear2, mod, mod_map, cos, sin, heads, head_dim,
                                     rows: Optional[np.ndarray] = None, norm=None, q_norm=None, k_norm=None,
                                     eps=1e-6, qk_eps=1e-6, smooth1=None, smooth2=None):
    """The parallel block (see oracle.dit.parallel_block_forward_rows) with its two linears in W8A8
    form, as the klein article quantises a single block: linear1 = [Wqkv ; Wup] ([3H + 2F, H], rows
    Q|K|V then gate/up interleaved) over the normed rows h, and linear2 = [Wout | Wdown] ([H, H + F])
    over the joined row [o | a] of the attention output and the SwiGLU output, each an (int8 codes,
    float32 per-output-channel scales) pair quantised over its whole row (smooth1 [H] and smooth2
    [H + F] the SmoothQuant divisors used for it, or None). Each activation (h, then [o | a]) enters
    at its bfloat16 value and is quantised per token over its whole row.
    [klein, section 5 (int8 detail: single linear1 and linear2) and its D4 / D5 entries]"""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    rows = np.arange(R) if rows is None else np.asarray(rows)
    m = np.asarray(mod, dtype=np.float64)[np.asarray(mod_map)]
    h = modulated_layernorm(x, norm, m[:, 0], m[:, 1], eps)
    # linear1's output channels split at 3H (each channel's codes and scale are its own row, and each
    # row of h has its own codes): the Q|K|V part for every row, the gate/up part for `rows` only
    q1, s1 = np.asarray(linear1[0]), np.asarray(linear1[1])
    u = w8a8_linear_f(h, q1[:3 * H], s1[:3 * H], smooth1)
    q = rotate(qk_rmsnorm(u[:, 0:H].reshape(R, nh, d), q_norm, qk_eps), cos, sin)
    k = rotate(qk_rmsnorm(u[:, H:2 * H].reshape(R, nh, d), k_norm, qk_eps), cos, sin)
    v = u[:, 2 * H:3 * H].reshape(R, nh, d)
    o = attention(q, k, v, rows)
    a = swiglu_interleaved(w8a8_linear_f(h[rows], q1[3 * H:], s1[3 * H:], smooth1))
    y = w8a8_linear_f(np.concatenate([o, a], axis=1), linear2[0], linear2[1], smooth2)
    return x[rows] + m[rows, 2] * y


def double_block_forward_w8a8_rows(x, qweights_txt, qweights_img, mod, mod_map, cos, sin, heads, head_dim, L,
                                   rows: Optional[np.ndarray] = None, norms_txt=(None, None, None, None),
                                   norms_img=(None, None, None, None), eps=1e-6, qk_eps=1e-6, smooth_txt=None,
                                   smooth_img=None):
    """The double-stream block (see oracle.dit.double_block_forward_rows) with each stream's four
    linears in W8A8 form: qweights_* are four (codes, scales) pairs (qkv, out, up, down) quantised
    with that stream's SmoothQuant divisors smooth_* (four [in] arrays or None), as the klein article
    quantises a double block's image and text qkv, proj, mlp.0 and mlp.2 linears. Each activation
    enters at its bfloat16 value and is quantised per token with its own stream's divisors.
    [klein, section 5 (int8 detail) and its D4 / D5 entries; klein, sections 4.3-4.4 (double blocks)]"""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    rows = np.arange(R) if rows is None else np.asarray(rows)
    m = np.asarray(mod, dtype=np.float64)[np.asarray(mod_map)]
    streams = [(np.arange(0, L), qweights_txt, norms_txt, smooth_txt),
               (np.arange(L, R), qweights_img, norms_img, smooth_img)]
    q = np.empty((R, nh, d))
    k = np.empty((R, nh, d))
    v = np.empty((R, nh, d))
    for idx, qw, nrm, sm in streams:
        if len(idx) == 0:
            continue
        sm = sm if sm is not None else (None, None, None, None)
        h = modulated_rmsnorm(x[idx], nrm[0], m[idx, 0], m[idx, 1], eps)
        u = w8a8_linear_f(h, qw[0][0], qw[0][1], sm[0])
        n = len(idx)
        q[idx] = rotate(qk_rmsnorm(u[:, 0:H].reshape(n, nh, d), nrm[2], qk_eps), cos[idx], sin[idx])
        k[idx] = rotate(qk_rmsnorm(u[:, H:2 * H].reshape(n, nh, d), nrm[3], qk_eps), cos[idx], sin[idx])
        v[idx] = u[:, 2 * H:3 * H].reshape(n, nh, d)
    o = attention(q, k, v, rows)
    out = np.empty((len(rows), H))
    for idx, qw, nrm, sm in streams:
        sel = np.nonzero(np.isin(rows, idx))[0]
        if len(sel) == 0:
            continue
        sm = sm if sm is not None else (None, None, None, None)
        r = rows[sel]
        xr = x[r] + m[r, 2] * w8a8_linear_f(o[sel], qw[1][0], qw[1][1], sm[1])
        h2 = modulated_rmsnorm(xr, nrm[1], m[r, 3], m[r, 4], eps)
        a = swiglu_interleaved(w8a8_linear_f(h2, qw[2][0], qw[2][1], sm[2]))
        out[sel] = xr + m[r, 5] * w8a8_linear_f(a, qw[3][0], qw[3][1], sm[3])
    return out
