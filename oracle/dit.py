"""Plain float64 NumPy definitions of the DiT block forward and the denoise loop (test oracle).

Sources, cited by page title and section:

* [host contract]  "Host contract - RGBA-Image-2.1-Turbo (Core AI port of Qwen-Image-2.1-Turbo)":
  section 1 (graph I/O, int8lin weights), section 4 (sequence layout and RoPE tables), section 5
  (latent packing), section 6 (FlowMatch Euler sampler).
* [gizai:dit]  the "gizai:dit" module reference: ``Block.forward``, ``normedInto``, ``Modulation``,
  ``Sequence``, ``prepOf``, ``gatedInto``, ``gluRows``, ``weightAt``, ``sinusoids``.
* [klein]  "944 -> 346 ms: optimizing FLUX.2 klein-4B on one TPU v6e chip": section 2 (cast
  points), section 4.3 (attention: softmax with 1/sqrt(d) applied in fp32), section 4.4 (qk prep:
  QK-RMSNorm as mean of squares + eps -> rsqrt).

Readings where the pages are silent, each with its basis:
* modulation uses (1 + scale): the pages name shift, scale and gate only [gizai:dit, Modulation];
  (1 + scale) is the AdaLN convention and keeps the norm's gain near 1 for small scales;
* RMSNorm is x * (mean(x^2) + eps)^-1/2 with eps = 1e-6 for both norms and the QK norm [klein,
  section 4.4: "mean of squares + eps -> rsqrt"];
* RoPE rotates adjacent pairs (2i, 2i+1) of the whole head [host contract, section 4: complex
  pairs built with torch.polar]; d = 64 heads scale the d = 128 axis widths (16, 56, 56) by d / 128,
  giving (8, 28, 28), since the pages give only d = 128;
* the block is sequential, the attention residual landing before the second norm [gizai:dit,
  Block.forward, as opposed to Block.parallel];
* the final norm of the denoise loop is a modulated RMSNorm without an affine weight, and no linear
  has a bias [gizai:dit, Block: a block's linear biases are optional, and a block built from
  weights alone has none; the pages show no head or tail weights].
"""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "bf16_to_f64", "bf16_rne_bits", "positions", "axis_widths", "rope_tables", "rope_axis_table",
    "modulated_rmsnorm", "qk_rmsnorm", "rope_apply", "attention", "silu", "swiglu_interleaved",
    "block_forward", "block_forward_rows", "dequant_int8", "euler_step", "shift_sigmas",
    "timestep_sinusoids", "time_embedding", "denoise", "pack_latents", "block_weights_f64",
    "modulated_layernorm", "parallel_block_forward", "parallel_block_forward_rows", "double_block_forward_rows",
    "rope_apply_split", "rotate", "lora_linear", "lora_merge",
]


# ----------------------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_rne_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to nearest bfloat16, ties to even, as uint16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    rest = u & np.uint64(0xFFFF)
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & np.uint64(1)) == 1))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# sequence layout and rotary tables  [host contract, section 4]
# ----------------------------------------------------------------------------------------------

def positions(L: int, h: int, w: int) -> np.ndarray:
    """3-axis (frame, height, width) positions of the packed [text L | image h*w] sequence.

    Text token i sits at (i, i, i); the image token at row y, column x (index y*w + x) sits at
    (L, y - (h - h//2), x - (w - w//2)), a grid centred on zero.  [host contract, section 4]"""
    pos = np.zeros((L + h * w, 3), dtype=np.int64)
    for i in range(L):
        pos[i] = (i, i, i)
    for y in range(h):
        for x in range(w):
            pos[L + y * w + x] = (L, y - (h - h // 2), x - (w - w // 2))
    return pos


def axis_widths(head_dim: int) -> tuple:
    """Rotary widths of the three axes. The contract gives (16, 56, 56) for a 128-wide head
    [host contract, section 4]; other head sizes scale them by head_dim / 128 (our reading)."""
    if head_dim == 128:
        return (16, 56, 56)
    if (16 * head_dim) % 256 or (56 * head_dim) % 256:
        raise ValueError("head_dim must scale the (16, 56, 56) widths to even integers")
    return (16 * head_dim // 128, 56 * head_dim // 128, 56 * head_dim // 128)


def _axis_frequencies(width: int, theta: float) -> np.ndarray:
    # 1 / theta^(arange(0, width, 2) / width)   [host contract, section 4]
    k = np.arange(0, width, 2, dtype=np.float64)
    return 1.0 / np.power(float(theta), k / width)


def rope_axis_table(width: int, theta: float = 10000.0, first: int = -1024, last: int = 8191):
    """One axis table as the contract stores it: row p - first holds cos/sin of p * f_k for
    positions first..last, [rows, width/2], float32.  [host contract, section 4]"""
    p = np.arange(first, last + 1, dtype=np.float64)
    ang = np.outer(p, _axis_frequencies(width, theta))
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope_tables(pos: np.ndarray, head_dim: int, theta: float = 10000.0):
    """Per-row cos/sin [R, head_dim/2] float32: the three axes' angle columns concatenated in axis
    order, angle = position * frequency evaluated in float64 and rounded once to float32.
    [host contract, section 4]"""
    cols_c, cols_s = [], []
    for a, width in enumerate(axis_widths(head_dim)):
        ang = np.outer(pos[:, a].astype(np.float64), _axis_frequencies(width, theta))
        cols_c.append(np.cos(ang))
        cols_s.append(np.sin(ang))
    return (np.concatenate(cols_c, axis=1).astype(np.float32),
            np.concatenate(cols_s, axis=1).astype(np.float32))


# ----------------------------------------------------------------------------------------------
# block pieces
# ----------------------------------------------------------------------------------------------

def modulated_rmsnorm(x, w, shift, scale, eps):
    """y = x * (mean(x^2) + eps)^-1/2 * w * (1 + scale) + shift, row by row.
    [gizai:dit, normedInto and Modulation; klein, section 4.4 for mean of squares + eps]"""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return y * (1.0 + np.asarray(scale, dtype=np.float64)) + np.asarray(shift, dtype=np.float64)


def qk_rmsnorm(t, w, eps):
    """Each head vector over its own RMS times the head-norm weight: t [R, heads, d].
    [gizai:dit, prepOf; klein, section 4.4]"""
    ms = np.mean(t * t, axis=-1, keepdims=True)
    y = t / np.sqrt(ms + eps)
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return y


def rope_apply(t, cos, sin):
    """Rotate the adjacent pairs (2i, 2i+1) of each head by the row's angle i:
    (a, b) -> (a cos - b sin, a sin + b cos).  t [R, heads, d], cos/sin [R, d/2].
    [host contract, section 4 (complex pairs, torch.polar); klein, section D3 (-sin even, +sin odd)]"""
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    a = t[..., 0::2]
    b = t[..., 1::2]
    out = np.empty_like(t)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def rope_apply_split(t, cos, sin):
    """The split-halves partial rotation: with h = cos.shape[1] (3d/8 of a d-wide head), value i and
    value i + h (i < h) of each head form a pair turned by the row's angle i,
    (a, b) -> (a cos - b sin, a sin + b cos); values from 2h on (the last quarter) are unchanged.
    t [R, heads, d], cos/sin [R, h].  [gizai:dit, prepOf ("its first 2 half values turned") and HEAD
    (a head rotates its first 3/4, head/8 frequencies per axis, twice: split halves)]"""
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    h = c.shape[-1]
    a = t[..., 0:h]
    b = t[..., h:2 * h]
    out = np.array(t, dtype=np.float64, copy=True)
    out[..., 0:h] = a * c - b * s
    out[..., h:2 * h] = a * s + b * c
    return out


def rotate(t, cos, sin):
    """The rotary step of a block, its layout told by the table width: d/2 columns rotate adjacent
    pairs over the whole head (rope_apply), 3d/8 columns the first 3/4 in split halves
    (rope_apply_split)."""
    d = t.shape[-1]
    w = np.asarray(cos).shape[-1]
    if w == d // 2:
        return rope_apply(t, cos, sin)
    if 8 * w == 3 * d:
        return rope_apply_split(t, cos, sin)
    raise ValueError(f"rotary tables of width {w} fit neither layout of a {d}-wide head")


def attention(q, k, v, rows: Optional[np.ndarray] = None):
    """Unmasked softmax attention of every query row over every key row, per head, with scale
    1/sqrt(d):  o = softmax(q k^T / sqrt(d)) v  (max-subtracted).  q/k/v [R, heads, d].
    ``rows`` restricts the query rows. Returns [len(rows), heads * d] with column head*d + j.
    [host contract, section 4 (joint text|image sequence); klein, section 4.3]"""
    R, nh, d = k.shape
    qs = q if rows is None else q[rows]
    out = np.empty((qs.shape[0], nh, d), dtype=np.float64)
    for n in range(nh):
        S = (qs[:, n, :] @ k[:, n, :].T) / math.sqrt(d)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=1, keepdims=True)
        out[:, n, :] = P @ v[:, n, :]
    return out.reshape(qs.shape[0], nh * d)


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_interleaved(u):
    """SwiGLU over interleaved rows: a_j = silu(u_{2j}) * u_{2j+1}.  [gizai:dit, gluRows and Block]"""
    return silu(u[..., 0::2]) * u[..., 1::2]


def block_weights_f64(inp):
    """The four linears of a bf16 block as float64 matrices [out, in]."""
    return (bf16_to_f64(inp.wqkv), bf16_to_f64(inp.wout), bf16_to_f64(inp.wup), bf16_to_f64(inp.wdown))


def _mod_rows(mod, mod_map, rows):
    m = np.asarray(mod, dtype=np.float64)[np.asarray(mod_map)[rows]]
    return [m[:, i, :] for i in range(6)]


def block_forward_rows(x, weights, mod, mod_map, cos, sin, heads, head_dim,
                       rows: Optional[np.ndarray] = None, norm1=None, norm2=None,
                       q_norm=None, k_norm=None, eps=1e-6, qk_eps=1e-6, post_attn=None, post_mlp=None):
    """One AdaLN block over the packed rows x [R, H] (float64 copy returned; x untouched).

    1. h  = modnorm(x; norm1, shift_a, scale_a)
    2. [q|k|v] = h Wqkv^T (columns all-Q, all-K, all-V, head-major inside each)
    3. q, k  <- per-head RMS norm times q_norm / k_norm
    4. rotate q, k by the per-row cos/sin tables (adjacent pairs, or split halves: see rotate)
    5. o = softmax(q k^T / sqrt(d)) v over all rows
    6. x += gate_a * (o Wout^T)
    7. h2 = modnorm(x; norm2, shift_m, scale_m)
    8. a_j = silu(u_{2j}) u_{2j+1}, u = h2 Wup^T
    9. x += gate_m * (a Wdown^T)

    Steps 1-4 run for every row (keys and values need them); steps 5-9 only for ``rows`` (all by
    default), which lets tests check sampled rows of large sequences.
    A sandwich block (post_attn / post_mlp, [H] norm weights) norms each branch's output before its
    gate: x += gate * rmsnorm(y) * post (the block's RMS norm and eps; gizai:dit, POST_ATTN/POST_MLP).
    [gizai:dit, Block.forward, normedInto, weightAt (QKV row order), prepOf, gatedInto, gluRows]"""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    Wqkv, Wout, Wup, Wdown = weights
    all_rows = np.arange(R)
    rows = all_rows if rows is None else np.asarray(rows)
    sa, ca, ga, _, _, _ = _mod_rows(mod, mod_map, all_rows)
    h = modulated_rmsnorm(x, norm1, sa, ca, eps)
    qkv = h @ Wqkv.T
    q = qkv[:, 0:H].reshape(R, nh, d)
    k = qkv[:, H:2 * H].reshape(R, nh, d)
    v = qkv[:, 2 * H:3 * H].reshape(R, nh, d)
    q = rotate(qk_rmsnorm(q, q_norm, qk_eps), cos, sin)
    k = rotate(qk_rmsnorm(k, k_norm, qk_eps), cos, sin)
    o = attention(q, k, v, rows)
    _, _, ga_r, sm_r, cm_r, gm_r = _mod_rows(mod, mod_map, rows)
    post = lambda y, w: y if w is None else modulated_rmsnorm(y, w, 0.0, 0.0, eps)
    xr = x[rows] + ga_r * post(o @ Wout.T, post_attn)
    h2 = modulated_rmsnorm(xr, norm2, sm_r, cm_r, eps)
    a = swiglu_interleaved(h2 @ Wup.T)
    return xr + gm_r * post(a @ Wdown.T, post_mlp)


def block_forward(inp, weights=None, rows=None):
    """Block forward on a ``dit_inputs.BlockInputs``: returns (txt_out, img_out) float64 for all rows,
    or the packed output rows ``rows`` when given. Uses the bf16 weights, or ``weights`` if given."""
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img], axis=0).astype(np.float64)
    cos, sin = rope_tables(positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    W = block_weights_f64(inp) if weights is None else weights
    y = block_forward_rows(x, W, inp.mod, inp.mod_map, cos, sin, sh.heads, sh.head_dim, rows=rows,
                           norm1=inp.norm1, norm2=inp.norm2, q_norm=inp.q_norm, k_norm=inp.k_norm,
                           eps=sh.eps, qk_eps=sh.qk_eps)
    if rows is not None:
        return y
    return y[:sh.L], y[sh.L:]


# ----------------------------------------------------------------------------------------------
# LoRA adapters  [gizai:dit, Block (lora), withLora, loraOf, weightAt]
# ----------------------------------------------------------------------------------------------

def lora_linear(x, W, A, B):
    """A linear with its LoRA adapter beside it: x W^T + (x A^T) B^T, A [rank, in], B [out, rank]
    (the down product, then B's). Float64.  [gizai:dit, loraOf (A product), withLora (B product)]"""
    x = np.asarray(x, dtype=np.float64)
    return x @ np.asarray(W, dtype=np.float64).T + (x @ np.asarray(A, dtype=np.float64).T) @ \
        np.asarray(B, dtype=np.float64).T


def lora_merge(W, A, B):
    """The merged weight W + B A that the adapter stands for.  [gizai:dit, weightAt]"""
    return np.asarray(W, dtype=np.float64) + np.asarray(B, dtype=np.float64) @ np.asarray(A, dtype=np.float64)


# ----------------------------------------------------------------------------------------------
# parallel (single-stream) block  [gizai:dit, Block.parallel]
# ----------------------------------------------------------------------------------------------

def modulated_layernorm(x, w, shift, scale, eps):
    """y = (x - mean(x)) * (var(x) + eps)^-1/2 * w * (1 + scale) + shift, row by row, var the mean
    of squared deviations (biased). w None means ones. Float64.

    The parallel block names a modulated LayerNorm (gizai:dit, Block.parallel); the pages give no
    formula, so this is the textbook LayerNorm with the block's shift/scale modulation and eps."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    dev = x - mu
    var = (dev * dev).mean(axis=-1, keepdims=True)
    y = dev / np.sqrt(var + eps)
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return y * (1.0 + np.asarray(scale, dtype=np.float64)) + np.asarray(shift, dtype=np.float64)


def parallel_block_forward_rows(x, weights, mod, mod_map, cos, sin, heads, head_dim,
                                rows: Optional[np.ndarray] = None, norm=None, q_norm=None, k_norm=None,
                                eps=1e-6, qk_eps=1e-6, post_attn=None, post_mlp=None):
    """The parallel block over the packed rows x [R, H]: both branches read one modulated norm.

    1. h = modulated LayerNorm(x; norm, shift, scale)         mod rows [M, 3, H] = shift, scale, gate
    2. [q|k|v] = h Wqkv^T; q, k per-head RMS norm, rotated    (as in the sequential block)
    3. o = softmax(q k^T / sqrt(d)) v
    4. a_j = silu(u_{2j}) u_{2j+1}, u = h Wup^T               (gate/up rows interleaved)
    5. x + gate * (o Wout^T + a Wdown^T)

    Steps 1-2 run for every row, 3-5 for ``rows`` (all by default).
    With post_attn / post_mlp ([H] norm weights, a sandwich block) each branch's output is RMS-normed
    with its own weight before the shared gate: x + gate * (rmsnorm(o Wout^T) post_attn +
    rmsnorm(a Wdown^T) post_mlp). The pages name the post-norm weights of a block and norm its outputs
    before their gates (gizai:dit, POST_ATTN / POST_MLP) without showing them in the parallel form;
    this is the reading with one gate over both normed branches.
    [gizai:dit, Block.parallel; weightAt, prepOf and gluRows for the shared pieces]"""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    Wqkv, Wout, Wup, Wdown = weights
    rows = np.arange(R) if rows is None else np.asarray(rows)
    m = np.asarray(mod, dtype=np.float64)[np.asarray(mod_map)]
    h = modulated_layernorm(x, norm, m[:, 0], m[:, 1], eps)
    qkv = h @ Wqkv.T
    q = rotate(qk_rmsnorm(qkv[:, 0:H].reshape(R, nh, d), q_norm, qk_eps), cos, sin)
    k = rotate(qk_rmsnorm(qkv[:, H:2 * H].reshape(R, nh, d), k_norm, qk_eps), cos, sin)
    v = qkv[:, 2 * H:3 * H].reshape(R, nh, d)
    o = attention(q, k, v, rows)
    a = swiglu_interleaved(h[rows] @ Wup.T)
    post = lambda y, w: y if w is None else modulated_rmsnorm(y, w, 0.0, 0.0, eps)
    return x[rows] + m[rows, 2] * (post(o @ Wout.T, post_attn) + post(a @ Wdown.T, post_mlp))


def parallel_block_forward(inp, weights=None, rows=None, post_attn=None, post_mlp=None):
    """Parallel block on ``dit_inputs.parallel_block_inputs``: (txt_out, img_out) float64, or the
    packed output rows ``rows`` when given."""
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img], axis=0).astype(np.float64)
    cos, sin = rope_tables(positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    W = block_weights_f64(inp) if weights is None else weights
    y = parallel_block_forward_rows(x, W, inp.mod, inp.mod_map, cos, sin, sh.heads, sh.head_dim, rows=rows,
                                    norm=inp.norm1, q_norm=inp.q_norm, k_norm=inp.k_norm, eps=sh.eps,
                                    qk_eps=sh.qk_eps, post_attn=post_attn, post_mlp=post_mlp)
    if rows is not None:
        return y
    return y[:sh.L], y[sh.L:]


# ----------------------------------------------------------------------------------------------
# double-stream block  [klein article, sections 4.3-4.4 (double blocks); gizai:dit, Block.forward]
# ----------------------------------------------------------------------------------------------

def double_block_forward_rows(x, weights_txt, weights_img, mod, mod_map, cos, sin, heads, head_dim, L,
                              rows: Optional[np.ndarray] = None, norms_txt=(None, None, None, None),
                              norms_img=(None, None, None, None), eps=1e-6, qk_eps=1e-6, post_txt=(None, None),
                              post_img=(None, None)):
    """The double-stream block over the packed rows x [R, H] (text rows 0..L-1, image rows L..R-1):
    the sequential block of ``block_forward_rows`` in which each stream has its own four linears
    and its own norm weights (norm1, norm2, q_norm, k_norm), while the attention is one softmax over
    the concatenated text and image keys. Modulation rows come through ``mod_map`` as for the
    sequential block, so each stream's rows pick their own rows of ``mod`` [M, 6, H]. post_txt /
    post_img are each stream's sandwich post-norm weights (post_attn, post_mlp; None: that branch
    un-normed), as in ``block_forward_rows``."""
    x = np.asarray(x, dtype=np.float64)
    R, H = x.shape
    nh, d = heads, head_dim
    rows = np.arange(R) if rows is None else np.asarray(rows)
    m = np.asarray(mod, dtype=np.float64)[np.asarray(mod_map)]
    streams = [(np.arange(0, L), weights_txt, norms_txt), (np.arange(L, R), weights_img, norms_img)]
    posts = [post_txt, post_img]
    post = lambda y, w: y if w is None else modulated_rmsnorm(y, w, 0.0, 0.0, eps)
    q = np.empty((R, nh, d))
    k = np.empty((R, nh, d))
    v = np.empty((R, nh, d))
    for idx, W, nrm in streams:
        if idx.size == 0:
            continue
        h = modulated_rmsnorm(x[idx], nrm[0], m[idx, 0], m[idx, 1], eps)
        qkv = h @ W[0].T
        q[idx] = rotate(qk_rmsnorm(qkv[:, 0:H].reshape(-1, nh, d), nrm[2], qk_eps), cos[idx], sin[idx])
        k[idx] = rotate(qk_rmsnorm(qkv[:, H:2 * H].reshape(-1, nh, d), nrm[3], qk_eps), cos[idx], sin[idx])
        v[idx] = qkv[:, 2 * H:3 * H].reshape(-1, nh, d)
    o = attention(q, k, v, rows)
    out = np.empty((rows.size, H))
    for (idx, W, nrm), pw in zip(streams, posts):
        sel = np.isin(rows, idx)
        if not sel.any():
            continue
        r = rows[sel]
        xr = x[r] + m[r, 2] * post(o[sel] @ W[1].T, pw[0])
        h2 = modulated_rmsnorm(xr, nrm[1], m[r, 3], m[r, 4], eps)
        out[sel] = xr + m[r, 5] * post(swiglu_interleaved(h2 @ W[2].T) @ W[3].T, pw[1])
    return out


# ----------------------------------------------------------------------------------------------
# int8lin weights  [host contract, section 1]
# ----------------------------------------------------------------------------------------------

def dequant_int8(q: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """W[o, i] = bf16_rne(q[o, i] * s[o, i // 32]) as bf16 bit patterns.

    The int8 value times the bf16 scale has at most 16 significant bits, so the product is exact in
    float64 (and float32) before the one rounding to bfloat16.  [host contract, section 1]"""
    o, k = q.shape
    if k % 32:
        raise ValueError("input dimension must be a multiple of 32")
    s = bf16_to_f64(s_bits)
    prod = q.astype(np.float64) * np.repeat(s, 32, axis=1)
    return bf16_rne_bits(prod.astype(np.float32))  # exact conversion, then one RNE rounding


# ----------------------------------------------------------------------------------------------
# sampler and denoise loop  [host contract, sections 5 and 6; gizai:dit, sinusoids]
# ----------------------------------------------------------------------------------------------

def euler_step(x: np.ndarray, vel: np.ndarray, sigma: float, sigma_next: float) -> np.ndarray:
    """x + (sigma_next - sigma) * vel, every operation in float32.  [host contract, section 6]"""
    x = np.asarray(x, dtype=np.float32)
    vel = np.asarray(vel, dtype=np.float32)
    dt = np.float32(sigma_next) - np.float32(sigma)
    return (x + (dt * vel).astype(np.float32)).astype(np.float32)


def shift_sigmas(sigmas, shift: float) -> np.ndarray:
    """shift * s / (1 + (shift - 1) * s) in float32.  [host contract, section 6]"""
    s = np.asarray(sigmas, dtype=np.float32)
    sh = np.float32(shift)
    return (sh * s / (np.float32(1) + (sh - np.float32(1)) * s)).astype(np.float32)


def pack_latents(z: np.ndarray) -> np.ndarray:
    """Channel-major latent z [C, h, w] to tokens x [h*w, C] with x[y*w + x, c] = z[c, y, x].
    [host contract, section 5]"""
    C, h, w = z.shape
    out = np.empty((h * w, C), dtype=z.dtype)
    for y in range(h):
        for xx in range(w):
            out[y * w + xx, :] = z[:, y, xx]
    return out


def timestep_sinusoids(t: Sequence[float], dim: int = 256) -> np.ndarray:
    """Rows [cos | sin] of 1000 * t times the dim/2 frequencies 10000^(-i / (dim/2)).
    [gizai:dit, sinusoids; klein, section 2 (the model sees 1000 t)]"""
    half = dim // 2
    f = np.power(10000.0, -np.arange(half, dtype=np.float64) / half)
    ang = np.outer(1000.0 * np.asarray(t, dtype=np.float64), f)
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def time_embedding(t, w_t1, w_t2):
    """temb = W2 silu(W1 sinusoids(t)) (no biases, our reading)."""
    e = timestep_sinusoids(t, dim=bf16_to_f64(w_t1).shape[1])
    return silu(e @ bf16_to_f64(w_t1).T) @ bf16_to_f64(w_t2).T


def denoise(inp, steps: Optional[int] = None, blocks: Optional[int] = None, trace: Optional[list] = None):
    """The full loop of the host contract's section 6 with a plain DiT around the blocks:

    for each step i with t = sigma_i:
        X     = x W_in^T                                  (patch in, image rows)
        temb  = W2 silu(W1 sinusoids(t))                  (time embedding)
        rows  = [txt_feats ; X], then every block with its modulation W_ada,b silu(temb), M = 1
        vel   = modnorm(image rows; shift_f, scale_f) W_proj^T,  [shift_f, scale_f] = W_ada,f silu(temb)
        x     = x + (sigma_{i+1} - sigma_i) vel            (float32)

    Returns x (float32 [N, C]). ``trace`` collects each step's vel when given."""
    sh = inp.shape
    H, L, N = sh.hidden, sh.L, sh.N
    nsteps = len(inp.steps_sigmas) - 1 if steps is None else steps
    nblocks = inp.blocks if blocks is None else blocks
    cos, sin = rope_tables(positions(L, sh.grid_h, sh.grid_w), sh.head_dim)
    W_in = bf16_to_f64(inp.w_in)
    W_ada_f = bf16_to_f64(inp.w_ada_f)
    W_proj = bf16_to_f64(inp.w_out)
    mod_map = np.zeros(L + N, dtype=np.int32)
    x = np.asarray(inp.latents, dtype=np.float32).copy()
    sig = inp.steps_sigmas
    for i in range(nsteps):
        t = float(sig[i])
        temb = time_embedding([t], inp.w_t1, inp.w_t2)[0]
        st = silu(temb)
        rows = np.concatenate([inp.txt_feats.astype(np.float64), x.astype(np.float64) @ W_in.T], axis=0)
        for b in range(nblocks):
            mod = (bf16_to_f64(inp.w_ada[b]) @ st).reshape(1, 6, H)
            bw = inp.block_w[b]
            rows = block_forward_rows(rows, block_weights_f64(bw), mod, mod_map, cos, sin,
                                      sh.heads, sh.head_dim, eps=sh.eps, qk_eps=sh.qk_eps)
        fin = W_ada_f @ st
        shift_f, scale_f = fin[:H], fin[H:]
        vel = modulated_rmsnorm(rows[L:], None, shift_f, scale_f, sh.eps) @ W_proj.T
        if trace is not None:
            trace.append(vel.copy())
        x = euler_step(x, vel.astype(np.float32), sig[i], sig[i + 1])
    return x
