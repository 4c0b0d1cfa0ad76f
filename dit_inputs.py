"""Seeded synthetic inputs for the AdaLN DiT block, shared by the CPU oracle and the CUDA path.

This module draws random numbers and nothing else: it holds none of the block's arithmetic
(no norm, rotary table, product, softmax or dequantisation). Both sides of every parity test
take their inputs from here and compute everything else on their own.

Workloads (shapes follow the pages' problem statements):

* ``tiny``      hidden 256, 4 heads x 64, SwiGLU ffn 768, L=8 text + N=64 image rows (8x8 grid), seed 0
* ``512sq``     hidden 3072, 24 heads x 128, ffn 12288, L=64 + N=1024 (32x32 grid), seed 1
* ``1024sq``    same architecture, L=128 + N=4096 (64x64 grid), seed 2
* ``1024sq_int8`` the 1024sq block with all four linears int8 + one bf16 scale per 32 inputs, seed 3
* ``denoise``   32 blocks of the 1024sq architecture, L=512 + N=4096, 4 Euler steps, seed 4

Page basis: an S x S image has (S/16)^2 image tokens and up to 512 text tokens (the RGBA-Image-2.1
host contract, sections 1 and 4); the 4608-row sequence of FLUX.2 klein is 512 + 4096 (the klein-4B
TPU article, section 4.3).

Weights are drawn N(0, 0.02) in float32 and rounded to nearest-even bfloat16; they are returned as
raw bfloat16 bit patterns (``np.uint16``). Activations (text/image rows) are N(0, 1) float32; the
per-row shift/scale/gate modulation rows are N(0, 0.1) float32.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "BlockShape",
    "SHAPES",
    "bf16_bits_from_f32",
    "block_inputs",
    "int8_block_inputs",
    "parallel_block_inputs",
    "denoise_inputs",
]


@dataclass(frozen=True)
class BlockShape:
    name: str
    hidden: int
    heads: int
    head_dim: int
    ffn: int
    L: int           # text rows
    grid_h: int      # image grid rows
    grid_w: int      # image grid columns
    seed: int
    eps: float = 1e-6
    qk_eps: float = 1e-6

    @property
    def N(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def R(self) -> int:
        return self.L + self.N

    def flops(self) -> float:
        """Algorithmic FLOP of one block forward: the four linears plus the two attention products."""
        H, F, R = self.hidden, self.ffn, self.R
        return 2.0 * R * (3 * H * H + H * H + 2 * H * F + F * H) + 4.0 * R * R * H


SHAPES: Dict[str, BlockShape] = {
    "tiny": BlockShape("tiny", 256, 4, 64, 768, 8, 8, 8, seed=0),
    "512sq": BlockShape("512sq", 3072, 24, 128, 12288, 64, 32, 32, seed=1),
    "1024sq": BlockShape("1024sq", 3072, 24, 128, 12288, 128, 64, 64, seed=2),
    "1024sq_int8": BlockShape("1024sq_int8", 3072, 24, 128, 12288, 128, 64, 64, seed=3),
    "denoise": BlockShape("denoise", 3072, 24, 128, 12288, 512, 64, 64, seed=4),
}


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to nearest-even bfloat16, returned as uint16 bit patterns.

    Used only to turn random draws into bf16 weights (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _rng(seed: int, *stream: int) -> np.random.Generator:
    # An independent PCG64 stream per (seed, stream ids): arrays can be drawn in any order.
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


@dataclass
class BlockInputs:
    shape: BlockShape
    txt: np.ndarray            # [L, H] float32 (residual rows, updated by the block)
    img: np.ndarray            # [N, H] float32
    mod: np.ndarray            # [M, 6, H] float32: shift_a, scale_a, gate_a, shift_m, scale_m, gate_m
    mod_map: np.ndarray        # [R] int32: modulation row of each packed row
    wqkv: Optional[np.ndarray] = None   # [3H, H] bf16 bits; rows all-Q, all-K, all-V (head-major)
    wout: Optional[np.ndarray] = None   # [H, H]
    wup: Optional[np.ndarray] = None    # [2F, H], gate row j at 2j, up row j at 2j+1
    wdown: Optional[np.ndarray] = None  # [H, F]
    norm1: Optional[np.ndarray] = None  # [H] float32 or None (= ones)
    norm2: Optional[np.ndarray] = None
    q_norm: Optional[np.ndarray] = None  # [d] float32 or None (= ones)
    k_norm: Optional[np.ndarray] = None
    # int8 variant: per linear (qkv, out, up, down) int8 values [out, in] and bf16 scale bits [out, in/32]
    q8: Optional[List[np.ndarray]] = None
    s8: Optional[List[np.ndarray]] = None
    extra: dict = field(default_factory=dict)


def _activations(shape: BlockShape, M: Optional[int], rng_seed: int):
    H, L, N, R = shape.hidden, shape.L, shape.N, shape.R
    txt = _rng(rng_seed, 1).standard_normal((L, H), dtype=np.float32)
    img = _rng(rng_seed, 2).standard_normal((N, H), dtype=np.float32)
    if M is None:
        M = R
    mod = _rng(rng_seed, 3).standard_normal((M, 6, H), dtype=np.float32) * np.float32(0.1)
    if M == R:
        mod_map = np.arange(R, dtype=np.int32)
    elif M == 1:
        mod_map = np.zeros(R, dtype=np.int32)
    else:
        # M modulation rows: the text rows take row 0, image rows cycle over the rest.
        mod_map = np.zeros(R, dtype=np.int32)
        mod_map[L:] = 1 + (np.arange(N, dtype=np.int32) % (M - 1))
    return txt, img, mod, mod_map


def block_inputs(shape: BlockShape | str, M: Optional[int] = None, norm_weights: bool = False,
                 seed: Optional[int] = None) -> BlockInputs:
    """Inputs of one bf16-weight block. ``M`` modulation rows (default: one per packed row).

    ``norm_weights`` draws the four norm weights as 1 + N(0, 0.02) (the workloads use ones)."""
    if isinstance(shape, str):
        shape = SHAPES[shape]
    s = shape.seed if seed is None else seed
    H, F, d = shape.hidden, shape.ffn, shape.head_dim
    txt, img, mod, mod_map = _activations(shape, M, s)
    out = BlockInputs(shape, txt, img, mod, mod_map)
    out.wqkv = _normal_bf16(_rng(s, 10), (3 * H, H), 0.02)
    out.wout = _normal_bf16(_rng(s, 11), (H, H), 0.02)
    out.wup = _normal_bf16(_rng(s, 12), (2 * F, H), 0.02)
    out.wdown = _normal_bf16(_rng(s, 13), (H, F), 0.02)
    if norm_weights:
        g = _rng(s, 14)
        out.norm1 = (1 + 0.02 * g.standard_normal(H)).astype(np.float32)
        out.norm2 = (1 + 0.02 * g.standard_normal(H)).astype(np.float32)
        out.q_norm = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
        out.k_norm = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
    return out


def parallel_block_inputs(shape: BlockShape | str, M: Optional[int] = None, norm_weights: bool = False,
                          seed: Optional[int] = None) -> BlockInputs:
    """Inputs of one parallel (single-stream) block: the weights and rows of ``block_inputs`` and
    its own modulation rows [M, 3, H] (shift, scale, gate), N(0, 0.1). Only ``norm1`` is used."""
    out = block_inputs(shape, M=M, norm_weights=norm_weights, seed=seed)
    s = out.shape.seed if seed is None else seed
    Mr = out.mod.shape[0]
    out.mod = _rng(s, 4).standard_normal((Mr, 3, out.shape.hidden), dtype=np.float32) * np.float32(0.1)
    return out


INT8_S0 = 0.02 * np.sqrt(3.0) / 127.0


def int8_block_inputs(shape: BlockShape | str = "1024sq_int8", M: Optional[int] = None,
                      seed: Optional[int] = None) -> BlockInputs:
    """Inputs of one int8lin block: each linear's values uniform in [-127, 127] and one bf16 scale
    per 32 consecutive input elements, s = bf16(s0 * (0.75 + 0.5 U(0,1))), s0 = 0.02 sqrt(3) / 127,
    so the weights they stand for have a standard deviation near 0.02."""
    if isinstance(shape, str):
        shape = SHAPES[shape]
    s = shape.seed if seed is None else seed
    H, F = shape.hidden, shape.ffn
    txt, img, mod, mod_map = _activations(shape, M, s)
    out = BlockInputs(shape, txt, img, mod, mod_map)
    dims = [(3 * H, H), (H, H), (2 * F, H), (H, F)]
    out.q8, out.s8 = [], []
    for i, (o, k) in enumerate(dims):
        g = _rng(s, 20 + i)
        out.q8.append(g.integers(-127, 128, size=(o, k), dtype=np.int8))
        u = g.random((o, k // 32), dtype=np.float32)
        out.s8.append(bf16_bits_from_f32(np.float32(INT8_S0) * (np.float32(0.75) + np.float32(0.5) * u)))
    return out


def int8_parallel_block_inputs(shape: BlockShape | str = "1024sq_int8", M: Optional[int] = None,
                               seed: Optional[int] = None) -> BlockInputs:
    """int8lin weights and rows of ``int8_block_inputs`` with the parallel block's own modulation
    rows [M, 3, H] (shift, scale, gate), N(0, 0.1), drawn as in ``parallel_block_inputs``."""
    out = int8_block_inputs(shape, M=M, seed=seed)
    s = out.shape.seed if seed is None else seed
    Mr = out.mod.shape[0]
    out.mod = _rng(s, 4).standard_normal((Mr, 3, out.shape.hidden), dtype=np.float32) * np.float32(0.1)
    return out


@dataclass
class DenoiseInputs:
    shape: BlockShape
    blocks: int
    steps_sigmas: np.ndarray   # [steps + 1] float32
    latents: np.ndarray        # [N, 64] float32 noise (packed image tokens)
    txt_feats: np.ndarray      # [L, H] float32
    w_in: np.ndarray           # [H, 64] bf16 bits  (patch in)
    w_t1: np.ndarray           # [H, 256] bf16 bits (time MLP, first linear)
    w_t2: np.ndarray           # [H, H] bf16 bits   (time MLP, second linear)
    w_ada: np.ndarray          # [blocks, 6H, H] bf16 bits (per-block modulation)
    w_ada_f: np.ndarray        # [2H, H] bf16 bits (final norm shift, scale)
    w_out: np.ndarray          # [64, H] bf16 bits (patch out)
    block_w: List[BlockInputs]  # per block: wqkv, wout, wup, wdown


def denoise_inputs(shape: BlockShape | str = "denoise", blocks: int = 32,
                   sigmas=(1.0, 0.75, 0.5, 0.25, 0.0), seed: Optional[int] = None,
                   latent_channels: int = 64) -> DenoiseInputs:
    """Inputs of the full denoise loop: latents ~ N(0,1), text features ~ N(0,1), every weight
    ~ N(0, 0.02) in bf16, fixed sigmas."""
    if isinstance(shape, str):
        shape = SHAPES[shape]
    s = shape.seed if seed is None else seed
    H, F, L, N = shape.hidden, shape.ffn, shape.L, shape.N
    C = latent_channels
    latents = _rng(s, 1).standard_normal((N, C), dtype=np.float32)
    txt_feats = _rng(s, 2).standard_normal((L, H), dtype=np.float32)
    w_in = _normal_bf16(_rng(s, 30), (H, C), 0.02)
    w_t1 = _normal_bf16(_rng(s, 31), (H, 256), 0.02)
    w_t2 = _normal_bf16(_rng(s, 32), (H, H), 0.02)
    w_ada = np.stack([_normal_bf16(_rng(s, 40, b), (6 * H, H), 0.02) for b in range(blocks)])
    w_ada_f = _normal_bf16(_rng(s, 33), (2 * H, H), 0.02)
    w_out = _normal_bf16(_rng(s, 34), (C, H), 0.02)
    block_w = []
    for b in range(blocks):
        bi = BlockInputs(shape, None, None, None, None)
        bi.wqkv = _normal_bf16(_rng(s, 50, b, 0), (3 * H, H), 0.02)
        bi.wout = _normal_bf16(_rng(s, 50, b, 1), (H, H), 0.02)
        bi.wup = _normal_bf16(_rng(s, 50, b, 2), (2 * F, H), 0.02)
        bi.wdown = _normal_bf16(_rng(s, 50, b, 3), (H, F), 0.02)
        block_w.append(bi)
    return DenoiseInputs(shape, blocks, np.asarray(sigmas, dtype=np.float32), latents, txt_feats,
                         w_in, w_t1, w_t2, w_ada, w_ada_f, w_out, block_w)
