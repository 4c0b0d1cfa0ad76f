"""Helpers for the GPU parity tests: host <-> device marshalling and error measures.

Nothing here computes any part of the block; the CUDA side runs through the C ABI and the
expected values come from ``oracle/``."""

import numpy as np
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return (bf16_bits(t).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def workspace(nbytes: int) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def dims_of(shape: DI.BlockShape) -> D.DitDims:
    return D.DitDims(shape.hidden, shape.heads, shape.head_dim, shape.ffn, shape.eps, shape.qk_eps)


def rope_dev(shape: DI.BlockShape):
    """Rotary tables built by the library (dit_rope_tables): (txt_cos, txt_sin, img_cos, img_sin)."""
    R, half = shape.R, shape.head_dim // 2
    cos = torch.empty(R, half, dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    D.dit_rope_tables(shape.L, shape.grid_h, shape.grid_w, shape.head_dim, cos, sin)
    L = shape.L
    return cos[:L].contiguous(), sin[:L].contiguous(), cos[L:].contiguous(), sin[L:].contiguous()


def opt_dev(a):
    return None if a is None else dev(a)


def block_weights_dev(inp) -> D.BlockWeights:
    return D.BlockWeights(dev_bf16(inp.wqkv), dev_bf16(inp.wout), dev_bf16(inp.wup), dev_bf16(inp.wdown),
                          opt_dev(inp.norm1), opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))


def int8_weights_dev(inp) -> D.Int8BlockWeights:
    return D.Int8BlockWeights([dev(q) for q in inp.q8], [dev_bf16(s) for s in inp.s8], opt_dev(inp.norm1),
                              opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))


def modulation_dev(inp) -> D.Modulation:
    return D.Modulation(dev(inp.mod), dev(inp.mod_map))


def run_block_gpu(inp, int8: bool = False):
    """Run one block through the C ABI on the inputs; returns (txt_out, img_out) as float64 arrays."""
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    mod = modulation_dev(inp)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 1 if int8 else 0))
    if int8:
        D.dit_block_forward_int8(dims, int8_weights_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    else:
        D.dit_block_forward(dims, block_weights_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return t, img.cpu().numpy().astype(np.float64)


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rms(a):
    return float(np.sqrt(np.mean(np.square(np.asarray(a, np.float64))))) if np.size(a) else 0.0
