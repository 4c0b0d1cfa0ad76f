"""GB300 (sm_103a) AdaLN diffusion-transformer block library: thin Python binding of libdit.so.

Every function here only marshals arguments (torch CUDA tensors -> device pointers, the current
torch stream) and calls the C ABI of the same name declared in ``include/dit.h``; all arithmetic
runs in the library's CUDA kernels. There is no fallback: if libdit.so is missing or fails to load,
every call raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int64, c_size_t, c_void_p
from typing import List, Optional, Sequence

__all__ = [
    "DitError", "lib", "library_path", "DitDims", "BlockWeights", "Int8BlockWeights", "Modulation",
    "DenoiseModel", "dit_block_forward", "dit_block_forward_int8", "dit_parallel_block_forward",
    "dit_parallel_block_forward_int8", "dit_double_block_forward_int8",
    "W8A8BlockWeights", "dit_block_forward_w8a8", "dit_w8a8_quantize_weight", "dit_w8a8_quantize_rows",
    "ParallelW8A8Weights", "dit_parallel_block_forward_w8a8", "dit_double_block_forward_w8a8",
    "dit_linear_w8a8", "dit_linear_w8a8_workspace_bytes",
    "dit_double_block_forward", "dit_block_forward_lora", "dit_lora_workspace_bytes", "LoRA", "dit_lora_merge",
    "dit_parallel_block_forward_lora", "dit_double_block_forward_lora", "dit_parallel_block_forward_sandwich",
    "dit_double_block_forward_sandwich",
    "dit_block_forward_sandwich", "dit_euler_step",
    "dit_rope_tables",
    "dit_denoise", "dit_block_forward_noalloc", "dit_block_noalloc_max_bytes", "dit_workspace_bytes", "dit_denoise_workspace_bytes", "dit_modnorm", "dit_qkv_rope",
    "dit_vt_stride", "dit_stream_k_workspace_bytes", "dit_attention", "dit_attention_qknorm", "dit_attention_workspace_bytes", "dit_linear_gated", "dit_linear_swiglu", "dit_linear",
    "dit_dequant_int8", "dit_linear_int8", "dit_linear_int8_workspace_bytes", "dit_check", "dit_selftest_bounded_wait", "dit_status_string", "dit_version",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libdit.so")

DIT_OK, DIT_EINVAL, DIT_EUNSUPPORTED, DIT_EWORKSPACE, DIT_ECUDA, DIT_ETIMEOUT = 0, -1, -2, -3, -4, -5


class DitError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({dit_status_string(status)})")


# ----------------------------------------------------------------------------------------------
# C structs (mirror include/dit.h)
# ----------------------------------------------------------------------------------------------
class dit_dims(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("heads", c_int), ("head_dim", c_int), ("ffn", c_int),
                ("eps", c_float), ("qk_eps", c_float), ("rope_split", c_int)]


class dit_block_w(ctypes.Structure):
    _fields_ = [("wqkv", c_void_p), ("wout", c_void_p), ("wup", c_void_p), ("wdown", c_void_p),
                ("norm1", c_void_p), ("norm2", c_void_p), ("q_norm", c_void_p), ("k_norm", c_void_p)]


class dit_lora(ctypes.Structure):
    _fields_ = [("A", c_void_p * 4), ("B", c_void_p * 4), ("rank", c_int)]


class dit_block_w8(ctypes.Structure):
    _fields_ = [("q", c_void_p * 4), ("s", c_void_p * 4), ("norm1", c_void_p), ("norm2", c_void_p),
                ("q_norm", c_void_p), ("k_norm", c_void_p)]


class dit_block_w8a8(ctypes.Structure):
    _fields_ = [("q", c_void_p * 4), ("scale", c_void_p * 4), ("smooth", c_void_p * 4), ("norm1", c_void_p),
                ("norm2", c_void_p), ("q_norm", c_void_p), ("k_norm", c_void_p)]


class dit_parallel_w8a8(ctypes.Structure):
    _fields_ = [("q1", c_void_p), ("scale1", c_void_p), ("smooth1", c_void_p), ("q2", c_void_p), ("scale2", c_void_p),
                ("smooth2", c_void_p), ("norm1", c_void_p), ("q_norm", c_void_p), ("k_norm", c_void_p)]


class dit_mod(ctypes.Structure):
    _fields_ = [("rows", c_void_p), ("map", c_void_p), ("M", c_int)]


class dit_model(ctypes.Structure):
    _fields_ = [("dims", dit_dims), ("blocks", c_int), ("latent_channels", c_int), ("w_in", c_void_p),
                ("w_t1", c_void_p), ("w_t2", c_void_p), ("w_ada", c_void_p), ("w_ada_f", c_void_p),
                ("w_out", c_void_p), ("block", POINTER(dit_block_w))]


_SIGNATURES = {
    "dit_block_forward": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_int, c_void_p, c_int,
                                  c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod), c_void_p, c_size_t,
                                  c_void_p]),
    "dit_double_block_forward": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), POINTER(dit_block_w), c_void_p,
                                         c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                         POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_block_forward_lora": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), POINTER(dit_lora), c_void_p, c_int,
                                       c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod),
                                       c_void_p, c_size_t, c_void_p]),
    "dit_lora_workspace_bytes": (c_size_t, [POINTER(dit_dims), c_int, c_int, c_int]),
    "dit_parallel_block_forward_sandwich": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_void_p,
                                                    c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                                    c_void_p, POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_double_block_forward_sandwich": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_void_p,
                                                  POINTER(dit_block_w), c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                                  c_int, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod),
                                                  c_void_p, c_size_t, c_void_p]),
    "dit_parallel_block_forward_lora": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), POINTER(dit_lora), c_void_p,
                                                c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_double_block_forward_lora": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), POINTER(dit_lora),
                                              POINTER(dit_block_w), POINTER(dit_lora), c_void_p, c_int, c_void_p,
                                              c_int, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod),
                                              c_void_p, c_size_t, c_void_p]),
    "dit_block_forward_sandwich": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_void_p, c_void_p,
                                           c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                           POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_parallel_block_forward": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_int, c_void_p, c_int,
                                           c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod), c_void_p,
                                           c_size_t, c_void_p]),
    "dit_block_forward_int8": (c_int, [POINTER(dit_dims), POINTER(dit_block_w8), c_void_p, c_int, c_void_p, c_int,
                                       c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod), c_void_p,
                                       c_size_t, c_void_p]),
    "dit_parallel_block_forward_int8": (c_int, [POINTER(dit_dims), POINTER(dit_block_w8), c_void_p, c_int, c_void_p,
                                                c_int, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod),
                                                c_void_p, c_size_t, c_void_p]),
    "dit_double_block_forward_int8": (c_int, [POINTER(dit_dims), POINTER(dit_block_w8), POINTER(dit_block_w8),
                                              c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                              c_void_p, POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_block_forward_w8a8": (c_int, [POINTER(dit_dims), POINTER(dit_block_w8a8), c_void_p, c_int, c_void_p, c_int,
                                       c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod), c_void_p,
                                       c_size_t, c_void_p]),
    "dit_parallel_block_forward_w8a8": (c_int, [POINTER(dit_dims), POINTER(dit_parallel_w8a8), c_void_p, c_int,
                                                c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_double_block_forward_w8a8": (c_int, [POINTER(dit_dims), POINTER(dit_block_w8a8), POINTER(dit_block_w8a8),
                                              c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                              c_void_p, POINTER(dit_mod), c_void_p, c_size_t, c_void_p]),
    "dit_lora_merge": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p]),
    "dit_w8a8_quantize_weight": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dit_w8a8_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "dit_linear_w8a8": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                c_size_t, c_void_p]),
    "dit_linear_w8a8_workspace_bytes": (c_size_t, [c_int, c_int, c_int]),
    "dit_block_forward_noalloc": (c_int, [POINTER(dit_dims), POINTER(dit_block_w), c_void_p, c_int, c_void_p, c_int,
                                          c_void_p, c_void_p, c_void_p, c_void_p, POINTER(dit_mod), c_void_p]),
    "dit_block_noalloc_max_bytes": (c_size_t, []),
    "dit_euler_step": (c_int, [c_void_p, c_void_p, c_int64, c_float, c_float, c_void_p]),
    "dit_rope_tables": (c_int, [c_int, c_int, c_int, c_int, c_float, c_void_p, c_void_p, c_void_p]),
    "dit_denoise": (c_int, [POINTER(dit_model), c_void_p, c_int, c_void_p, c_int, POINTER(c_float), c_int,
                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "dit_workspace_bytes": (c_size_t, [POINTER(dit_dims), c_int, c_int, c_int]),
    "dit_denoise_workspace_bytes": (c_size_t, [POINTER(dit_model), c_int, c_int, c_int]),
    "dit_modnorm": (c_int, [POINTER(dit_dims), c_void_p, c_int, c_void_p, c_int, c_void_p, POINTER(dit_mod), c_int,
                            c_void_p, c_void_p]),
    "dit_qkv_rope": (c_int, [POINTER(dit_dims), c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                             c_void_p]),
    "dit_stream_k_workspace_bytes": (c_size_t, []),
    "dit_vt_stride": (c_int, [c_int]),
    "dit_attention": (c_int, [POINTER(dit_dims), c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                              c_void_p]),
    "dit_attention_workspace_bytes": (c_size_t, [POINTER(dit_dims), c_int]),
    "dit_attention_qknorm": (c_int, [POINTER(dit_dims), c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_size_t, c_void_p]),
    "dit_linear_gated": (c_int, [POINTER(dit_dims), c_void_p, c_int, c_int, c_void_p, POINTER(dit_mod), c_int,
                                 c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "dit_linear_swiglu": (c_int, [POINTER(dit_dims), c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_size_t,
                                  c_void_p]),
    "dit_linear": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_void_p, c_int, c_void_p]),
    "dit_dequant_int8": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "dit_linear_int8": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_size_t,
                                c_void_p]),
    "dit_linear_int8_workspace_bytes": (c_size_t, [c_int, c_int]),
    "dit_check": (c_int, [c_void_p]),
    "dit_selftest_bounded_wait": (c_int, [c_int, c_void_p]),
    "dit_status_string": (c_char_p, [c_int]),
    "dit_version": (c_int, []),
}

_lib = None


def lib():
    """Load libdit.so (built in-tree by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"libdit.so not built ({library_path}); run __graft_entry__.build()")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def dit_status_string(status: int) -> str:
    return lib().dit_status_string(int(status)).decode()


def dit_version() -> int:
    return lib().dit_version()


def _ok(status: int, where: str):
    if status != DIT_OK:
        raise DitError(status, where)


# ----------------------------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------------------------
def _ptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: expected dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


def _bf16():
    import torch
    return (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class DitDims:
    def __init__(self, hidden: int, heads: int, head_dim: int, ffn: int, eps: float = 1e-6, qk_eps: float = 1e-6,
                 rope_split: bool = False):
        self.c = dit_dims(hidden, heads, head_dim, ffn, eps, qk_eps, 1 if rope_split else 0)
        self.hidden, self.heads, self.head_dim, self.ffn = hidden, heads, head_dim, ffn
        self.eps, self.qk_eps, self.rope_split = eps, qk_eps, bool(rope_split)


class BlockWeights:
    """Device tensors of one bf16 block (kept alive by this object)."""

    def __init__(self, wqkv, wout, wup, wdown, norm1=None, norm2=None, q_norm=None, k_norm=None):
        import torch
        bf = _bf16()
        f32 = torch.float32
        self.tensors = (wqkv, wout, wup, wdown, norm1, norm2, q_norm, k_norm)
        self.c = dit_block_w(_ptr(wqkv, bf, "wqkv"), _ptr(wout, bf, "wout"), _ptr(wup, bf, "wup"),
                             _ptr(wdown, bf, "wdown"), _ptr(norm1, f32, "norm1"), _ptr(norm2, f32, "norm2"),
                             _ptr(q_norm, f32, "q_norm"), _ptr(k_norm, f32, "k_norm"))


class Int8BlockWeights:
    """Device tensors of one int8lin block: q [4] int8 [out, in], s [4] bf16 [out, in/32]."""

    def __init__(self, q: Sequence, s: Sequence, norm1=None, norm2=None, q_norm=None, k_norm=None):
        import torch
        f32 = torch.float32
        self.tensors = (tuple(q), tuple(s), norm1, norm2, q_norm, k_norm)
        qp = (c_void_p * 4)(*[_ptr(t, torch.int8, "q") for t in q])
        sp = (c_void_p * 4)(*[_ptr(t, _bf16(), "s") for t in s])
        self.c = dit_block_w8(qp, sp, _ptr(norm1, f32, "norm1"), _ptr(norm2, f32, "norm2"),
                              _ptr(q_norm, f32, "q_norm"), _ptr(k_norm, f32, "k_norm"))


class W8A8BlockWeights:
    """Device tensors of one W8A8 block: q [4] int8 [out, in], scale [4] fp32 [out], smooth [4] fp32
    [in] or None (SmoothQuant divisors folded into q), and the norm weights."""

    def __init__(self, q: Sequence, scale: Sequence, smooth: Optional[Sequence] = None, norm1=None, norm2=None,
                 q_norm=None, k_norm=None):
        import torch
        f32 = torch.float32
        smooth = list(smooth) if smooth is not None else [None] * 4
        self.tensors = (tuple(q), tuple(scale), tuple(smooth), norm1, norm2, q_norm, k_norm)
        self.c = dit_block_w8a8((c_void_p * 4)(*[_ptr(t, torch.int8, "q") for t in q]),
                                (c_void_p * 4)(*[_ptr(t, f32, "scale") for t in scale]),
                                (c_void_p * 4)(*[_ptr(t, f32, "smooth") for t in smooth]),
                                _ptr(norm1, f32, "norm1"), _ptr(norm2, f32, "norm2"), _ptr(q_norm, f32, "q_norm"),
                                _ptr(k_norm, f32, "k_norm"))


class ParallelW8A8Weights:
    """Device tensors of one W8A8 parallel block: linear1 = [Wqkv ; Wup] codes q1 int8 [3H + 2F, H] with
    scale1 fp32 [3H + 2F], linear2 = [Wout | Wdown] codes q2 int8 [H, H + F] with scale2 fp32 [H], the
    SmoothQuant divisors smooth1 [H] and smooth2 [H + F] (or None), and the norm weights."""

    def __init__(self, q1, scale1, q2, scale2, smooth1=None, smooth2=None, norm1=None, q_norm=None, k_norm=None):
        import torch
        f32 = torch.float32
        self.tensors = (q1, scale1, q2, scale2, smooth1, smooth2, norm1, q_norm, k_norm)
        self.c = dit_parallel_w8a8(_ptr(q1, torch.int8, "q1"), _ptr(scale1, f32, "scale1"), _ptr(smooth1, f32, "smooth1"),
                                   _ptr(q2, torch.int8, "q2"), _ptr(scale2, f32, "scale2"), _ptr(smooth2, f32, "smooth2"),
                                   _ptr(norm1, f32, "norm1"), _ptr(q_norm, f32, "q_norm"), _ptr(k_norm, f32, "k_norm"))


class Modulation:
    """rows [M, 6, H] fp32 device tensor and map [R] int32 (or None)."""

    def __init__(self, rows, map=None):
        import torch
        self.tensors = (rows, map)
        self.c = dit_mod(_ptr(rows, torch.float32, "mod rows"), _ptr(map, torch.int32, "map"), rows.shape[0])


class LoRA:
    """Adapters of a block's four linears (qkv, out, up, down): lists of bf16 device tensors
    A[i] [rank, in_i] and B[i] [out_i, rank], or None for a linear without one."""

    def __init__(self, A, B, rank: int):
        bf = _bf16()
        self.tensors = (A, B)
        self.c = dit_lora((c_void_p * 4)(*[_ptr(a, bf, "lora A") for a in A]),
                          (c_void_p * 4)(*[_ptr(b, bf, "lora B") for b in B]), rank)


class DenoiseModel:
    def __init__(self, dims: DitDims, w_in, w_t1, w_t2, w_ada, w_ada_f, w_out, blocks: List[BlockWeights],
                 latent_channels: int = 64):
        bf = _bf16()
        self.dims, self.blocks = dims, blocks
        self.tensors = (w_in, w_t1, w_t2, w_ada, w_ada_f, w_out)
        self._arr = (dit_block_w * max(1, len(blocks)))(*[b.c for b in blocks])
        self.c = dit_model(dims.c, len(blocks), latent_channels, _ptr(w_in, bf, "w_in"), _ptr(w_t1, bf, "w_t1"),
                           _ptr(w_t2, bf, "w_t2"), _ptr(w_ada, bf, "w_ada"), _ptr(w_ada_f, bf, "w_ada_f"),
                           _ptr(w_out, bf, "w_out"), ctypes.cast(self._arr, POINTER(dit_block_w)))


# ----------------------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------------------------
def dit_workspace_bytes(dims: DitDims, L: int, N: int, variant: int = 0) -> int:
    return lib().dit_workspace_bytes(ctypes.byref(dims.c), L, N, variant)


def dit_denoise_workspace_bytes(model: DenoiseModel, L: int, N: int, steps: int) -> int:
    return lib().dit_denoise_workspace_bytes(ctypes.byref(model.c), L, N, steps)


def dit_vt_stride(R: int) -> int:
    return lib().dit_vt_stride(R)


def dit_block_forward(dims: DitDims, w: BlockWeights, txt, img, txt_cos, txt_sin, img_cos, img_sin,
                      mod: Modulation, ws, stream=None):
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                ws.numel() * ws.element_size(), _stream(stream)), "dit_block_forward")


def dit_block_forward_int8(dims: DitDims, w: Int8BlockWeights, txt, img, txt_cos, txt_sin, img_cos, img_sin,
                           mod: Modulation, ws, stream=None):
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward_int8(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                     _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                     _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                     _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_block_forward_int8")


def dit_block_forward_lora(dims: DitDims, w: BlockWeights, lora: "LoRA", txt, img, txt_cos, txt_sin, img_cos,
                           img_sin, mod: Modulation, ws, stream=None):
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward_lora(ctypes.byref(dims.c), ctypes.byref(w.c), ctypes.byref(lora.c),
                                     _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"), img.shape[0],
                                     _ptr(txt_cos, f32), _ptr(txt_sin, f32), _ptr(img_cos, f32), _ptr(img_sin, f32),
                                     ctypes.byref(mod.c), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                     _stream(stream)), "dit_block_forward_lora")


def dit_parallel_block_forward_lora(dims: DitDims, w: BlockWeights, lora: "LoRA", txt, img, txt_cos, txt_sin,
                                    img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The parallel block with LoRA adapters; mod rows are [M, 3, H] (shift, scale, gate)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_parallel_block_forward_lora(ctypes.byref(dims.c), ctypes.byref(w.c), ctypes.byref(lora.c),
                                              _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"), img.shape[0],
                                              _ptr(txt_cos, f32), _ptr(txt_sin, f32), _ptr(img_cos, f32),
                                              _ptr(img_sin, f32), ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                              ws.numel() * ws.element_size(), _stream(stream)),
        "dit_parallel_block_forward_lora")


def dit_double_block_forward_lora(dims: DitDims, w_txt: Optional[BlockWeights], lora_txt: Optional["LoRA"],
                                  w_img: BlockWeights, lora_img: Optional["LoRA"], txt, img, txt_cos, txt_sin,
                                  img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The double-stream block with per-stream LoRA adapters (either set may be None, not both)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    ref = lambda x: None if x is None else ctypes.byref(x.c)
    _ok(lib().dit_double_block_forward_lora(ctypes.byref(dims.c), ref(w_txt), ref(lora_txt), ctypes.byref(w_img.c),
                                            ref(lora_img), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"),
                                            img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32), _ptr(img_cos, f32),
                                            _ptr(img_sin, f32), ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                            ws.numel() * ws.element_size(), _stream(stream)),
        "dit_double_block_forward_lora")


def dit_parallel_block_forward_sandwich(dims: DitDims, w: BlockWeights, post_attn, post_mlp, txt, img, txt_cos,
                                        txt_sin, img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The parallel sandwich block; post_attn / post_mlp [H] fp32 (None: that branch un-normed)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_parallel_block_forward_sandwich(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(post_attn, f32),
                                                  _ptr(post_mlp, f32), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"),
                                                  img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                                  _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                                  _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                                  _stream(stream)),
        "dit_parallel_block_forward_sandwich")


def dit_double_block_forward_sandwich(dims: DitDims, w_txt: Optional[BlockWeights], post_txt, w_img: BlockWeights,
                                      post_img, txt, img, txt_cos, txt_sin, img_cos, img_sin, mod: Modulation, ws,
                                      stream=None):
    """The double-stream sandwich block; post_txt / post_img = (post_attn, post_mlp) [H] fp32 or None each."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    pt = post_txt if post_txt is not None else (None, None)
    pi = post_img if post_img is not None else (None, None)
    _ok(lib().dit_double_block_forward_sandwich(ctypes.byref(dims.c), None if w_txt is None else ctypes.byref(w_txt.c),
                                                _ptr(pt[0], f32), _ptr(pt[1], f32), ctypes.byref(w_img.c),
                                                _ptr(pi[0], f32), _ptr(pi[1], f32), _ptr(txt, f32, "txt"), L,
                                                _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32),
                                                _ptr(txt_sin, f32), _ptr(img_cos, f32), _ptr(img_sin, f32),
                                                ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                                ws.numel() * ws.element_size(), _stream(stream)),
        "dit_double_block_forward_sandwich")


def dit_block_forward_sandwich(dims: DitDims, w: BlockWeights, post_attn, post_mlp, txt, img, txt_cos, txt_sin,
                               img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The sandwich block: post_attn / post_mlp [H] fp32 norm weights (None: that branch un-normed)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward_sandwich(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(post_attn, f32, "post_attn"),
                                         _ptr(post_mlp, f32, "post_mlp"), _ptr(txt, f32, "txt"), L,
                                         _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                         _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                         _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_block_forward_sandwich")


def dit_lora_workspace_bytes(dims: DitDims, L: int, N: int, rank: int) -> int:
    return lib().dit_lora_workspace_bytes(ctypes.byref(dims.c), L, N, rank)


def dit_parallel_block_forward(dims: DitDims, w: BlockWeights, txt, img, txt_cos, txt_sin, img_cos, img_sin,
                               mod: Modulation, ws, stream=None):
    """The parallel block; mod rows are [M, 3, H] (shift, scale, gate)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_parallel_block_forward(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                         _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                         _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                         _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_parallel_block_forward")


def dit_double_block_forward(dims: DitDims, w_txt: Optional[BlockWeights], w_img: BlockWeights, txt, img, txt_cos,
                             txt_sin, img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The double-stream block: text rows use w_txt, image rows w_img, one joint attention."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_double_block_forward(ctypes.byref(dims.c), None if w_txt is None else ctypes.byref(w_txt.c),
                                       ctypes.byref(w_img.c), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"),
                                       img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32), _ptr(img_cos, f32),
                                       _ptr(img_sin, f32), ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                       ws.numel() * ws.element_size(), _stream(stream)),
        "dit_double_block_forward")


def dit_lora_merge(W, A, B, merged, stream=None):
    """merged = bf16(W + B A): W [out, in], A [rank, in], B [out, rank], merged [out, in] (may be W)."""
    bf = _bf16()
    n_out, n_in = W.shape
    rank = A.shape[0]
    if tuple(A.shape) != (rank, n_in) or tuple(B.shape) != (n_out, rank) or tuple(merged.shape) != (n_out, n_in):
        raise ValueError("dit_lora_merge: W [out, in], A [rank, in], B [out, rank], merged [out, in]")
    _ok(lib().dit_lora_merge(_ptr(W, bf, "W"), n_out, n_in, _ptr(A, bf, "A"), _ptr(B, bf, "B"), rank,
                             _ptr(merged, bf, "merged"), _stream(stream)), "dit_lora_merge")


def dit_parallel_block_forward_int8(dims: DitDims, w: Int8BlockWeights, txt, img, txt_cos, txt_sin, img_cos,
                                    img_sin, mod: Modulation, ws, stream=None):
    """The parallel block with int8lin weights; mod rows are [M, 3, H] (shift, scale, gate)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_parallel_block_forward_int8(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                              _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32),
                                              _ptr(txt_sin, f32), _ptr(img_cos, f32), _ptr(img_sin, f32),
                                              ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                              ws.numel() * ws.element_size(), _stream(stream)),
        "dit_parallel_block_forward_int8")


def dit_double_block_forward_int8(dims: DitDims, w_txt: Optional[Int8BlockWeights], w_img: Int8BlockWeights, txt,
                                  img, txt_cos, txt_sin, img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The double-stream block with int8lin weights: text rows use w_txt, image rows w_img."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_double_block_forward_int8(ctypes.byref(dims.c), None if w_txt is None else ctypes.byref(w_txt.c),
                                            ctypes.byref(w_img.c), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"),
                                            img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                            _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                            _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_double_block_forward_int8")


def dit_block_forward_noalloc(dims: DitDims, w: BlockWeights, txt, img, txt_cos, txt_sin, img_cos, img_sin,
                              mod: Modulation, stream=None):
    """dit_block_forward with its scratch in the library's static device array (no allocation)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward_noalloc(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                        _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                        _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c), _stream(stream)),
        "dit_block_forward_noalloc")


def dit_block_noalloc_max_bytes() -> int:
    return lib().dit_block_noalloc_max_bytes()


def dit_euler_step(x, vel, sigma: float, sigma_next: float, stream=None):
    import torch
    _ok(lib().dit_euler_step(_ptr(x, torch.float32, "x"), _ptr(vel, torch.float32, "vel"), x.numel(), sigma,
                             sigma_next, _stream(stream)), "dit_euler_step")


def dit_rope_tables(L: int, grid_h: int, grid_w: int, head_dim: int, cos, sin, theta: float = 10000.0,
                    stream=None):
    import torch
    _ok(lib().dit_rope_tables(L, grid_h, grid_w, head_dim, theta, _ptr(cos, torch.float32, "cos"),
                              _ptr(sin, torch.float32, "sin"), _stream(stream)), "dit_rope_tables")


def dit_denoise(model: DenoiseModel, img_tokens, txt_feats, sigmas: Sequence[float], txt_cos, txt_sin, img_cos,
                img_sin, ws, stream=None):
    import torch
    f32 = torch.float32
    steps = len(sigmas) - 1
    sig = (c_float * len(sigmas))(*[float(s) for s in sigmas])
    L = 0 if txt_feats is None else txt_feats.shape[0]
    _ok(lib().dit_denoise(ctypes.byref(model.c), _ptr(img_tokens, f32, "img_tokens"), img_tokens.shape[0],
                          _ptr(txt_feats, f32, "txt_feats"), L, sig, steps, _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                          _ptr(img_cos, f32), _ptr(img_sin, f32), _ptr(ws, None, "ws"),
                          ws.numel() * ws.element_size(), _stream(stream)), "dit_denoise")


def dit_modnorm(dims: DitDims, txt, img, w, mod: Modulation, which: int, h, stream=None):
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_modnorm(ctypes.byref(dims.c), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"), img.shape[0],
                          _ptr(w, f32, "w"), ctypes.byref(mod.c), which, _ptr(h, _bf16(), "h"), _stream(stream)),
        "dit_modnorm")


def dit_stream_k_workspace_bytes() -> int:
    return lib().dit_stream_k_workspace_bytes()


def _ws_bytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def dit_qkv_rope(dims: DitDims, h, L: int, N: int, wqkv, q_norm, k_norm, txt_cos, txt_sin, img_cos, img_sin,
                 q, k, vt, ws=None, stream=None):
    import torch
    f32, bf = torch.float32, _bf16()
    _ok(lib().dit_qkv_rope(ctypes.byref(dims.c), _ptr(h, bf, "h"), L, N, _ptr(wqkv, bf, "wqkv"),
                           _ptr(q_norm, f32), _ptr(k_norm, f32), _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                           _ptr(img_cos, f32), _ptr(img_sin, f32), _ptr(q, bf, "q"), _ptr(k, bf, "k"),
                           _ptr(vt, bf, "vt"), _ptr(ws), _ws_bytes(ws), _stream(stream)), "dit_qkv_rope")


def dit_attention_workspace_bytes(dims: DitDims, R: int) -> int:
    return int(lib().dit_attention_workspace_bytes(ctypes.byref(dims.c), R))


def dit_attention(dims: DitDims, R: int, q, k, vt, o, ws=None, stream=None):
    """ws: optional scratch of dit_attention_workspace_bytes (persistent schedule)."""
    bf = _bf16()
    _ok(lib().dit_attention(ctypes.byref(dims.c), R, _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(vt, bf, "vt"),
                            _ptr(o, bf, "o"), _ptr(ws), _ws_bytes(ws), _stream(stream)), "dit_attention")


def dit_attention_qknorm(dims: DitDims, R: int, q, k, vt, q_norm, k_norm, o, ws=None, stream=None):
    """dit_attention for q and k rows that are QK-RMS-normalised with q_norm / k_norm (None = ones)."""
    import torch
    bf = _bf16()
    f32 = torch.float32
    _ok(lib().dit_attention_qknorm(ctypes.byref(dims.c), R, _ptr(q, bf, "q"), _ptr(k, bf, "k"), _ptr(vt, bf, "vt"),
                                   _ptr(q_norm, f32), _ptr(k_norm, f32), _ptr(o, bf, "o"), _ptr(ws), _ws_bytes(ws),
                                   _stream(stream)),
        "dit_attention_qknorm")


def dit_linear_gated(dims: DitDims, a, L: int, N: int, w, mod: Modulation, which: int, txt, img, ws=None,
                     stream=None):
    import torch
    bf, f32 = _bf16(), torch.float32
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _ok(lib().dit_linear_gated(ctypes.byref(dims.c), _ptr(a, bf, "a"), L, N, _ptr(w, bf, "w"), ctypes.byref(mod.c),
                               which, _ptr(txt, f32, "txt"), _ptr(img, f32, "img"), _ptr(ws), ws_bytes,
                               _stream(stream)),
        "dit_linear_gated")


def dit_linear_swiglu(dims: DitDims, h2, wup, a, ws=None, stream=None):
    bf = _bf16()
    _ok(lib().dit_linear_swiglu(ctypes.byref(dims.c), _ptr(h2, bf, "h2"), h2.shape[0], _ptr(wup, bf, "wup"),
                                _ptr(a, bf, "a"), _ptr(ws), _ws_bytes(ws), _stream(stream)), "dit_linear_swiglu")


def dit_linear(a, w, out, stream=None):
    import torch
    bf = _bf16()
    M, K = a.shape
    N = w.shape[0]
    out_bf16 = 1 if out.dtype != torch.float32 else 0
    _ok(lib().dit_linear(_ptr(a, bf, "a"), M, K, _ptr(w, bf, "w"), N, _ptr(out, None, "out"), out_bf16,
                         _stream(stream)), "dit_linear")


def dit_linear_int8_workspace_bytes(N: int, K: int) -> int:
    return lib().dit_linear_int8_workspace_bytes(N, K)


def dit_block_forward_w8a8(dims: DitDims, w: W8A8BlockWeights, txt, img, txt_cos, txt_sin, img_cos, img_sin,
                           mod: Modulation, ws, stream=None):
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_block_forward_w8a8(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                     _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                     _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                     _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_block_forward_w8a8")


def dit_parallel_block_forward_w8a8(dims: DitDims, w: ParallelW8A8Weights, txt, img, txt_cos, txt_sin, img_cos,
                                    img_sin, mod: Modulation, ws, stream=None):
    """The parallel block with W8A8 linear1 / linear2; mod rows are [M, 3, H] (shift, scale, gate)."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_parallel_block_forward_w8a8(ctypes.byref(dims.c), ctypes.byref(w.c), _ptr(txt, f32, "txt"), L,
                                              _ptr(img, f32, "img"), img.shape[0], _ptr(txt_cos, f32),
                                              _ptr(txt_sin, f32), _ptr(img_cos, f32), _ptr(img_sin, f32),
                                              ctypes.byref(mod.c), _ptr(ws, None, "ws"),
                                              ws.numel() * ws.element_size(), _stream(stream)),
        "dit_parallel_block_forward_w8a8")


def dit_double_block_forward_w8a8(dims: DitDims, w_txt: Optional[W8A8BlockWeights], w_img: W8A8BlockWeights, txt,
                                  img, txt_cos, txt_sin, img_cos, img_sin, mod: Modulation, ws, stream=None):
    """The double-stream block with W8A8 linears: text rows use w_txt, image rows w_img."""
    import torch
    f32 = torch.float32
    L = 0 if txt is None else txt.shape[0]
    _ok(lib().dit_double_block_forward_w8a8(ctypes.byref(dims.c), None if w_txt is None else ctypes.byref(w_txt.c),
                                            ctypes.byref(w_img.c), _ptr(txt, f32, "txt"), L, _ptr(img, f32, "img"),
                                            img.shape[0], _ptr(txt_cos, f32), _ptr(txt_sin, f32),
                                            _ptr(img_cos, f32), _ptr(img_sin, f32), ctypes.byref(mod.c),
                                            _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_double_block_forward_w8a8")


def dit_w8a8_quantize_weight(w, smooth, q, scale, stream=None):
    import torch
    N, K = w.shape
    _ok(lib().dit_w8a8_quantize_weight(_ptr(w, _bf16(), "w"), N, K, _ptr(smooth, torch.float32, "smooth"),
                                       _ptr(q, torch.int8, "q"), _ptr(scale, torch.float32, "scale"), _stream(stream)),
        "dit_w8a8_quantize_weight")


def dit_w8a8_quantize_rows(x, smooth, scale, stream=None):
    """Per-token codes of x (bf16 [R, K]) written over x; scale [R] fp32."""
    import torch
    R, K = x.shape
    _ok(lib().dit_w8a8_quantize_rows(_ptr(x, _bf16(), "x"), R, K, _ptr(smooth, torch.float32, "smooth"),
                                     _ptr(scale, torch.float32, "scale"), _stream(stream)), "dit_w8a8_quantize_rows")


def dit_linear_w8a8_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().dit_linear_w8a8_workspace_bytes(M, N, K)


def dit_linear_w8a8(a, q, scale, smooth, out, ws, stream=None):
    import torch
    M, K = a.shape
    N = q.shape[0]
    _ok(lib().dit_linear_w8a8(_ptr(a, _bf16(), "a"), M, K, _ptr(q, torch.int8, "q"), _ptr(scale, torch.float32, "scale"),
                              _ptr(smooth, torch.float32, "smooth"), N, _ptr(out, torch.float32, "out"),
                              _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "dit_linear_w8a8")


def dit_linear_int8(a, wq, wscale, out, ws, stream=None):
    import torch
    M, K = a.shape
    N = wq.shape[0]
    _ok(lib().dit_linear_int8(_ptr(a, _bf16(), "a"), M, K, _ptr(wq, torch.int8, "wq"), _ptr(wscale, _bf16(), "s"), N,
                              _ptr(out, torch.float32, "out"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                              _stream(stream)), "dit_linear_int8")


def dit_dequant_int8(q, s, w, stream=None):
    import torch
    rows, cols = q.shape
    _ok(lib().dit_dequant_int8(_ptr(q, torch.int8, "q"), _ptr(s, _bf16(), "s"), rows, cols, _ptr(w, _bf16(), "w"),
                               _stream(stream)), "dit_dequant_int8")


def dit_selftest_bounded_wait(complete: bool, stream=None):
    """Launch the bounded-wait diagnostic; dit_check() afterwards raises DIT_ETIMEOUT unless complete."""
    _ok(lib().dit_selftest_bounded_wait(1 if complete else 0, _stream(stream)), "dit_selftest_bounded_wait")


def dit_check(stream=None):
    _ok(lib().dit_check(_stream(stream)), "dit_check")
