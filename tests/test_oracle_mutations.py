"""Planted mistakes in the oracle (on the CPU) must each fail a pin.

Each case replaces one oracle function with a plausible wrong variant and reruns the scalar
brute-force comparison; a pin set that let any of them through would not pin the oracle."""

import math

import numpy as np
import pytest

import oracle.dit as OD
from tests import test_oracle_block as TB


def _mod_plain_scale(x, w, shift, scale, eps):
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    if w is not None:
        y = y * w
    return y * scale + shift


def _mod_no_eps(x, w, shift, scale, eps):
    return OD.__dict__["_orig_modnorm"](x, w, shift, scale, 0.0)


def _rope_sign(t, cos, sin):
    return OD.__dict__["_orig_rope"](t, cos, -np.asarray(sin))


def _rope_halves(t, cos, sin):
    d = t.shape[-1]
    c = np.asarray(cos)[:, None, :]
    s = np.asarray(sin)[:, None, :]
    a, b = t[..., : d // 2], t[..., d // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _attn_no_scale(q, k, v, rows=None):
    return OD.__dict__["_orig_attn"](q * math.sqrt(q.shape[-1]), k, v, rows)


def _glu_swapped(u):
    return OD.silu(u[..., 1::2]) * u[..., 0::2]


def _qk_no_eps(t, w, eps):
    return OD.__dict__["_orig_qk"](t, w, 0.0)


MUTATIONS = [
    ("modulated_rmsnorm", _mod_plain_scale),
    ("modulated_rmsnorm", _mod_no_eps),
    ("rope_apply", _rope_sign),
    ("rope_apply", _rope_halves),
    ("attention", _attn_no_scale),
    ("swiglu_interleaved", _glu_swapped),
    ("qk_rmsnorm", _qk_no_eps),
]


@pytest.mark.parametrize("name,fn", MUTATIONS, ids=[f"{n}:{f.__name__}" for n, f in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn):
    OD._orig_modnorm = OD.modulated_rmsnorm
    OD._orig_rope = OD.rope_apply
    OD._orig_attn = OD.attention
    OD._orig_qk = OD.qk_rmsnorm
    monkeypatch.setattr(OD, name, fn)
    with pytest.raises(AssertionError):
        TB.test_block_matches_scalar_brute_force(0, None)


# ------------------------------------------------------------------ quantisation: W8A8 and int8lin

import oracle as O  # noqa: E402
import oracle.w8a8 as OW  # noqa: E402
from tests import test_oracle_sampler as TS  # noqa: E402
from tests import test_oracle_w8a8 as TW  # noqa: E402

_orig_codes = OW.quantize_codes
_orig_rows = OW.quantize_rows
_orig_dequant = OD.dequant_int8


def _codes_half_away(v32, scale32):
    v = np.asarray(v32, np.float32)
    s = np.asarray(scale32, np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        x = v / s
        r = np.sign(x) * np.floor(np.abs(x) + np.float32(0.5))  # ties away from zero
    r = np.where(s == 0, np.float32(0), r)
    return np.clip(r, -127, 127).astype(np.int8)


def _codes_clip_128(v32, scale32):
    v = np.asarray(v32, np.float32)
    s = np.asarray(scale32, np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(v / s)
    r = np.where(s == 0, np.float32(0), r)
    return np.clip(r, -128, 127).astype(np.int8)


def _rows_over_128(x32, smooth=None):
    x = np.asarray(x32, np.float32)
    if smooth is not None:
        x = (x / np.asarray(smooth, np.float32)[None, :]).astype(np.float32)
    scale = (np.max(np.abs(x), axis=1) / np.float32(128)).astype(np.float32)
    return _orig_codes(x, scale[:, None]), scale


def _linear_f64_activation(x, qw, sw, smooth=None):
    # the activation quantised from its float64 value instead of its bfloat16 value
    qx, sx = _orig_rows(np.asarray(x, np.float64).astype(np.float32), smooth)
    return OW.w8a8_linear(qx, sx, qw, sw)


def _dequant_truncating(q, s_bits):
    s = OD.bf16_to_f64(s_bits)
    prod = (q.astype(np.float64) * np.repeat(s, 32, axis=1)).astype(np.float32)
    return (prod.view(np.uint32) >> 16).astype(np.uint16)  # truncation instead of nearest-even


QUANT_MUTATIONS = [
    (OW, "quantize_codes", _codes_half_away, lambda: TW.test_codes_round_half_to_even_and_clip()),
    (OW, "quantize_codes", _codes_clip_128, lambda: TW.test_codes_round_half_to_even_and_clip()),
    (OW, "quantize_rows", _rows_over_128, lambda: TW.test_rows_scale_is_absmax_over_127_and_error_is_half_a_step()),
    (OW, "w8a8_linear_f", _linear_f64_activation, lambda: TW.test_w8a8_block_matches_scalar_brute_force(0, False)),
    (OD, "dequant_int8", _dequant_truncating, lambda: TS.test_dequant_definition_and_block_index()),
]


@pytest.mark.parametrize("mod,name,fn,pin", QUANT_MUTATIONS,
                         ids=[f"{n}:{f.__name__}" for _, n, f, _ in QUANT_MUTATIONS])
def test_planted_quantisation_mistake_is_caught(monkeypatch, mod, name, fn, pin):
    monkeypatch.setattr(mod, name, fn)
    monkeypatch.setattr(O, name, fn)  # the package re-exports the same name
    with pytest.raises(AssertionError):
        pin()
