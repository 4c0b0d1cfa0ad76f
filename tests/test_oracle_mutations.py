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
