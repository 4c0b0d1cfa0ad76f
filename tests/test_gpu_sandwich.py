"""The sandwich block (post-norms before the gates) through the C ABI against the float64 oracle
[gizai:dit, POST_ATTN, POST_MLP], with the gates of the block tests."""

import numpy as np
import pytest

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import block_weights_dev, dev, dims_of, modulation_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _posts(sh, which, seed=0):
    g = np.random.default_rng(seed)
    mk = lambda: (1 + 0.2 * g.standard_normal(sh.hidden)).astype(np.float32)
    pa, pm = mk(), mk()
    return (pa if "a" in which else None), (pm if "m" in which else None)


def _run(inp, pa, pm):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 0))
    D.dit_block_forward_sandwich(dims, block_weights_dev(inp), None if pa is None else dev(pa),
                                 None if pm is None else dev(pm), txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


def _oracle(inp, pa, pm, rows=None):
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    return O.block_forward_rows(x, O.block_weights_f64(inp), inp.mod, inp.mod_map, cos, sin, sh.heads, sh.head_dim,
                                rows=rows, norm1=inp.norm1, norm2=inp.norm2, q_norm=inp.q_norm, k_norm=inp.k_norm,
                                eps=sh.eps, qk_eps=sh.qk_eps, post_attn=pa, post_mlp=pm)


@pytest.mark.parametrize("which", ["am", "a", "m"])
def test_sandwich_tiny_all_rows(which):
    inp = DI.block_inputs("tiny", M=2, norm_weights=True)
    pa, pm = _posts(inp.shape, which)
    got = _run(inp, pa, pm)
    ref = _oracle(inp, pa, pm)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(got, ref, x, f"sandwich tiny ({which})")
    plain = _oracle(inp, None, None)
    assert np.sqrt(np.mean((ref - plain) ** 2)) > 0.1 * np.sqrt(np.mean((ref - x) ** 2))  # the norms matter


def test_sandwich_head64_ragged():
    sh = DI.BlockShape("sw64", 256, 4, 64, 768, 13, 9, 10, seed=91)
    inp = DI.block_inputs(sh, M=2)
    pa, pm = _posts(sh, "am", seed=1)
    got = _run(inp, pa, pm)
    _check(got, _oracle(inp, pa, pm), np.concatenate([inp.txt, inp.img]).astype(np.float64), "sandwich d=64 ragged")


@pytest.mark.parametrize("shape", ["512sq", "1024sq"])
def test_sandwich_sampled_rows(shape):
    inp = DI.block_inputs(shape)
    pa, pm = _posts(inp.shape, "am", seed=2)
    got = _run(inp, pa, pm)
    rows = _sample_rows(inp.shape, seed=23)
    ref = _oracle(inp, pa, pm, rows=rows)
    _check(got[rows], ref, np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows], f"sandwich {shape}")
