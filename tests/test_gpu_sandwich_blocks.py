"""The parallel and the double-stream sandwich blocks (branch outputs RMS-normed before their gates)
through the C ABI against the float64 oracle [gizai:dit, POST_ATTN, POST_MLP; Block.parallel; klein
article, sections 4.3-4.4 (double blocks)], with the gates of the block tests. The post weights are
~1 + N(0, 0.2), so a branch normed with the wrong weight, or not normed, fails."""

import numpy as np
import pytest

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import block_weights_dev, dev, dims_of, modulation_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows
from tests.test_gpu_sandwich import _posts

pytestmark = pytest.mark.gpu

opt = lambda a: None if a is None else dev(a)


def _out(txt, img, sh):
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


@pytest.mark.parametrize("shape,which", [("tiny", "am"), ("tiny", "a"), ("tiny", "m"), ("512sq", "am")])
def test_parallel_sandwich(shape, which):
    inp = DI.parallel_block_inputs(shape, M=2 if shape == "tiny" else None, norm_weights=True)
    sh = inp.shape
    pa, pm = _posts(sh, which, seed=3)
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 2))
    D.dit_parallel_block_forward_sandwich(dims, block_weights_dev(inp), opt(pa), opt(pm), txt, img, tc, ts, ic, is_,
                                          modulation_dev(inp), ws)
    D.dit_check()
    got = _out(txt, img, sh)
    rows = np.arange(sh.R) if sh.R <= 512 else _sample_rows(sh, seed=41)
    ref = O.parallel_block_forward(inp, rows=rows, post_attn=pa, post_mlp=pm)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x, f"parallel sandwich {shape} posts {which}")


def _double_inputs(shape, L=None):
    img = DI.block_inputs(shape, M=2 if (isinstance(shape, str) and shape == "tiny") else None, norm_weights=True)
    txt_w = DI.block_inputs(shape, norm_weights=True, seed=img.shape.seed + 50)
    return img, txt_w


@pytest.mark.parametrize("shape,wt,wi", [("tiny", "am", "am"), ("tiny", "a", "m"), ("tiny", "", "am"),
                                         ("512sq", "am", "a")])
def test_double_sandwich(shape, wt, wi):
    img, txt_w = _double_inputs(shape)
    sh = img.shape
    dims = dims_of(sh)
    pt, pi = _posts(sh, wt, seed=5), _posts(sh, wi, seed=6)
    txt, xi = dev(img.txt), dev(img.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 3))
    D.dit_double_block_forward_sandwich(dims, block_weights_dev(txt_w), tuple(opt(p) for p in pt),
                                        block_weights_dev(img), tuple(opt(p) for p in pi), txt, xi, tc, ts, ic, is_,
                                        modulation_dev(img), ws)
    D.dit_check()
    got = _out(txt, xi, sh)
    rows = np.arange(sh.R) if sh.R <= 512 else _sample_rows(sh, seed=43)
    x = np.concatenate([img.txt, img.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_rows(x, O.block_weights_f64(txt_w), O.block_weights_f64(img), img.mod, img.mod_map,
                                      cos, sin, sh.heads, sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w),
                                      norms_img=nrm(img), eps=sh.eps, qk_eps=sh.qk_eps, post_txt=pt, post_img=pi)
    _check(got[rows], ref, x[rows], f"double sandwich {shape} text {wt!r} image {wi!r}")


def test_double_sandwich_no_text_rows():
    sh = DI.BlockShape("dsw_L0", 256, 4, 64, 768, 0, 8, 8, seed=45)
    img = DI.block_inputs(sh, norm_weights=True)
    dims = dims_of(sh)
    pi = _posts(sh, "am", seed=7)
    xi = dev(img.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, 0, sh.N, 3))
    D.dit_double_block_forward_sandwich(dims, None, None, block_weights_dev(img), tuple(opt(p) for p in pi), None, xi,
                                        tc, ts, ic, is_, modulation_dev(img), ws)
    D.dit_check()
    x = img.img.astype(np.float64)
    cos, sin = O.rope_tables(O.positions(0, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_rows(x, O.block_weights_f64(img), O.block_weights_f64(img), img.mod, img.mod_map,
                                      cos, sin, sh.heads, sh.head_dim, 0, norms_txt=nrm(img), norms_img=nrm(img),
                                      eps=sh.eps, qk_eps=sh.qk_eps, post_img=pi)
    _check(xi.cpu().numpy().astype(np.float64), ref, x, "double sandwich L=0")
