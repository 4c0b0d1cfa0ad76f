"""Parity of the double-stream block through the C ABI (dit_double_block_forward) against the
float64 oracle (text rows use the text stream's linears and norm weights, image rows the image
stream's, one joint attention), with the gates of the sequential block, plus two bitwise
reductions to dit_block_forward: no text rows, and both streams sharing their weights."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import block_weights_dev, dev, dims_of, modulation_dev, rope_dev, run_block_gpu, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _inputs(shape, M=None, norm_weights=False):
    img = DI.block_inputs(shape, M=M, norm_weights=norm_weights)
    txt_w = DI.block_inputs(shape, norm_weights=norm_weights, seed=img.shape.seed + 50)
    return img, txt_w


def run_double_gpu(inp, txt_w):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 3))
    wt = block_weights_dev(txt_w) if sh.L > 0 else None
    D.dit_double_block_forward(dims, wt, block_weights_dev(inp), txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return t, img.cpu().numpy().astype(np.float64)


def oracle_double(inp, txt_w, rows=None):
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    return O.double_block_forward_rows(x, O.block_weights_f64(txt_w), O.block_weights_f64(inp), inp.mod, inp.mod_map,
                                       cos, sin, sh.heads, sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w),
                                       norms_img=nrm(inp), eps=sh.eps, qk_eps=sh.qk_eps)


@pytest.mark.parametrize("M,nw", [(None, False), (2, True), (1, False)])
def test_double_tiny_all_rows(M, nw):
    inp, tw = _inputs("tiny", M=M, norm_weights=nw)
    t, i = run_double_gpu(inp, tw)
    ref = oracle_double(inp, tw)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, i]), ref, x_in, f"double tiny M={M} norm_weights={nw}")


@pytest.mark.parametrize("L,gh,gw", [(13, 9, 10), (1, 5, 7), (8, 16, 20), (100, 16, 20), (200, 16, 20)])
def test_double_head64_unaligned_text_rows(L, gh, gw):
    # L = 13, 1 and 100: the image stream's rows start at an offset that is not a multiple of 8; with
    # 420 and 520 rows the GEMMs run on CTA pairs (256-row tiles), each stream padded to whole tiles
    sh = DI.BlockShape(f"dd64_{L}_{gh}x{gw}", 256, 4, 64, 768, L, gh, gw, seed=L + gh + 60)
    inp, tw = _inputs(sh, M=2, norm_weights=True)
    t, i = run_double_gpu(inp, tw)
    ref = oracle_double(inp, tw)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, i]), ref, x_in, f"double d=64 L={L} grid {gh}x{gw}")


@pytest.mark.parametrize("shape", ["512sq", "1024sq"])
def test_double_sampled_rows(shape):
    inp, tw = _inputs(shape)
    sh = inp.shape
    t, i = run_double_gpu(inp, tw)
    rows = _sample_rows(sh, seed=13)
    ref = oracle_double(inp, tw, rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(np.concatenate([t, i])[rows], ref, x_in, f"double {shape} sampled rows")


def test_double_without_text_rows_is_the_sequential_block_bitwise():
    sh = DI.BlockShape("img_only_d", 256, 4, 64, 768, 0, 9, 9, seed=71)
    inp, tw = _inputs(sh)
    _, i = run_double_gpu(inp, tw)
    _, i_seq = run_block_gpu(inp)
    assert np.array_equal(i, i_seq)


def test_double_with_shared_weights_is_the_sequential_block_bitwise():
    # 512sq: fewer tiles than SMs in every linear, so no K-split; each output row then depends on
    # its own A row and the weights only, whichever launch computes it
    inp = DI.block_inputs("512sq")
    t, i = run_double_gpu(inp, inp)
    t_seq, i_seq = run_block_gpu(inp)
    assert np.array_equal(t, t_seq) and np.array_equal(i, i_seq)


def test_double_deterministic():
    inp, tw = _inputs("512sq", M=2)
    a = run_double_gpu(inp, tw)
    b = run_double_gpu(inp, tw)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_double_grouped_path_vs_oracle():
    # L = 128: each norm and linear is one launch over all rows (image weights from row 128 on; on CTA
    # pairs the text rows fill half of a padded 256-row tile); norm weights per stream
    sh = DI.BlockShape("dgrp", 256, 4, 64, 768, 128, 12, 12, seed=81)
    inp, tw = _inputs(sh, M=3, norm_weights=True)
    t, i = run_double_gpu(inp, tw)
    ref = oracle_double(inp, tw)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, i]), ref, x_in, "double, one launch per linear (L = 128)")


def test_double_grouped_path_with_shared_weights_is_the_sequential_block_bitwise():
    sh = DI.BlockShape("dgrp_shared", 256, 4, 64, 768, 128, 8, 8, seed=82)
    inp = DI.block_inputs(sh, norm_weights=True)
    t, i = run_double_gpu(inp, inp)
    t_seq, i_seq = run_block_gpu(inp)
    assert np.array_equal(t, t_seq) and np.array_equal(i, i_seq)
