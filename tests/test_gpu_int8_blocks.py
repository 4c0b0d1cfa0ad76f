"""Parity of the int8lin parallel and double-stream blocks through the C ABI
(dit_parallel_block_forward_int8, dit_double_block_forward_int8) [host contract, section 1 (int8
weights, W = bf16_rne(q s) with one bf16 scale per 32 inputs); gizai:dit, Block.parallel; klein
article, sections 4.3-4.4 (double blocks)]:
* against the float64 oracle run on the dequantised weights (oracle.dequant_int8, itself pinned
  bit for bit), with the gates of the bf16 blocks;
* bit for bit against the bf16 blocks run on dit_dequant_int8 of the same weights: the int8lin
  blocks dequantise once and then run the same GEMMs on the same bf16 operands."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import dev, dev_bf16, dims_of, int8_weights_dev, modulation_dev, opt_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu

SHAPE64 = lambda L, gh, gw, seed: DI.BlockShape(f"i8d64_{L}_{gh}x{gw}", 256, 4, 64, 768, L, gh, gw, seed=seed)


def _with_norms(inp, seed):
    g = np.random.default_rng(seed)
    H, d = inp.shape.hidden, inp.shape.head_dim
    inp.norm1 = (1 + 0.02 * g.standard_normal(H)).astype(np.float32)
    inp.norm2 = (1 + 0.02 * g.standard_normal(H)).astype(np.float32)
    inp.q_norm = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
    inp.k_norm = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
    return inp


def _deq_f64(inp):
    return tuple(O.bf16_to_f64(O.dequant_int8(q, s)) for q, s in zip(inp.q8, inp.s8))


def _deq_dev(inp):
    """dit_dequant_int8 of the four linears: the bf16 weights (BlockWeights) the int8lin blocks stand for."""
    out = []
    for q, s in zip(inp.q8, inp.s8):
        w = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
        D.dit_dequant_int8(dev(q), dev_bf16(s), w)
        out.append(w)
    return D.BlockWeights(*out, opt_dev(inp.norm1), opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))


def _rows_out(txt, img, sh):
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


# ------------------------------------------------------------------------------------- parallel

def run_parallel_int8(inp, int8=True):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    mod = modulation_dev(inp)
    if int8:
        ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 5))
        D.dit_parallel_block_forward_int8(dims, int8_weights_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    else:
        ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 2))
        D.dit_parallel_block_forward(dims, _deq_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    D.dit_check()
    return _rows_out(txt, img, sh)


@pytest.mark.parametrize("M,nw", [(None, False), (2, True)])
def test_int8_parallel_tiny_vs_oracle(M, nw):
    inp = DI.int8_parallel_block_inputs("tiny", M=M, seed=5)
    if nw:
        _with_norms(inp, 15)
    got = run_parallel_int8(inp)
    rt, ri = O.parallel_block_forward(inp, weights=_deq_f64(inp))
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(got, np.concatenate([rt, ri]), x_in, f"int8 parallel tiny M={M} norm_weights={nw}")


@pytest.mark.parametrize("shape", ["tiny", "512sq", "1024sq_int8"])
def test_int8_parallel_bitwise_equals_bf16_on_dequantized_weights(shape):
    inp = _with_norms(DI.int8_parallel_block_inputs(shape, seed=6), 16)
    assert np.array_equal(run_parallel_int8(inp), run_parallel_int8(inp, int8=False))


def test_int8_parallel_full_size_sampled_rows():
    inp = DI.int8_parallel_block_inputs("1024sq_int8")
    sh = inp.shape
    got = run_parallel_int8(inp)
    rows = _sample_rows(sh, seed=21)
    ref = O.parallel_block_forward(inp, weights=_deq_f64(inp), rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x_in, "int8 parallel 1024sq sampled rows")


# -------------------------------------------------------------------------------- double-stream

def _double_inputs(shape, seed, nw=False, M=None):
    img = DI.int8_block_inputs(shape, M=M, seed=seed)
    txt_w = DI.int8_block_inputs(shape, seed=seed + 50)
    if nw:
        _with_norms(img, seed + 1)
        _with_norms(txt_w, seed + 2)
    return img, txt_w


def run_double_int8(inp, txt_w, int8=True):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    mod = modulation_dev(inp)
    if int8:
        ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 6))
        wt = int8_weights_dev(txt_w) if sh.L > 0 else None
        D.dit_double_block_forward_int8(dims, wt, int8_weights_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    else:
        ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 3))
        wt = _deq_dev(txt_w) if sh.L > 0 else None
        D.dit_double_block_forward(dims, wt, _deq_dev(inp), txt, img, tc, ts, ic, is_, mod, ws)
    D.dit_check()
    return _rows_out(txt, img, sh)


def oracle_double_int8(inp, txt_w, rows=None):
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    return O.double_block_forward_rows(x, _deq_f64(txt_w), _deq_f64(inp), inp.mod, inp.mod_map, cos, sin, sh.heads,
                                       sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w), norms_img=nrm(inp),
                                       eps=sh.eps, qk_eps=sh.qk_eps)


@pytest.mark.parametrize("shape,nw", [("tiny", False), ("tiny", True), (SHAPE64(13, 9, 10, 71), True),
                                      (SHAPE64(0, 9, 9, 72), False), (SHAPE64(100, 16, 20, 73), True)])
def test_int8_double_vs_oracle(shape, nw):
    # L = 13 and 100: the image rows start off a tile boundary (each stream padded to whole tiles);
    # L = 0: the image stream alone
    inp, tw = _double_inputs(shape, 7, nw=nw, M=2 if nw else None)
    got = run_double_int8(inp, tw)
    ref = oracle_double_int8(inp, tw)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(got, ref, x_in, f"int8 double {inp.shape.name} norm_weights={nw}")


@pytest.mark.parametrize("shape", ["tiny", SHAPE64(0, 9, 9, 74), "512sq", "1024sq_int8"])
def test_int8_double_bitwise_equals_bf16_on_dequantized_weights(shape):
    inp, tw = _double_inputs(shape, 8, nw=True)
    assert np.array_equal(run_double_int8(inp, tw), run_double_int8(inp, tw, int8=False))


def test_int8_double_full_size_sampled_rows():
    inp, tw = _double_inputs("1024sq_int8", 3)
    sh = inp.shape
    got = run_double_int8(inp, tw)
    rows = _sample_rows(sh, seed=23)
    ref = oracle_double_int8(inp, tw, rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x_in, "int8 double 1024sq sampled rows")
