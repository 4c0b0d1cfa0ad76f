"""The split-halves partial rotary layout (dims.rope_split = 1) through the C ABI against the float64
oracle [gizai:dit, prepOf, HEAD]: the QKV epilogue alone (q, k, v element by element) and the three
block forms with the gates of the block tests. The tables are inputs ([rows, 3d/8]); here they
hold seeded angles."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_f64, block_weights_dev, dev, dev_bf16, modulation_dev, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _dims(sh):
    return D.DitDims(sh.hidden, sh.heads, sh.head_dim, sh.ffn, sh.eps, sh.qk_eps, rope_split=True)


def _tables(sh, seed):
    g = np.random.default_rng(seed)
    ang = g.uniform(-20.0, 20.0, size=(sh.R, 3 * sh.head_dim // 8))
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _tables_dev(sh, cos, sin):
    L = sh.L
    return dev(cos[:L]), dev(sin[:L]), dev(cos[L:]), dev(sin[L:])


@pytest.mark.parametrize("shape,nw", [("tiny", True), ("512sq", False)])
def test_qkv_epilogue_split_halves(shape, nw):
    inp = DI.block_inputs(shape, norm_weights=nw)
    sh = inp.shape
    R, H, nh, d = sh.R, sh.hidden, sh.heads, sh.head_dim
    g = np.random.default_rng(9)
    h = DI.bf16_bits_from_f32(g.standard_normal((R, H), dtype=np.float32))
    cos, sin = _tables(sh, 1)
    q = torch.empty(nh, R, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty_like(q)
    vt = torch.zeros(nh, d, D.dit_vt_stride(R), dtype=torch.bfloat16, device="cuda")
    qn = None if inp.q_norm is None else dev(inp.q_norm)
    kn = None if inp.k_norm is None else dev(inp.k_norm)
    D.dit_qkv_rope(_dims(sh), dev_bf16(h), sh.L, sh.N, dev_bf16(inp.wqkv), qn, kn, *_tables_dev(sh, cos, sin), q, k, vt)
    D.dit_check()
    qkv = O.bf16_to_f64(h) @ O.bf16_to_f64(inp.wqkv).T
    c64, s64 = cos.astype(np.float64), sin.astype(np.float64)
    rq = O.rope_apply_split(O.qk_rmsnorm(qkv[:, :H].reshape(R, nh, d), inp.q_norm, sh.qk_eps), c64, s64)
    rk = O.rope_apply_split(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(R, nh, d), inp.k_norm, sh.qk_eps), c64, s64)
    rv = qkv[:, 2 * H:].reshape(R, nh, d)
    np.testing.assert_allclose(bf16_f64(q), rq.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
    np.testing.assert_allclose(bf16_f64(k), rk.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
    np.testing.assert_allclose(bf16_f64(vt)[:, :, :R], rv.transpose(1, 2, 0), rtol=2 ** -8, atol=1e-4)


def _run(kind, inp, cos, sin, txt_w=None):
    sh = inp.shape
    dims = _dims(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tabs = _tables_dev(sh, cos, sin)
    variant = {"seq": 0, "par": 2, "dbl": 3}[kind]
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, variant))
    if kind == "seq":
        D.dit_block_forward(dims, block_weights_dev(inp), txt, img, *tabs, modulation_dev(inp), ws)
    elif kind == "par":
        D.dit_parallel_block_forward(dims, block_weights_dev(inp), txt, img, *tabs, modulation_dev(inp), ws)
    else:
        D.dit_double_block_forward(dims, block_weights_dev(txt_w), block_weights_dev(inp), txt, img, *tabs,
                                   modulation_dev(inp), ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


def _oracle(kind, inp, cos, sin, rows=None, txt_w=None):
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    c64, s64 = cos.astype(np.float64), sin.astype(np.float64)
    W = O.block_weights_f64(inp)
    if kind == "seq":
        return O.block_forward_rows(x, W, inp.mod, inp.mod_map, c64, s64, sh.heads, sh.head_dim, rows=rows,
                                    norm1=inp.norm1, norm2=inp.norm2, q_norm=inp.q_norm, k_norm=inp.k_norm)
    if kind == "par":
        return O.parallel_block_forward_rows(x, W, inp.mod, inp.mod_map, c64, s64, sh.heads, sh.head_dim, rows=rows,
                                             norm=inp.norm1, q_norm=inp.q_norm, k_norm=inp.k_norm)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    return O.double_block_forward_rows(x, O.block_weights_f64(txt_w), W, inp.mod, inp.mod_map, c64, s64, sh.heads,
                                       sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w), norms_img=nrm(inp))


@pytest.mark.parametrize("kind", ["seq", "par", "dbl"])
@pytest.mark.parametrize("d", [64, 128])
def test_blocks_with_split_halves_rotary(kind, d):
    sh = DI.BlockShape(f"split_{kind}_{d}", 256 if d == 64 else 512, 4, d, 768, 13, 9, 10, seed=400 + d)
    gen = DI.parallel_block_inputs if kind == "par" else DI.block_inputs
    inp = gen(sh, M=2, norm_weights=True)
    tw = DI.block_inputs(sh, norm_weights=True, seed=sh.seed + 50) if kind == "dbl" else None
    cos, sin = _tables(sh, 2)
    got = _run(kind, inp, cos, sin, tw)
    ref = _oracle(kind, inp, cos, sin, txt_w=tw)
    _check(got, ref, np.concatenate([inp.txt, inp.img]).astype(np.float64), f"split rotary {kind} d={d}")


def test_block_1024sq_split_halves_sampled_rows():
    inp = DI.block_inputs("1024sq")
    sh = inp.shape
    cos, sin = _tables(sh, 3)
    got = _run("seq", inp, cos, sin)
    rows = _sample_rows(sh, seed=17)
    ref = _oracle("seq", inp, cos, sin, rows=rows)
    _check(got[rows], ref, np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows], "split rotary 1024sq")
