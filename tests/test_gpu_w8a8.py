"""Parity of the W8A8 path through the C ABI against the oracle (oracle/w8a8.py) [klein, section 5
and its D4/D5 entries]: the quantisers bit for bit (codes and float32 scales, with and without the
SmoothQuant divisor), one W8A8 linear within float32 rounding of the exact integer product, and the
whole W8A8 block (tiny, 512sq and 1024sq sampled rows).

Block gates. An activation entering a W8A8 linear is rounded to bf16 and quantised with step
s = max|x| / 127; wherever the GPU's and the oracle's activation differ (they do at the bf16 level
downstream of the attention, whose GPU output carries the bf16 path's ~2^-9 relative error), a code
may differ by one step. With codes of RMS ~127/4 ~ 32 for Gaussian-like rows, a fraction p of
flipped codes moves the linear's output by ~sqrt(p) / 32 of its RMS: up to ~3 % RMS for p = 1.
* MLP branch alone (the attention gate zeroed): its linears' inputs come from the norm and agree to
  fp32 rounding, so the bf16 block's gates of test_gpu_block apply;
* whole block: RMS(delta error) <= 4e-2 RMS(delta) and max |out error| <= 1e-1 RMS(out)."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import (bf16_bits, dev, dev_bf16, dims_of, max_abs, modulation_dev, opt_dev, rms, rope_dev,
                            workspace)
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _bf16_rand(g, shape, std):
    return DI.bf16_bits_from_f32((g.standard_normal(shape) * std).astype(np.float32))


@pytest.mark.parametrize("R,K,smooth", [(5, 256, False), (77, 3072, True), (300, 12288, False), (33, 768, True)])
def test_quantize_rows_bit_exact(R, K, smooth):
    g = np.random.default_rng(R + K)
    x = _bf16_rand(g, (R, K), 1.0)
    x[R // 2] = 0  # a zero row: scale 0, codes 0
    sm = g.uniform(0.5, 2.0, size=K).astype(np.float32) if smooth else None
    xd = dev_bf16(x)
    sc = torch.empty(R, dtype=torch.float32, device="cuda")
    D.dit_w8a8_quantize_rows(xd, opt_dev(sm), sc)
    D.dit_check()
    q_ref, s_ref = O.quantize_rows(O.bf16_to_f64(x).astype(np.float32), sm)
    got_codes = O.bf16_to_f64(bf16_bits(xd))
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(got_codes, q_ref.astype(np.float64))


@pytest.mark.parametrize("N,K,smooth", [(64, 256, False), (384, 3072, True), (3072, 12288, False)])
def test_quantize_weight_bit_exact(N, K, smooth):
    g = np.random.default_rng(N * 3 + K)
    w = _bf16_rand(g, (N, K), 0.02)
    sm = g.uniform(0.5, 2.0, size=K).astype(np.float32) if smooth else None
    q = torch.empty(N, K, dtype=torch.int8, device="cuda")
    sc = torch.empty(N, dtype=torch.float32, device="cuda")
    D.dit_w8a8_quantize_weight(dev_bf16(w), opt_dev(sm), q, sc)
    D.dit_check()
    q_ref, s_ref = O.quantize_weight(O.bf16_to_f64(w).astype(np.float32), sm)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)


@pytest.mark.parametrize("M,N,K,smooth", [(72, 256, 256, False), (333, 512, 1024, True), (1088, 768, 3072, False),
                                          (4224, 256, 12288, True)])
def test_linear_w8a8(M, N, K, smooth):
    g = np.random.default_rng(M + N + K)
    a = _bf16_rand(g, (M, K), 1.0)
    w = _bf16_rand(g, (N, K), 0.02)
    sm = g.uniform(0.5, 2.0, size=K).astype(np.float32) if smooth else None
    qw, sw = O.quantize_weight(O.bf16_to_f64(w).astype(np.float32), sm)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ad = dev_bf16(a)
    D.dit_linear_w8a8(ad, dev(qw), dev(sw), opt_dev(sm), out, workspace(D.dit_linear_w8a8_workspace_bytes(M, N, K)))
    D.dit_check()
    assert np.array_equal(bf16_bits(ad), a)  # the input is not modified
    qa, sa = O.quantize_rows(O.bf16_to_f64(a).astype(np.float32), sm)
    ref = O.w8a8_linear(qa, sa, qw, sw)
    # the products are exact in fp32; the accumulation is exact while partial sums stay below 2^24,
    # and in any case within fp32 rounding of sum |qa| |qw|; the two scalings round once each
    bound = (np.abs(qa.astype(np.float64)) @ np.abs(qw.astype(np.float64)).T) * sa[:, None].astype(np.float64) * \
        sw[None, :].astype(np.float64)
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 2 ** -22 * np.abs(ref) + 2 ** -22 * bound + 1e-30), float((err / (bound + 1e-30)).max())


def _w8a8_case(shape, smooth, seed=7):
    inp = DI.block_inputs(shape, norm_weights=True)
    sh = inp.shape
    g = np.random.default_rng(seed)
    ins = [sh.hidden, sh.hidden, sh.hidden, sh.ffn]
    sm = [g.uniform(0.5, 2.0, size=k).astype(np.float32) for k in ins] if smooth else [None] * 4
    qws = [O.quantize_weight(O.bf16_to_f64(W).astype(np.float32), s)
           for W, s in zip((inp.wqkv, inp.wout, inp.wup, inp.wdown), sm)]
    return inp, qws, sm


def _run_w8a8_gpu(inp, qws, sm):
    sh = inp.shape
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    w = D.W8A8BlockWeights([dev(q) for q, _ in qws], [dev(s) for _, s in qws], [opt_dev(s) for s in sm],
                           opt_dev(inp.norm1), opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 4))
    D.dit_block_forward_w8a8(dims, w, txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    return np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)


def _oracle_w8a8(inp, qws, sm, rows=None):
    sh = inp.shape
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    return O.block_forward_w8a8_rows(x, qws, inp.mod, inp.mod_map, cos, sin, sh.heads, sh.head_dim, rows=rows,
                                     norm1=inp.norm1, norm2=inp.norm2, q_norm=inp.q_norm, k_norm=inp.k_norm,
                                     eps=sh.eps, qk_eps=sh.qk_eps, smooth=None if sm[0] is None else sm)


def _check_w8a8(got, ref, x_in, label):
    d_got, d_ref = got - x_in, ref - x_in
    e_out = max_abs(got, ref) / rms(ref)
    e_rms = rms(d_got - d_ref) / rms(d_ref)
    print(f"{label}: max|out err|/RMS(out) = {e_out:.3e}; delta: RMS err {e_rms:.3e}")
    assert e_rms <= 4e-2, label
    assert e_out <= 1e-1, label


@pytest.mark.parametrize("smooth", [False, True])
def test_w8a8_block_tiny_all_rows(smooth):
    inp, qws, sm = _w8a8_case("tiny", smooth)
    got = _run_w8a8_gpu(inp, qws, sm)
    ref = _oracle_w8a8(inp, qws, sm)
    _check_w8a8(got, ref, np.concatenate([inp.txt, inp.img]).astype(np.float64), f"w8a8 tiny smooth={smooth}")


@pytest.mark.parametrize("shape,smooth", [("512sq", True), ("1024sq", False)])
def test_w8a8_block_sampled_rows(shape, smooth):
    inp, qws, sm = _w8a8_case(shape, smooth)
    sh = inp.shape
    got = _run_w8a8_gpu(inp, qws, sm)
    rows = _sample_rows(sh, seed=17)
    ref = _oracle_w8a8(inp, qws, sm, rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check_w8a8(got[rows], ref, x_in, f"w8a8 {shape} sampled rows smooth={smooth}")


@pytest.mark.parametrize("shape,smooth", [("tiny", True), ("512sq", False), ("512sq", True)])
def test_w8a8_mlp_branch_within_the_bf16_gates(shape, smooth):
    inp, qws, sm = _w8a8_case(shape, smooth)
    inp.mod[:, 2, :] = 0.0  # attention gate: x reaches the second norm unchanged
    sh = inp.shape
    got = _run_w8a8_gpu(inp, qws, sm)
    rows = _sample_rows(sh, seed=19) if sh.R > 512 else np.arange(sh.R)
    ref = _oracle_w8a8(inp, qws, sm, rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x_in, f"w8a8 MLP branch {shape} smooth={smooth}")


def test_w8a8_block_deterministic():
    inp, qws, sm = _w8a8_case("512sq", True)
    a = _run_w8a8_gpu(inp, qws, sm)
    b = _run_w8a8_gpu(inp, qws, sm)
    assert np.array_equal(a, b)
