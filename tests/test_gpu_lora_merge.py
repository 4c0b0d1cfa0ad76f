"""The LoRA merge through the C ABI (dit_lora_merge) [gizai:dit, weightAt and loadBlock: a BF16
block is loaded with each adapter's update added, W + B A], against the exact merged weight:
* bit for bit where every partial sum is exact in fp32 (small dyadic values);
* otherwise each element lies between the bf16 roundings of the exact value minus and plus the fp32
  sum's error bound (the fp32 value lies in that interval and the rounding is monotone), and almost
  all elements are the bf16 rounding of the exact value itself;
* in place (merged = W) equal to out of place;
* the parallel and double-stream blocks on merged weights against the oracle's blocks on the exact
  merged weights (oracle.lora_merge), with the bf16 blocks' gates."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_bits, dev, dev_bf16, dims_of, modulation_dev, opt_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _bf16_rne_f64(x):
    """Round float64 values to bfloat16 (8 significant bits), nearest with ties to even; float64 out."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def _merge_gpu(W, A, B, in_place=False):
    w = dev_bf16(W)
    out = w if in_place else torch.empty_like(w)
    D.dit_lora_merge(w, dev_bf16(A), dev_bf16(B), out)
    D.dit_check()
    return O.bf16_to_f64(bf16_bits(out))


def _rand_bf16(g, shape, std):
    return DI.bf16_bits_from_f32((g.standard_normal(shape) * std).astype(np.float32))


@pytest.mark.parametrize("n_out,n_in,rank", [(1, 1, 1), (100, 72, 8), (130, 257, 24), (3072, 3072, 64)])
def test_merge_bit_exact_on_exact_sums(n_out, n_in, rank):
    g = np.random.default_rng(n_out + n_in + rank)
    # W = k / 64, A = a / 8, B = b / 8 with small integers: every partial sum is a multiple of 1/64
    # below 2^10, exact in fp32, so the one rounding is the bf16 one
    W = DI.bf16_bits_from_f32((g.integers(-64, 65, (n_out, n_in)) / 64.0).astype(np.float32))
    A = DI.bf16_bits_from_f32((g.integers(-8, 9, (rank, n_in)) / 8.0).astype(np.float32))
    B = DI.bf16_bits_from_f32((g.integers(-8, 9, (n_out, rank)) / 8.0).astype(np.float32))
    exact = O.lora_merge(O.bf16_to_f64(W), O.bf16_to_f64(A), O.bf16_to_f64(B))
    np.testing.assert_array_equal(_merge_gpu(W, A, B), _bf16_rne_f64(exact))


@pytest.mark.parametrize("n_out,n_in,rank", [(333, 200, 16), (3072, 3072, 64), (24576, 3072, 64), (512, 1024, 1024)])
def test_merge_random_within_one_rounding(n_out, n_in, rank):
    g = np.random.default_rng(7 * n_out + n_in + rank)
    W = _rand_bf16(g, (n_out, n_in), 0.02)
    A = _rand_bf16(g, (rank, n_in), 0.02)
    B = _rand_bf16(g, (n_out, rank), 0.02)
    Wf, Af, Bf = O.bf16_to_f64(W), O.bf16_to_f64(A), O.bf16_to_f64(B)
    exact = O.lora_merge(Wf, Af, Bf)
    bound = 2.0 * (rank + 2) * 2.0 ** -24 * (np.abs(Wf) + np.abs(Bf) @ np.abs(Af))
    got = _merge_gpu(W, A, B)
    # the fp32 value lies in [exact - bound, exact + bound] and the rounding is monotone
    ok = (got >= _bf16_rne_f64(exact - bound)) & (got <= _bf16_rne_f64(exact + bound))
    assert ok.all(), int((~ok).sum())
    assert np.mean(got == _bf16_rne_f64(exact)) >= 0.999


def test_merge_in_place_equals_out_of_place():
    g = np.random.default_rng(3)
    W, A, B = _rand_bf16(g, (768, 256), 0.02), _rand_bf16(g, (64, 256), 0.02), _rand_bf16(g, (768, 64), 0.02)
    np.testing.assert_array_equal(_merge_gpu(W, A, B, in_place=True), _merge_gpu(W, A, B))


# ------------------------------------------------------------------ blocks on merged weights

def _adapters(inp, rank, seed):
    g = np.random.default_rng(seed)
    W = (inp.wqkv, inp.wout, inp.wup, inp.wdown)
    return [(_rand_bf16(g, (rank, w.shape[1]), 0.02), _rand_bf16(g, (w.shape[0], rank), 0.02)) for w in W]


def _merged_dev(inp, ad):
    out = []
    for w, (a, b) in zip((inp.wqkv, inp.wout, inp.wup, inp.wdown), ad):
        m = dev_bf16(w)
        D.dit_lora_merge(m, dev_bf16(a), dev_bf16(b), m)
        out.append(m)
    return D.BlockWeights(*out, opt_dev(inp.norm1), opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))


def _merged_f64(inp, ad):
    W = O.block_weights_f64(inp)
    return tuple(O.lora_merge(w, O.bf16_to_f64(a), O.bf16_to_f64(b)) for w, (a, b) in zip(W, ad))


@pytest.mark.parametrize("shape", ["tiny", "512sq"])
def test_parallel_block_on_merged_lora_vs_oracle(shape):
    inp = DI.parallel_block_inputs(shape, norm_weights=True)
    sh = inp.shape
    ad = _adapters(inp, 64 if sh.hidden > 256 else 16, 31)
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 2))
    D.dit_parallel_block_forward(dims, _merged_dev(inp, ad), txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    got = np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)
    rows = np.arange(sh.R) if sh.R <= 512 else _sample_rows(sh, seed=33)
    ref = O.parallel_block_forward(inp, weights=_merged_f64(inp, ad), rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x_in, f"parallel block, merged LoRA, {shape}")


def test_double_block_on_merged_lora_vs_oracle():
    inp = DI.block_inputs("tiny", norm_weights=True)
    tw = DI.block_inputs("tiny", norm_weights=True, seed=inp.shape.seed + 50)
    sh = inp.shape
    ad_i, ad_t = _adapters(inp, 16, 41), _adapters(tw, 16, 42)
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 3))
    D.dit_double_block_forward(dims, _merged_dev(tw, ad_t), _merged_dev(inp, ad_i), txt, img, tc, ts, ic, is_,
                               modulation_dev(inp), ws)
    D.dit_check()
    got = np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_rows(x, _merged_f64(tw, ad_t), _merged_f64(inp, ad_i), inp.mod, inp.mod_map, cos,
                                      sin, sh.heads, sh.head_dim, sh.L, norms_txt=nrm(tw), norms_img=nrm(inp),
                                      eps=sh.eps, qk_eps=sh.qk_eps)
    _check(got, ref, x, "double-stream block, merged LoRA, tiny")
