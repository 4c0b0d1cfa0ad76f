"""Parity of dit_denoise (the full Euler loop through the C ABI) against the float64 oracle.

Gates as for the block (max |err| <= 2e-2 RMS(out)), plus the same bar on the change the loop
makes, x0 - noise, which the noise would otherwise dominate."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import dev, dev_bf16, dims_of, max_abs, rms, rope_dev, workspace

pytestmark = pytest.mark.gpu


def _model_dev(inp, block_ws=None, w_ada=None):
    sh = inp.shape
    blocks = block_ws if block_ws is not None else [
        D.BlockWeights(dev_bf16(b.wqkv), dev_bf16(b.wout), dev_bf16(b.wup), dev_bf16(b.wdown)) for b in inp.block_w]
    w_ada_t = w_ada if w_ada is not None else dev_bf16(inp.w_ada)
    return D.DenoiseModel(dims_of(sh), dev_bf16(inp.w_in), dev_bf16(inp.w_t1), dev_bf16(inp.w_t2), w_ada_t,
                          dev_bf16(inp.w_ada_f), dev_bf16(inp.w_out), blocks, latent_channels=inp.latents.shape[1])


def _run(inp, model):
    sh = inp.shape
    x = dev(inp.latents)
    tc, ts, ic, is_ = rope_dev(sh)
    steps = len(inp.steps_sigmas) - 1
    ws = workspace(D.dit_denoise_workspace_bytes(model, sh.L, sh.N, steps))
    D.dit_denoise(model, x, dev(inp.txt_feats), [float(s) for s in inp.steps_sigmas], tc, ts, ic, is_, ws)
    D.dit_check()
    return x.cpu().numpy().astype(np.float64)


def _check(got, ref, x_T, label):
    e_out = max_abs(got, ref) / rms(ref)
    d_got, d_ref = got - x_T, ref - x_T
    e_d = max_abs(d_got, d_ref) / rms(d_ref)
    e_rms = rms(d_got - d_ref) / rms(d_ref)
    print(f"{label}: max|err|/RMS(out) {e_out:.3e}; change: max {e_d:.3e}, RMS {e_rms:.3e}")
    assert e_out <= 2e-2 and e_d <= 8e-2 and e_rms <= 2e-2, label


@pytest.mark.parametrize("blocks", [1, 32])
def test_denoise_tiny_architecture(blocks):
    sh = DI.BlockShape("tiny_denoise", 256, 4, 64, 768, 8, 8, 8, seed=4)
    inp = DI.denoise_inputs(sh, blocks=blocks)
    got = _run(inp, _model_dev(inp))
    ref = O.denoise(inp).astype(np.float64)
    _check(got, ref, inp.latents.astype(np.float64), f"tiny denoise, {blocks} blocks")


def test_denoise_512sq_architecture_two_blocks():
    sh = DI.BlockShape("512sq_denoise", 3072, 24, 128, 12288, 64, 32, 32, seed=4)
    inp = DI.denoise_inputs(sh, blocks=2)
    got = _run(inp, _model_dev(inp))
    ref = O.denoise(inp).astype(np.float64)
    _check(got, ref, inp.latents.astype(np.float64), "512sq denoise, 2 blocks")


def test_denoise_full_size_identity_blocks():
    # Full denoise workload (32 blocks, L=512, N=4096): with every block's modulation weight zero,
    # shift = scale = gate = 0 and each block returns its input exactly, whatever its linears hold;
    # the loop then reduces to patch-in, time embedding, final modulated norm, patch-out and Euler,
    # which the oracle computes at full size with zero blocks.
    inp = DI.denoise_inputs("denoise", blocks=1)
    sh = inp.shape
    gen = torch.Generator(device="cuda").manual_seed(1234)
    H, F = sh.hidden, sh.ffn
    rnd = lambda *s: (torch.randn(*s, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    blk = D.BlockWeights(rnd(3 * H, H), rnd(H, H), rnd(2 * F, H), rnd(H, F))
    w_ada = torch.zeros(32, 6 * H, H, dtype=torch.bfloat16, device="cuda")
    model = _model_dev(inp, block_ws=[blk] * 32, w_ada=w_ada)
    got = _run(inp, model)
    ref = O.denoise(inp, blocks=0).astype(np.float64)
    _check(got, ref, inp.latents.astype(np.float64), "full-size denoise, identity blocks")


def test_denoise_full_size_real_blocks():
    # The denoise workload's own sequence (L = 512 text rows + N = 4096 image rows, seed 4) through
    # the whole loop, all four Euler steps over sigmas [1, .75, .5, .25, 0], with two real blocks of
    # the 1024sq architecture: non-zero modulation weights, so every block's modulation comes from
    # the hoisted adaLN rows of its own (step, block), the blocks chain through the residual rows,
    # and the final norm and patch-out run on real residuals. The oracle runs the same loop with the
    # same two blocks (about 13 TFLOP in float64).
    inp = DI.denoise_inputs("denoise", blocks=2)
    assert (inp.shape.L, inp.shape.N, len(inp.steps_sigmas)) == (512, 4096, 5)
    assert np.count_nonzero(inp.w_ada) > 0
    got = _run(inp, _model_dev(inp))
    ref = O.denoise(inp).astype(np.float64)
    _check(got, ref, inp.latents.astype(np.float64), "full-size denoise, 2 real blocks")
