"""LoRA adapters beside the block's linears through the C ABI (dit_block_forward_lora) against the
float64 oracle on merged weights W + B A [gizai:dit, withLora, loraOf, weightAt], with the gates of
the block tests. The adapters are scaled to carry a large share of each linear's output, so a
missing or misplaced adapter fails."""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import (block_weights_dev, dev, dev_bf16, dims_of, modulation_dev, rope_dev, run_block_gpu,
                            workspace)
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def _adapters(inp, rank, which=(0, 1, 2, 3), seed=0, scale=0.05):
    sh = inp.shape
    H, F = sh.hidden, sh.ffn
    shapes = [(3 * H, H), (H, H), (2 * F, H), (H, F)]
    g = np.random.default_rng(seed)
    A, B = [None] * 4, [None] * 4
    for i in which:
        out, inn = shapes[i]
        A[i] = DI.bf16_bits_from_f32(g.standard_normal((rank, inn), dtype=np.float32) * np.float32(scale))
        B[i] = DI.bf16_bits_from_f32(g.standard_normal((out, rank), dtype=np.float32) * np.float32(scale))
    return A, B


def _run(inp, A, B, rank):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    lora = D.LoRA([None if a is None else dev_bf16(a) for a in A], [None if b is None else dev_bf16(b) for b in B],
                  rank)
    ws = workspace(D.dit_lora_workspace_bytes(dims, sh.L, sh.N, rank))
    D.dit_block_forward_lora(dims, block_weights_dev(inp), lora, txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


def _oracle(inp, A, B, rows=None):
    W = O.block_weights_f64(inp)
    merged = tuple(w if a is None else O.lora_merge(w, O.bf16_to_f64(a), O.bf16_to_f64(b)) for w, a, b in zip(W, A, B))
    return O.block_forward(inp, weights=merged, rows=rows)


@pytest.mark.parametrize("rank,which", [(16, (0, 1, 2, 3)), (64, (0, 1, 2, 3)), (24, (1, 3))])
def test_lora_tiny_all_rows(rank, which):
    inp = DI.block_inputs("tiny", M=2, norm_weights=True)
    A, B = _adapters(inp, rank, which, seed=rank)
    got = _run(inp, A, B, rank)
    ref = _oracle(inp, A, B)
    ref = np.concatenate(ref) if isinstance(ref, tuple) else ref
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(got, ref, x, f"lora tiny rank {rank} on {which}")
    plain = np.concatenate(O.block_forward(inp))
    d_ref, d_plain = ref - x, plain - x
    assert np.sqrt(np.mean((d_ref - d_plain) ** 2)) > 0.1 * np.sqrt(np.mean(d_ref ** 2))  # adapters matter


@pytest.mark.parametrize("shape,rank", [("512sq", 32), ("1024sq", 64)])
def test_lora_sampled_rows(shape, rank):
    inp = DI.block_inputs(shape)
    A, B = _adapters(inp, rank, seed=7, scale=0.02)
    got = _run(inp, A, B, rank)
    rows = _sample_rows(inp.shape, seed=19)
    ref = _oracle(inp, A, B, rows=rows)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x, f"lora {shape} rank {rank}")


def test_lora_with_zero_B_is_the_plain_block_bitwise():
    inp = DI.block_inputs("tiny")
    A, B = _adapters(inp, 16, seed=3)
    B = [np.zeros_like(b) for b in B]
    got = _run(inp, A, B, 16)
    t, i = run_block_gpu(inp)
    assert np.array_equal(got, np.concatenate([t, i]))
