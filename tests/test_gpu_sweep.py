"""Seeded sweep of small shapes for the three block forms (sequential, parallel, double-stream)
against the float64 oracle, with the gates of the block tests: head counts and widths, ffn sizes,
text and image lengths (ragged, empty text, text a multiple of 128) and modulation row counts."""

import numpy as np
import pytest

import dit_inputs as DI
import oracle as O
from tests.gpu_util import run_block_gpu
from tests.test_gpu_block import _check
from tests.test_gpu_double import oracle_double, run_double_gpu
from tests.test_gpu_parallel import run_parallel_gpu

pytestmark = pytest.mark.gpu

# (hidden, heads, head_dim, ffn, L, grid_h, grid_w, M)
SHAPES = [
    (256, 2, 128, 256, 5, 3, 7, None),
    (512, 8, 64, 1024, 0, 11, 13, 1),
    (512, 4, 128, 640, 31, 6, 6, 2),
    (768, 12, 64, 1536, 128, 4, 16, 3),
    (256, 4, 64, 384, 200, 1, 9, None),
    (1024, 8, 128, 2048, 17, 10, 10, 4),
]


def _shape(i, s):
    H, nh, d, F, L, gh, gw, _ = s
    return DI.BlockShape(f"sweep{i}", H, nh, d, F, L, gh, gw, seed=300 + i)


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_sweep_sequential(i):
    s = SHAPES[i]
    inp = DI.block_inputs(_shape(i, s), M=s[7], norm_weights=(i % 2 == 1))
    t, im = run_block_gpu(inp)
    rt, ri = O.block_forward(inp)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, im]), np.concatenate([rt, ri]), x, f"sweep sequential {s}")


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_sweep_parallel(i):
    s = SHAPES[i]
    if s[0] % 256 or s[3] % 128:
        pytest.skip("parallel block: hidden % 256 and ffn % 128")
    inp = DI.parallel_block_inputs(_shape(i, s), M=s[7], norm_weights=(i % 2 == 0))
    t, im = run_parallel_gpu(inp)
    rt, ri = O.parallel_block_forward(inp)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, im]), np.concatenate([rt, ri]), x, f"sweep parallel {s}")


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_sweep_double(i):
    s = SHAPES[i]
    sh = _shape(i, s)
    inp = DI.block_inputs(sh, M=s[7], norm_weights=True)
    tw = DI.block_inputs(sh, norm_weights=True, seed=sh.seed + 50)
    t, im = run_double_gpu(inp, tw)
    ref = oracle_double(inp, tw)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, im]), ref, x, f"sweep double {s}")
