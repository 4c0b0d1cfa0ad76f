"""Parity of the parallel (single-stream) block through the C ABI (dit_parallel_block_forward)
against the float64 oracle [gizai:dit, Block.parallel], with the gates of the sequential block:
max |out err| <= 2e-2 RMS(out); on the block's contribution delta = out - in, RMS err <= 1e-2 and
max err <= 8e-2 of RMS(delta) (the GPU rounds h, q, k, v, P, o and a to bf16 as GEMM operands)."""

import numpy as np
import pytest

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import block_weights_dev, dev, dims_of, modulation_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows

pytestmark = pytest.mark.gpu


def run_parallel_gpu(inp):
    sh = inp.shape
    dims = dims_of(sh)
    txt = dev(inp.txt) if sh.L > 0 else None
    img = dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 2))
    D.dit_parallel_block_forward(dims, block_weights_dev(inp), txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return t, img.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,nw", [(None, False), (2, True), (1, False)])
def test_parallel_tiny_all_rows(M, nw):
    inp = DI.parallel_block_inputs("tiny", M=M, norm_weights=nw)
    t, i = run_parallel_gpu(inp)
    rt, ri = O.parallel_block_forward(inp)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, i]), np.concatenate([rt, ri]), x_in, f"parallel tiny M={M} norm_weights={nw}")


@pytest.mark.parametrize("L,gh,gw", [(8, 16, 20), (13, 9, 10), (1, 5, 7)])
def test_parallel_head64_ragged(L, gh, gw):
    sh = DI.BlockShape(f"pd64_{L}_{gh}x{gw}", 256, 4, 64, 768, L, gh, gw, seed=L + gh + 40)
    inp = DI.parallel_block_inputs(sh, M=2, norm_weights=True)
    t, i = run_parallel_gpu(inp)
    rt, ri = O.parallel_block_forward(inp)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    _check(np.concatenate([t, i]), np.concatenate([rt, ri]), x_in, f"parallel d=64 L={L} grid {gh}x{gw}")


@pytest.mark.parametrize("shape", ["512sq", "1024sq"])
def test_parallel_sampled_rows(shape):
    inp = DI.parallel_block_inputs(shape)
    sh = inp.shape
    t, i = run_parallel_gpu(inp)
    rows = _sample_rows(sh, seed=11)
    ref = O.parallel_block_forward(inp, rows=rows)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(np.concatenate([t, i])[rows], ref, x_in, f"parallel {shape} sampled rows")


def test_parallel_zero_gate_leaves_residual_bitwise():
    inp = DI.parallel_block_inputs("512sq")
    inp.mod[:, 2, :] = 0.0
    t, i = run_parallel_gpu(inp)
    assert np.array_equal(t, inp.txt.astype(np.float64)) and np.array_equal(i, inp.img.astype(np.float64))


def test_parallel_deterministic():
    inp = DI.parallel_block_inputs("512sq", M=1)
    a = run_parallel_gpu(inp)
    b = run_parallel_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_parallel_abi_rejects_small_workspace():
    inp = DI.parallel_block_inputs("tiny")
    sh = inp.shape
    dims = dims_of(sh)
    need = D.dit_workspace_bytes(dims, sh.L, sh.N, 2)
    assert need == D.dit_workspace_bytes(dims, sh.L, sh.N, 0)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    with pytest.raises(D.DitError) as e:
        D.dit_parallel_block_forward(dims, block_weights_dev(inp), txt, img, tc, ts, ic, is_, modulation_dev(inp),
                                     workspace(need - 256))
    assert e.value.status == D.DIT_EWORKSPACE
    D.dit_check()
    assert np.array_equal(txt.cpu().numpy(), inp.txt) and np.array_equal(img.cpu().numpy(), inp.img)
