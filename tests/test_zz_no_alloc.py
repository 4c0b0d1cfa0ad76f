"""dit_block_forward_noalloc: the block forward for callers that cannot allocate device memory.

Such callers (a plugin inside a host application whose allocator owns the device memory, or a
latency-bound loop where an allocation's implicit synchronisation is not allowed) pass only inputs
and outputs; the scratch is the library's static device array. The test calls the entry point
through the C ABI, three calls in a row on shapes of different sizes (so the array holds another
call's contents each time), and checks each result against dit_block_forward with an allocated
workspace. Both run the same kernels, with the same launch plan, on the same inputs, and the block is
deterministic bit for bit, so the results must be equal bit for bit: a byte of the array left over
from the previous call and read before being written would show up here. It also checks that a
shape larger than the array is rejected before any launch. This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
from tests.gpu_util import (block_weights_dev, dev, dims_of, max_abs, modulation_dev, rms, rope_dev, run_block_gpu)

pytestmark = pytest.mark.gpu


def _noalloc(inp):
    sh = inp.shape
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    D.dit_block_forward_noalloc(dims_of(sh), block_weights_dev(inp), txt, img, tc, ts, ic, is_, modulation_dev(inp))
    D.dit_check()
    return np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)


def test_noalloc_matches_allocated_workspace_on_consecutive_calls():
    for shape in ("tiny", "512sq", "tiny"):
        inp = DI.block_inputs(shape)
        got = _noalloc(inp)
        t, i = run_block_gpu(inp)
        ref = np.concatenate([t, i])
        x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
        # bit for bit; the error relative to the block's change is printed when they differ
        assert np.array_equal(got, ref), (
            f"{shape}: {int(np.count_nonzero(got != ref))} outputs differ, max |diff| {max_abs(got, ref):.3e}, "
            f"RMS(diff) / RMS(delta) {rms(got - ref) / rms(ref - x_in):.3e}")


def test_noalloc_rejects_shapes_beyond_the_static_array():
    inp = DI.block_inputs("tiny")
    sh = DI.SHAPES["1024sq"]
    dims = dims_of(sh)
    assert D.dit_workspace_bytes(dims, sh.L, sh.N, 0) > D.dit_block_noalloc_max_bytes()
    x = torch.zeros(sh.N, sh.hidden, device="cuda")
    t = torch.zeros(sh.L, sh.hidden, device="cuda")
    tab = torch.zeros(sh.R, sh.head_dim // 2, device="cuda")
    mod = D.Modulation(torch.zeros(1, 6, sh.hidden, device="cuda"))
    w = block_weights_dev(inp)  # never read: the call is rejected before any launch
    with pytest.raises(D.DitError) as e:
        D.dit_block_forward_noalloc(dims, w, t, x, tab[:sh.L], tab[:sh.L], tab[sh.L:], tab[sh.L:], mod)
    assert e.value.status == D.DIT_EWORKSPACE
    assert torch.count_nonzero(x).item() == 0 and torch.count_nonzero(t).item() == 0
