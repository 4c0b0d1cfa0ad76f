"""LoRA adapters beside the linears of the parallel and the double-stream blocks through the C ABI
(dit_parallel_block_forward_lora, dit_double_block_forward_lora) against the float64 oracle on
merged weights W + B A [gizai:dit, Block.parallel; withLora, loraOf, weightAt; klein article,
sections 4.3-4.4], with the gates of the block tests. The adapters carry a large share of each
linear's output, so a missing, misplaced or wrong-stream adapter fails."""

import numpy as np
import pytest

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import block_weights_dev, dev, dev_bf16, dims_of, modulation_dev, rope_dev, workspace
from tests.test_gpu_block import _check, _sample_rows
from tests.test_gpu_lora import _adapters

pytestmark = pytest.mark.gpu


def _lora_dev(A, B, rank):
    return D.LoRA([None if a is None else dev_bf16(a) for a in A], [None if b is None else dev_bf16(b) for b in B],
                  rank)


def _merged(inp, A, B):
    W = O.block_weights_f64(inp)
    return tuple(w if a is None else O.lora_merge(w, O.bf16_to_f64(a), O.bf16_to_f64(b)) for w, a, b in zip(W, A, B))


def _out(txt, img, sh):
    t = txt.cpu().numpy().astype(np.float64) if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, img.cpu().numpy().astype(np.float64)])


@pytest.mark.parametrize("shape,rank,which", [("tiny", 16, (0, 1, 2, 3)), ("tiny", 24, (1, 2)),
                                              ("512sq", 32, (0, 1, 2, 3))])
def test_parallel_block_lora(shape, rank, which):
    inp = DI.parallel_block_inputs(shape, M=2 if shape == "tiny" else None, norm_weights=True)
    sh = inp.shape
    A, B = _adapters(inp, rank, which, seed=rank, scale=0.05 if shape == "tiny" else 0.02)
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_lora_workspace_bytes(dims, sh.L, sh.N, rank))
    D.dit_parallel_block_forward_lora(dims, block_weights_dev(inp), _lora_dev(A, B, rank), txt, img, tc, ts, ic, is_,
                                      modulation_dev(inp), ws)
    D.dit_check()
    got = _out(txt, img, sh)
    rows = np.arange(sh.R) if sh.R <= 512 else _sample_rows(sh, seed=23)
    ref = O.parallel_block_forward(inp, weights=_merged(inp, A, B), rows=rows)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)[rows]
    _check(got[rows], ref, x, f"parallel lora {shape} rank {rank} on {which}")
    plain = O.parallel_block_forward(inp, rows=rows)
    assert np.sqrt(np.mean((ref - plain) ** 2)) > 0.1 * np.sqrt(np.mean((ref - x) ** 2))  # adapters matter


def _double_inputs(shape):
    img = DI.block_inputs(shape, M=2 if shape == "tiny" else None, norm_weights=True)
    txt_w = DI.block_inputs(shape, norm_weights=True, seed=img.shape.seed + 50)
    return img, txt_w


@pytest.mark.parametrize("shape,ranks", [("tiny", (16, 32)), ("tiny", (None, 24)), ("tiny", (16, None)),
                                         ("512sq", (32, 16))])
def test_double_block_lora(shape, ranks):
    img, txt_w = _double_inputs(shape)
    sh = img.shape
    dims = dims_of(sh)
    ads = [(_adapters(b, r, seed=7 + k, scale=0.05 if shape == "tiny" else 0.02) if r else ([None] * 4, [None] * 4))
           for k, (b, r) in enumerate(zip((txt_w, img), ranks))]
    loras = [_lora_dev(A, B, r) if r else None for (A, B), r in zip(ads, ranks)]
    txt, xi = dev(img.txt), dev(img.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_lora_workspace_bytes(dims, sh.L, sh.N, max(r or 8 for r in ranks)))
    D.dit_double_block_forward_lora(dims, block_weights_dev(txt_w), loras[0], block_weights_dev(img), loras[1], txt, xi,
                                    tc, ts, ic, is_, modulation_dev(img), ws)
    D.dit_check()
    got = _out(txt, xi, sh)
    rows = np.arange(sh.R) if sh.R <= 512 else _sample_rows(sh, seed=29)
    x = np.concatenate([img.txt, img.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_rows(x, _merged(txt_w, *ads[0]), _merged(img, *ads[1]), img.mod, img.mod_map, cos,
                                      sin, sh.heads, sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w),
                                      norms_img=nrm(img), eps=sh.eps, qk_eps=sh.qk_eps)
    _check(got[rows], ref, x[rows], f"double lora {shape} ranks {ranks}")
    plain = O.double_block_forward_rows(x, O.block_weights_f64(txt_w), O.block_weights_f64(img), img.mod, img.mod_map,
                                        cos, sin, sh.heads, sh.head_dim, sh.L, rows=rows, norms_txt=nrm(txt_w),
                                        norms_img=nrm(img), eps=sh.eps, qk_eps=sh.qk_eps)
    assert np.sqrt(np.mean((ref - plain) ** 2)) > 0.05 * np.sqrt(np.mean((ref - x[rows]) ** 2))  # adapters matter


def test_double_block_lora_rejects_no_adapters():
    img, txt_w = _double_inputs("tiny")
    sh = img.shape
    dims = dims_of(sh)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_lora_workspace_bytes(dims, sh.L, sh.N, 16))
    with pytest.raises(D.DitError) as e:
        D.dit_double_block_forward_lora(dims, block_weights_dev(txt_w), None, block_weights_dev(img), None,
                                        dev(img.txt), dev(img.img), tc, ts, ic, is_, modulation_dev(img), ws)
    assert e.value.status == D.DIT_EINVAL
