"""Stream-K on the tcgen05 GEMM: the k-blocks of the tiles beyond whole waves divided evenly over
all work units, each unit's share of a tile written as an fp32 partial and summed in a fixed order
by the unit that delivers the tile's last share, which then runs the tile's epilogue.

For every epilogue that takes the scratch (gated residual, QK-norm + rotary, SwiGLU), on CTA pairs
(rows > 128) and single CTAs (rows <= 128): the result with scratch is deterministic bit for bit,
differs from the whole-tile result (no scratch) only by the order of the fp32 additions, and
matches the float64 definition of the linear on sampled rows with the tolerances of the epilogue
tests. A shape whose tiles make whole waves (228 pair tiles on 76 pairs) takes no stream-K: the
scratch changes nothing there.
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_f64, dev, dev_bf16, dims_of, rope_dev, workspace
from tests.test_gpu_kernels import GEMM_RTOL, _bf16_rand, _gemm_bound

pytestmark = pytest.mark.gpu


def _scratch():
    return workspace(D.dit_stream_k_workspace_bytes())


@pytest.mark.parametrize("L,gh,gw,which,sk", [
    (128, 64, 64, 1, True),    # R 4224: 17 row tiles x 12 = 204 pair tiles, 52 over two waves
    (128, 56, 64, 1, True),    # R 3712: 180 tiles, 28 over: region 28 + 76 tiles
    (100, 41, 80, 1, True),    # R 3380 (ragged): 168 tiles, 16 over
    (128, 64, 64, 0, True),    # the out linear (K = 3072) at R 4224
    (128, 64, 74, 1, False),   # R 4864: 228 tiles, three whole waves
])
def test_gated_stream_k(L, gh, gw, which, sk):
    sh = DI.BlockShape(f"sk_{L}_{gh}x{gw}", 3072, 24, 128, 12288, L, gh, gw, seed=21 + L)
    inp = DI.block_inputs(sh)
    g = np.random.default_rng(6 + which)
    K = sh.hidden if which == 0 else sh.ffn
    A = _bf16_rand(g, (sh.R, K), 1.0)
    W = inp.wout if which == 0 else inp.wdown
    dims, a, w = dims_of(sh), dev_bf16(A), dev_bf16(W)
    mod = D.Modulation(dev(inp.mod), dev(inp.mod_map))
    ws = _scratch()
    outs = []
    for scratch in (ws, ws, None):
        txt, img = dev(inp.txt), dev(inp.img)
        D.dit_linear_gated(dims, a, sh.L, sh.N, w, mod, which, txt, img, ws=scratch)
        D.dit_check()
        outs.append(np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64))
    streamk, streamk2, whole = outs
    assert np.array_equal(streamk, streamk2)
    assert np.array_equal(streamk, whole) != sk  # the stream-K path ran (other summation order) or not
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    gate = inp.mod[inp.mod_map, 2 if which == 0 else 5].astype(np.float64)
    Af, Wf = O.bf16_to_f64(A), O.bf16_to_f64(W)
    # |stream-K - whole| <= the fp32 rounding of a K-long sum of products (both orders), times the gate
    rows = np.unique(np.concatenate([g.choice(sh.R, 64, replace=False), np.arange(sh.R - 40, sh.R),
                                     np.arange(sh.L - 4, sh.L + 4)]))
    bnd = _gemm_bound(Af[rows], Wf)
    assert np.all(np.abs(streamk - whole)[rows] <= 2 * GEMM_RTOL * np.abs(gate[rows]) * bnd + 1e-30)
    ref = x[rows] + gate[rows] * (Af[rows] @ Wf.T)
    tol = GEMM_RTOL * np.abs(gate[rows]) * bnd + 2 ** -23 * np.abs(ref) + 1e-30
    assert np.all(np.abs(streamk[rows] - ref) <= tol), float(np.abs(streamk[rows] - ref).max())


def test_qkv_rope_stream_k():
    # R 4224: 612 pair tiles, 8 waves and 4 over: the last 80 tiles divided over the 76 pairs
    inp = DI.block_inputs("1024sq", norm_weights=True)
    sh = inp.shape
    R, H, nh, d = sh.R, sh.hidden, sh.heads, sh.head_dim
    g = np.random.default_rng(9)
    h = _bf16_rand(g, (R, H), 1.0)
    tc, ts, ic, is_ = rope_dev(sh)
    qn, kn = dev(inp.q_norm), dev(inp.k_norm)
    ws = _scratch()
    res = []
    for scratch in (ws, ws, None):
        q = torch.empty(nh, R, d, dtype=torch.bfloat16, device="cuda")
        k = torch.empty_like(q)
        vt = torch.zeros(nh, d, D.dit_vt_stride(R), dtype=torch.bfloat16, device="cuda")
        D.dit_qkv_rope(dims_of(sh), dev_bf16(h), sh.L, sh.N, dev_bf16(inp.wqkv), qn, kn, tc, ts, ic, is_, q, k, vt,
                       ws=scratch)
        D.dit_check()
        res.append((q, k, vt))
    (q, k, vt), (q2, k2, vt2), (qw, kw, vtw) = res
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(vt, vt2)
    assert not (torch.equal(q, qw) and torch.equal(k, kw) and torch.equal(vt, vtw))
    rows = np.unique(np.concatenate([g.choice(R, 48, replace=False), np.arange(R - 130, R)]))
    qkv = O.bf16_to_f64(h[rows]) @ O.bf16_to_f64(inp.wqkv).T
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), d)
    rq = O.rope_apply(O.qk_rmsnorm(qkv[:, :H].reshape(-1, nh, d), inp.q_norm, sh.qk_eps), cos[rows], sin[rows])
    rk = O.rope_apply(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(-1, nh, d), inp.k_norm, sh.qk_eps), cos[rows], sin[rows])
    rv = qkv[:, 2 * H:].reshape(-1, nh, d)
    for got_q, got_k, got_vt in ((q, k, vt), (qw, kw, vtw)):
        np.testing.assert_allclose(bf16_f64(got_q)[:, rows], rq.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
        np.testing.assert_allclose(bf16_f64(got_k)[:, rows], rk.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
        np.testing.assert_allclose(bf16_f64(got_vt)[:, :, rows], rv.transpose(1, 2, 0), rtol=2 ** -8, atol=1e-4)


@pytest.mark.parametrize("R", [4224, 100])
def test_swiglu_stream_k(R):
    # R 4224: 1632 pair tiles, 21 waves and 36 over (region 112 tiles); R 100: one 128-row block on
    # single CTAs, 96 tiles over 152 SMs, each CTA a share of about 30 of a tile's 48 k-blocks
    sh = DI.SHAPES["1024sq"]
    g = np.random.default_rng(R)
    H, F = sh.hidden, sh.ffn
    h2 = _bf16_rand(g, (R, H), 1.0)
    wup = _bf16_rand(g, (2 * F, H), 0.02)
    ws = _scratch()
    outs = []
    for scratch in (ws, ws, None):
        a = torch.empty(R, F, dtype=torch.bfloat16, device="cuda")
        D.dit_linear_swiglu(dims_of(sh), dev_bf16(h2), dev_bf16(wup), a, ws=scratch)
        D.dit_check()
        outs.append(a)
    assert torch.equal(outs[0], outs[1]) and not torch.equal(outs[0], outs[2])
    rows = np.unique(np.concatenate([g.choice(R, min(R, 48), replace=False), np.arange(R - 8, R)]))
    ref = O.swiglu_interleaved(O.bf16_to_f64(h2[rows]) @ O.bf16_to_f64(wup).T)
    for a in (outs[0], outs[2]):
        np.testing.assert_allclose(bf16_f64(a)[rows], ref, rtol=2 ** -8, atol=2e-4)


def test_block_1024sq_deterministic():
    # the 1024sq block (pair tiles, the fixed-maximum attention) bit for bit from run to run
    from tests.gpu_util import run_block_gpu
    inp = DI.block_inputs("1024sq")
    a = run_block_gpu(inp)
    b = run_block_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
