"""Step-level parity of the CUDA path (through the C ABI) against the CPU oracle.

Tolerances, derived from the arithmetic of each kernel:
* fp32-accumulated bf16 products over K terms: |err| <= 4e-5 * sum_k |a_k w_k| (well above the
  typical sqrt(K) * 2^-24 and far below any structural mistake);
* a bf16-rounded output adds half a bf16 ulp: rtol 2^-8;
* attention rounds P to bf16 (relative 2^-9 per weight) and the output to bf16:
  |err| <= 2^-8 * max|v| + 2^-8 |o|;
* bit-exact where both sides perform the same IEEE operations: Euler step (separately rounded
  fp32), int8lin dequantisation (one rounding of an exact product), rotary tables (fp64 angle,
  one rounding to fp32).
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import (bf16_bits, bf16_f64, dev, dev_bf16, dims_of, max_abs, rope_dev, workspace)

pytestmark = pytest.mark.gpu

GEMM_RTOL = 4e-5


def _bf16_rand(g, shape, std):
    return DI.bf16_bits_from_f32(g.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _gemm_bound(A, W):
    return np.abs(A) @ np.abs(W).T


# ---------------------------------------------------------------------------------- Euler

@pytest.mark.parametrize("n", [1, 7, 4096 * 64, 4096 * 64 + 3])
def test_euler_bit_exact(n):
    g = np.random.default_rng(n)
    sig = [1.0, 0.978453, 0.95418, 0.926626, 0.89508, 0.845148, 0.704534, 0.414568, 0.0]
    x = g.standard_normal(n).astype(np.float32)
    v = g.standard_normal(n).astype(np.float32)
    xd, vd = dev(x), dev(v)
    for i in range(8):
        D.dit_euler_step(xd, vd, sig[i], sig[i + 1])
        x = O.euler_step(x, v, np.float32(sig[i]), np.float32(sig[i + 1]))
    D.dit_check()
    assert np.array_equal(xd.cpu().numpy().view(np.uint32), x.view(np.uint32))


def test_euler_empty_is_noop():
    D.dit_euler_step(torch.empty(0, device="cuda"), torch.empty(0, device="cuda"), 1.0, 0.5)
    D.dit_check()


# ---------------------------------------------------------------------------------- rotary tables

@pytest.mark.parametrize("shape", ["tiny", "512sq", "1024sq", "denoise"])
def test_rope_tables_match_oracle(shape):
    sh = DI.SHAPES[shape]
    tc, ts, ic, is_ = rope_dev(sh)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), sh.head_dim)
    got_c = np.concatenate([tc.cpu().numpy(), ic.cpu().numpy()])
    got_s = np.concatenate([ts.cpu().numpy(), is_.cpu().numpy()])
    # fp64 angle rounded once to fp32 on both sides: equal unless the two fp64 libm results straddle
    # an fp32 rounding boundary (then one fp32 ulp)
    diff_c = np.abs(got_c.view(np.int32).astype(np.int64) - cos.view(np.int32).astype(np.int64))
    diff_s = np.abs(got_s.view(np.int32).astype(np.int64) - sin.view(np.int32).astype(np.int64))
    assert diff_c.max() <= 1 and diff_s.max() <= 1
    assert (diff_c > 0).mean() < 1e-4 and (diff_s > 0).mean() < 1e-4


# ---------------------------------------------------------------------------------- modulated norm

@pytest.mark.parametrize("shape,M,nw", [("tiny", None, False), ("tiny", 2, True), ("tiny", 1, False),
                                        ("512sq", None, True)])
@pytest.mark.parametrize("which", [0, 1])
def test_modnorm(shape, M, nw, which):
    inp = DI.block_inputs(shape, M=M, norm_weights=nw)
    sh = inp.shape
    dims = dims_of(sh)
    h = torch.empty(sh.R, sh.hidden, dtype=torch.bfloat16, device="cuda")
    w = inp.norm1 if which == 0 else inp.norm2
    D.dit_modnorm(dims, dev(inp.txt), dev(inp.img), None if w is None else dev(w),
                  D.Modulation(dev(inp.mod), dev(inp.mod_map)), which, h)
    D.dit_check()
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    m = inp.mod[inp.mod_map]
    ref = O.modulated_rmsnorm(x, w, m[:, 3 * which], m[:, 3 * which + 1], sh.eps)
    np.testing.assert_allclose(bf16_f64(h), ref, rtol=2 ** -8, atol=1e-5)


def test_modnorm_no_text_rows():
    inp = DI.block_inputs("tiny")
    sh = inp.shape
    h = torch.empty(sh.N, sh.hidden, dtype=torch.bfloat16, device="cuda")
    mod = inp.mod[sh.L:]
    D.dit_modnorm(dims_of(sh), None, dev(inp.img), None, D.Modulation(dev(mod), dev(np.arange(sh.N, dtype=np.int32))),
                  0, h)
    D.dit_check()
    ref = O.modulated_rmsnorm(inp.img.astype(np.float64), None, mod[:, 0], mod[:, 1], sh.eps)
    np.testing.assert_allclose(bf16_f64(h), ref, rtol=2 ** -8, atol=1e-5)


# ---------------------------------------------------------------------------------- int8 dequant

def test_dequant_bit_exact():
    g = np.random.default_rng(3)
    q = g.integers(-127, 128, size=(96, 4096), dtype=np.int8)
    q[0, :255] = np.arange(-127, 128, dtype=np.int8)       # every code value
    s = DI.bf16_bits_from_f32((DI.INT8_S0 * (0.75 + 0.5 * g.random((96, 128)))).astype(np.float32))
    s[1, :] = DI.bf16_bits_from_f32(np.float32(1.0 + 2 ** -7) * np.ones(128, np.float32))  # ties appear
    s[2, :] = s[0, :] | np.uint16(0x8000)          # negative scales (q = 0 must give -0)
    s[3, :] = 0                                    # zero scales
    s[4, :64] = np.uint16(0x0001)                  # subnormal scales
    s[4, 64:] = np.uint16(0x7F00)                  # huge scales (256 s overflows bf16)
    q[2:5, :255] = np.arange(-127, 128, dtype=np.int8)
    w = torch.empty(96, 4096, dtype=torch.bfloat16, device="cuda")
    D.dit_dequant_int8(dev(q), dev_bf16(s), w)
    D.dit_check()
    assert np.array_equal(bf16_bits(w), O.dequant_int8(q, s))


def test_dequant_bit_exact_every_code_and_finite_scale():
    # every pair (code in [-127, 127], finite bf16 scale bit pattern: zeros, subnormals, normals, the
    # largest exponents, both signs): one row per scale pattern, that scale on all of the row's
    # 8 blocks of 32, the row's 256 codes every code value once plus a 0
    sb = np.arange(0x10000, dtype=np.uint32)
    sb = sb[((sb >> 7) & 0xFF) != 0xFF].astype(np.uint16)  # drop infinities and NaNs
    codes = np.concatenate([np.arange(-127, 128), [0]]).astype(np.int8)
    q = np.tile(codes, (sb.size, 1))
    s = np.repeat(sb[:, None], 8, axis=1)
    w = torch.empty(sb.size, 256, dtype=torch.bfloat16, device="cuda")
    D.dit_dequant_int8(dev(q), dev_bf16(s), w)
    D.dit_check()
    got, ref = bf16_bits(w), O.dequant_int8(q, s)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, [(hex(int(sb[r])), int(q[r, c]), hex(int(got[r, c])), hex(int(ref[r, c]))) for r, c in bad[:8]]


# ---------------------------------------------------------------------------------- plain GEMM

@pytest.mark.parametrize("M,N,K", [(72, 256, 256), (128, 128, 64), (200, 64, 128), (1088, 768, 3072),
                                   (4, 3072, 256), (333, 512, 1024), (4224, 256, 3072), (129, 256, 64),
                                   (256, 384, 192), (2048, 2560, 256)])
def test_linear_f32(M, N, K):
    # rows > 128 and N a multiple of 128 run on CTA pairs (256-row tiles): 129 rows leave one valid
    # row in the second CTA's half; 256 x 384 is one 256 x 128 tile per 128 columns; 2048 x 2560 has
    # 80 tiles for 76 pairs, so some pairs take a second tile (both accumulator sets in use)
    g = np.random.default_rng(M + N + K)
    A = _bf16_rand(g, (M, K), 1.0)
    W = _bf16_rand(g, (N, K), 0.02)
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    D.dit_linear(dev_bf16(A), dev_bf16(W), out)
    D.dit_check()
    Af, Wf = O.bf16_to_f64(A), O.bf16_to_f64(W)
    ref = Af @ Wf.T
    err = np.abs(out.cpu().numpy() - ref)
    assert np.all(err <= GEMM_RTOL * _gemm_bound(Af, Wf) + 1e-30), float(err.max())


def test_linear_bf16_out_and_identity_exact():
    g = np.random.default_rng(11)
    M, K = 300, 256
    A = _bf16_rand(g, (M, K), 1.0)
    I = DI.bf16_bits_from_f32(np.eye(K, dtype=np.float32))
    out = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    D.dit_linear(dev_bf16(A), dev_bf16(I), out)
    out32 = torch.empty(M, K, dtype=torch.float32, device="cuda")
    D.dit_linear(dev_bf16(A), dev_bf16(I), out32)
    D.dit_check()
    assert np.array_equal(bf16_bits(out), A)                       # A I = A exactly
    assert np.array_equal(out32.cpu().numpy(), O.bf16_to_f64(A).astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(72, 256, 256), (1088, 384, 3072), (130, 128, 12288), (4224, 512, 768)])
def test_linear_int8_vs_oracle_and_bitwise_vs_dequant(M, N, K):
    g = np.random.default_rng(M * 7 + N)
    A = _bf16_rand(g, (M, K), 1.0)
    q = g.integers(-127, 128, size=(N, K), dtype=np.int8)
    s = DI.bf16_bits_from_f32((DI.INT8_S0 * (0.75 + 0.5 * g.random((N, K // 32)))).astype(np.float32))
    out8 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ws = workspace(D.dit_linear_int8_workspace_bytes(N, K))
    ws.fill_(0xAB)  # the call must not depend on the scratch's previous contents
    D.dit_linear_int8(dev_bf16(A), dev(q), dev_bf16(s), out8, ws)
    out8b = torch.empty_like(out8)
    D.dit_linear_int8(dev_bf16(A), dev(q), dev_bf16(s), out8b, ws)  # again, over the previous call's scratch
    wd = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    D.dit_dequant_int8(dev(q), dev_bf16(s), wd)
    out16 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    D.dit_linear(dev_bf16(A), wd, out16)
    D.dit_check()
    # the int8 mainloop feeds the MMA the same bf16 tile as dequant + bf16 GEMM: bitwise equal
    assert torch.equal(out8, out16) and torch.equal(out8b, out16)
    Af, Wf = O.bf16_to_f64(A), O.bf16_to_f64(O.dequant_int8(q, s))
    err = np.abs(out8.cpu().numpy() - Af @ Wf.T)
    assert np.all(err <= GEMM_RTOL * _gemm_bound(Af, Wf) + 1e-30), float(err.max())


# ---------------------------------------------------------------------------------- fused epilogues

@pytest.mark.parametrize("shape,R", [("tiny", 72), ("512sq", 1088), ("512sq", 200)])
def test_swiglu_epilogue(shape, R):
    sh = DI.SHAPES[shape]
    g = np.random.default_rng(R)
    H, F = sh.hidden, sh.ffn
    h2 = _bf16_rand(g, (R, H), 1.0)
    wup = _bf16_rand(g, (2 * F, H), 0.02)
    a = torch.empty(R, F, dtype=torch.bfloat16, device="cuda")
    D.dit_linear_swiglu(dims_of(sh), dev_bf16(h2), dev_bf16(wup), a)
    D.dit_check()
    u = O.bf16_to_f64(h2) @ O.bf16_to_f64(wup).T
    ref = O.swiglu_interleaved(u)
    np.testing.assert_allclose(bf16_f64(a), ref, rtol=2 ** -8, atol=2e-4)


@pytest.mark.parametrize("shape,M,which", [("tiny", None, 0), ("tiny", 2, 1), ("512sq", None, 0), ("512sq", 1, 1)])
def test_gated_epilogue(shape, M, which):
    inp = DI.block_inputs(shape, M=M)
    sh = inp.shape
    g = np.random.default_rng(5)
    K = sh.hidden if which == 0 else sh.ffn
    A = _bf16_rand(g, (sh.R, K), 1.0)
    W = inp.wout if which == 0 else inp.wdown
    txt, img = dev(inp.txt), dev(inp.img)
    D.dit_linear_gated(dims_of(sh), dev_bf16(A), sh.L, sh.N, dev_bf16(W), D.Modulation(dev(inp.mod), dev(inp.mod_map)),
                       which, txt, img)
    D.dit_check()
    Af, Wf = O.bf16_to_f64(A), O.bf16_to_f64(W)
    gate = inp.mod[inp.mod_map, 2 if which == 0 else 5].astype(np.float64)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    ref = x + gate * (Af @ Wf.T)
    got = np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)
    tol = GEMM_RTOL * np.abs(gate) * _gemm_bound(Af, Wf) + 2 ** -23 * np.abs(ref) + 1e-30
    assert np.all(np.abs(got - ref) <= tol), float(np.abs(got - ref).max())


@pytest.mark.parametrize("shape,nw", [("tiny", False), ("tiny", True), ("512sq", True)])
def test_qkv_rope_epilogue(shape, nw):
    inp = DI.block_inputs(shape, norm_weights=nw)
    sh = inp.shape
    R, H, nh, d = sh.R, sh.hidden, sh.heads, sh.head_dim
    g = np.random.default_rng(8)
    h = _bf16_rand(g, (R, H), 1.0)
    q = torch.empty(nh, R, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty_like(q)
    Rp = D.dit_vt_stride(R)
    vt = torch.zeros(nh, d, Rp, dtype=torch.bfloat16, device="cuda")
    tc, ts, ic, is_ = rope_dev(sh)
    qn = None if inp.q_norm is None else dev(inp.q_norm)
    kn = None if inp.k_norm is None else dev(inp.k_norm)
    D.dit_qkv_rope(dims_of(sh), dev_bf16(h), sh.L, sh.N, dev_bf16(inp.wqkv), qn, kn, tc, ts, ic, is_, q, k, vt)
    D.dit_check()
    qkv = O.bf16_to_f64(h) @ O.bf16_to_f64(inp.wqkv).T
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), d)
    rq = O.rope_apply(O.qk_rmsnorm(qkv[:, :H].reshape(R, nh, d), inp.q_norm, sh.qk_eps), cos, sin)
    rk = O.rope_apply(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(R, nh, d), inp.k_norm, sh.qk_eps), cos, sin)
    rv = qkv[:, 2 * H:].reshape(R, nh, d)
    np.testing.assert_allclose(bf16_f64(q), rq.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
    np.testing.assert_allclose(bf16_f64(k), rk.transpose(1, 0, 2), rtol=2 ** -8, atol=1e-3)
    np.testing.assert_allclose(bf16_f64(vt)[:, :, :R], rv.transpose(1, 2, 0), rtol=2 ** -8, atol=1e-4)


# ---------------------------------------------------------------------------------- attention

def _attn_case(R, nh, d, seed, qscale=1.0):
    g = np.random.default_rng(seed)
    q = _bf16_rand(g, (nh, R, d), qscale)
    k = _bf16_rand(g, (nh, R, d), 1.0)
    v = _bf16_rand(g, (nh, R, d), 1.0)
    return q, k, v


@pytest.mark.parametrize("R,nh,d", [(72, 4, 64), (128, 2, 128), (200, 2, 128), (1088, 2, 128), (257, 4, 64),
                                    (4224, 2, 128)])
@pytest.mark.parametrize("qscale", [1.0, 0.05])
def test_attention_vs_oracle(R, nh, d, qscale):
    q, k, v = _attn_case(R, nh, d, R + nh, qscale)
    Rp = D.dit_vt_stride(R)
    vt = np.zeros((nh, d, Rp), np.uint16)
    vt[:, :, :R] = v.transpose(0, 2, 1)
    o = torch.empty(R, nh * d, dtype=torch.bfloat16, device="cuda")
    D.dit_attention(D.DitDims(nh * d, nh, d, 256), R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), o)
    D.dit_check()
    f = lambda a: O.bf16_to_f64(a).transpose(1, 0, 2)
    ref = O.attention(f(q), f(k), f(v))
    got = bf16_f64(o)
    vmax = np.abs(O.bf16_to_f64(v)).max()
    assert np.all(np.abs(got - ref) <= 2 ** -8 * vmax + 2 ** -8 * np.abs(ref)), max_abs(got, ref)


def _qknormed(g, nh, R, d, w):
    """bf16 rows RMS-normalised per head and scaled by w ([d] or None), as the QKV epilogue writes them."""
    x = g.standard_normal((nh, R, d))
    x = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)
    if w is not None:
        x = x * w
    return DI.bf16_bits_from_f32(x.astype(np.float32))


@pytest.mark.parametrize("R,nh,d", [(72, 4, 64), (200, 2, 128), (1088, 2, 128), (4224, 2, 128)])
@pytest.mark.parametrize("wkind", ["ones", "near_one", "large"])
def test_attention_qknorm_vs_oracle(R, nh, d, wkind):
    # q and k as the QK-norm epilogue leaves them: with weights near one the scaled scores stay
    # within the fixed bound B = d max|w_q| max|w_k| / sqrt(d) < 60 (log2 units) and the softmax
    # subtracts B; weights of 4 put B above 60 and the kernel keeps the running maximum
    g = np.random.default_rng(R * 3 + nh + len(wkind))
    wq = wk = None
    if wkind == "near_one":
        wq = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
        wk = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
    elif wkind == "large":
        wq = np.full(d, 4.0, np.float32)
        wk = np.full(d, 1.5, np.float32)
    q, k = _qknormed(g, nh, R, d, wq), _qknormed(g, nh, R, d, wk)
    v = _bf16_rand(g, (nh, R, d), 1.0)
    Rp = D.dit_vt_stride(R)
    vt = np.zeros((nh, d, Rp), np.uint16)
    vt[:, :, :R] = v.transpose(0, 2, 1)
    dims = D.DitDims(nh * d, nh, d, 256)
    o = torch.empty(R, nh * d, dtype=torch.bfloat16, device="cuda")
    o_gen = torch.empty_like(o)
    tw = lambda w: None if w is None else dev(w)
    D.dit_attention_qknorm(dims, R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), tw(wq), tw(wk), o)
    D.dit_attention(dims, R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), o_gen)
    D.dit_check()
    f = lambda a: O.bf16_to_f64(a).transpose(1, 0, 2)
    ref = O.attention(f(q), f(k), f(v))
    vmax = np.abs(O.bf16_to_f64(v)).max()
    for got in (bf16_f64(o), bf16_f64(o_gen)):
        assert np.all(np.abs(got - ref) <= 2 ** -8 * vmax + 2 ** -8 * np.abs(ref)), max_abs(got, ref)
    if wkind == "large":  # B > 60: the same kernel path as dit_attention, bit for bit
        assert torch.equal(o, o_gen)


def test_attention_zero_query_gives_mean_value():
    R, nh, d = 300, 2, 128
    q, k, v = _attn_case(R, nh, d, 1)
    q[:] = 0
    vt = np.zeros((nh, d, D.dit_vt_stride(R)), np.uint16)
    vt[:, :, :R] = v.transpose(0, 2, 1)
    o = torch.empty(R, nh * d, dtype=torch.bfloat16, device="cuda")
    D.dit_attention(D.DitDims(nh * d, nh, d, 256), R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), o)
    D.dit_check()
    mean_v = O.bf16_to_f64(v).mean(axis=1).reshape(1, nh * d)
    got = bf16_f64(o)
    assert np.all(np.abs(got - mean_v) <= 2 ** -8 * np.abs(O.bf16_to_f64(v)).max())


@pytest.mark.parametrize("w,path", [(1.8559, "fixed"), (1.9188, "running")])
def test_attention_qknorm_near_the_fixed_maximum_cutoff(w, path):
    # Norm weights that put the bound B = (1 + 2^-6)^2 d w^2 log2(e) / sqrt(d) just below (58) and
    # just above (62) the cutoff of 60 at which the kernel leaves the fixed maximum for the running
    # one. Some key rows equal a query row (score near +B) and some its negation (score near -B), so
    # under the fixed maximum the weights exp2(s - B) reach down to about 2^-116 and their products
    # with small values near the bottom of the fp32 range; both paths must still match the oracle.
    R, nh, d = 1088, 2, 128
    B = (1 + 2 ** -6) ** 2 * d * w * w / np.log(2.0) / np.sqrt(d)
    assert (B < 60) == (path == "fixed") and abs(B - (58 if path == "fixed" else 62)) < 0.1
    g = np.random.default_rng(int(w * 1e4))
    wv = np.full(d, w, np.float32)
    q, k = _qknormed(g, nh, R, d, wv), _qknormed(g, nh, R, d, wv)
    idx = g.choice(R, 96, replace=False)
    k[:, idx[:48]] = q[:, idx[:48]]                     # aligned: s close to +B
    k[:, idx[48:]] = q[:, idx[48:]] ^ np.uint16(0x8000)  # anti-aligned: s close to -B
    v = _bf16_rand(g, (nh, R, d), 1.0)
    v[:, idx[48:64]] = DI.bf16_bits_from_f32((O.bf16_to_f64(v[:, idx[48:64]]) * 2.0 ** -10).astype(np.float32))
    Rp = D.dit_vt_stride(R)
    vt = np.zeros((nh, d, Rp), np.uint16)
    vt[:, :, :R] = v.transpose(0, 2, 1)
    dims = D.DitDims(nh * d, nh, d, 256)
    o = torch.empty(R, nh * d, dtype=torch.bfloat16, device="cuda")
    o_gen = torch.empty_like(o)
    D.dit_attention_qknorm(dims, R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), dev(wv), dev(wv), o)
    D.dit_attention(dims, R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), o_gen)
    D.dit_check()
    f = lambda a: O.bf16_to_f64(a).transpose(1, 0, 2)
    qf, kf = f(q), f(k)
    s = np.einsum("rhd,chd->hrc", qf, kf) / np.sqrt(d) / np.log(2.0)
    assert s.max() > 0.95 * B and s.min() < -0.95 * B  # the scores span nearly [-B, B]
    ref = O.attention(qf, kf, f(v))
    vmax = np.abs(O.bf16_to_f64(v)).max()
    for got in (bf16_f64(o), bf16_f64(o_gen)):
        assert np.all(np.abs(got - ref) <= 2 ** -8 * vmax + 2 ** -8 * np.abs(ref)), max_abs(got, ref)
    if path == "running":  # B > 60: the same kernel path as dit_attention, bit for bit
        assert torch.equal(o, o_gen)
    else:                  # B < 60: the fixed path, which rounds differently from the running one
        assert not torch.equal(o, o_gen)
