"""W8A8 forms of the parallel and the double-stream blocks through the C ABI against the oracle
(oracle/w8a8.py) [klein, section 5 (int8 detail: a single block's linear1 and linear2, a double
block's image and text qkv, proj, mlp.0 and mlp.2) and its D4 / D5 entries].

Gates. As for the sequential W8A8 block (tests/test_gpu_w8a8.py), a whole-block comparison has to
allow one-step code flips wherever the GPU's bf16 activation differs from the oracle's in the last
bit: RMS(delta error) <= 4e-2 RMS(delta) and max |out error| <= 1e-1 RMS(out), reported. The tight
gates are stage checks on the GPU's own codes and scales (read from the workspace, whose layout the
test restates and checks against dit_workspace_bytes): the parallel block's linear2 over the joined
codes [o | a] must reproduce the block's output to float32 rounding, its linear1 over the codes of h
the q, k and v the block stored to within one bf16 step; the double-stream block's down linear, per
stream, on its codes of a: the block's output, given its attention half (a second run with the MLP
gate zeroed), to float32 rounding.
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_bits, dev, dims_of, modulation_dev, opt_dev, rms, rope_dev, workspace
from tests.test_gpu_block import _sample_rows
from tests.test_gpu_w8a8 import _check_w8a8

pytestmark = pytest.mark.gpu


def _ru(n, a=256):
    return (n + a - 1) // a * a


def _block_regions(sh):
    R, H, F, nh, d = sh.R, sh.hidden, sh.ffn, sh.heads, sh.head_dim
    out, off = {}, 0
    for name, n in (("h", R * H * 2), ("q", nh * R * d * 2), ("k", nh * R * d * 2), ("vt", nh * d * _ru(R, 8) * 2),
                    ("o", R * H * 2), ("a", R * F * 2)):
        out[name] = off
        off += _ru(n)
    out["end"] = off
    return out


def _bf16_view(ws, off, shape):
    n = int(np.prod(shape))
    return ws[off:off + 2 * n].view(torch.bfloat16).view(*shape)


def _f32_view(ws, off, n):
    return ws[off:off + 4 * n].view(torch.float32).cpu().numpy()


def _fp32_close(got, ref, scale, label):
    worst = float(np.max(np.abs(got - ref) / (2.0 ** -20 * scale + 1e-30)))
    print(f"{label}: max |err| / (2^-20 x magnitude) = {worst:.3f}")
    assert worst <= 1.0, label


# ------------------------------------------------------------------------------- parallel block

def _parallel_case(shape, smooth, seed=7):
    inp = DI.parallel_block_inputs(shape, norm_weights=True)
    sh = inp.shape
    H, F = sh.hidden, sh.ffn
    g = np.random.default_rng(seed)
    sm1 = g.uniform(0.5, 2.0, size=H).astype(np.float32) if smooth else None
    sm2 = g.uniform(0.5, 2.0, size=H + F).astype(np.float32) if smooth else None
    f32 = lambda u: O.bf16_to_f64(u).astype(np.float32)
    l1 = O.quantize_weight(np.concatenate([f32(inp.wqkv), f32(inp.wup)], axis=0), sm1)
    l2 = O.quantize_weight(np.concatenate([f32(inp.wout), f32(inp.wdown)], axis=1), sm2)
    return inp, l1, l2, sm1, sm2


def _run_parallel(inp, l1, l2, sm1, sm2):
    sh = inp.shape
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    w = D.ParallelW8A8Weights(dev(l1[0]), dev(l1[1]), dev(l2[0]), dev(l2[1]), opt_dev(sm1), opt_dev(sm2),
                              opt_dev(inp.norm1), opt_dev(inp.q_norm), opt_dev(inp.k_norm))
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 7))
    D.dit_parallel_block_forward_w8a8(dims, w, txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    return np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64), ws


@pytest.mark.parametrize("shape,smooth", [("tiny", False), ("tiny", True), ("512sq", True)])
def test_parallel_w8a8_block(shape, smooth):
    inp, l1, l2, sm1, sm2 = _parallel_case(shape, smooth)
    sh = inp.shape
    R, H, F, nh, d = sh.R, sh.hidden, sh.ffn, sh.heads, sh.head_dim
    got, ws = _run_parallel(inp, l1, l2, sm1, sm2)
    rows = np.arange(R) if R <= 512 else _sample_rows(sh, seed=31)
    x = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(sh.L, sh.grid_h, sh.grid_w), d)
    ref = O.parallel_block_forward_w8a8_rows(x, l1, l2, inp.mod, inp.mod_map, cos, sin, nh, d, rows=rows,
                                             norm=inp.norm1, q_norm=inp.q_norm, k_norm=inp.k_norm, eps=sh.eps,
                                             qk_eps=sh.qk_eps, smooth1=sm1, smooth2=sm2)
    _check_w8a8(got[rows], ref, x[rows], f"parallel w8a8 {shape} smooth={smooth}")

    # stage checks on the block's own codes and scales
    reg = _block_regions(sh)
    slots = _ru((3 * H + 2 * F) * H * 2) + _ru(H * (H + F) * 2)
    sa1_off = reg["end"] + slots
    sa2_off = sa1_off + _ru(R, 64) * 4
    assert D.dit_workspace_bytes(dims_of(sh), sh.L, sh.N, 7) == sa2_off + _ru(R, 64) * 4
    m = np.asarray(inp.mod, np.float64)[np.asarray(inp.mod_map)[rows]]
    # linear2 over [o | a]: the block's output to float32 rounding
    codes = np.concatenate([O.bf16_to_f64(bf16_bits(_bf16_view(ws, reg["o"], (R, H))))[rows],
                            O.bf16_to_f64(bf16_bits(_bf16_view(ws, reg["a"], (R, F))))[rows]], axis=1)
    assert np.all(np.abs(codes) <= 127) and np.array_equal(codes, np.rint(codes))
    sa2 = _f32_view(ws, sa2_off, R)[rows]
    lin2 = O.w8a8_linear(codes.astype(np.int8), sa2, *l2)
    _fp32_close(got[rows], x[rows] + m[:, 2] * lin2, np.abs(x[rows]) + np.abs(m[:, 2] * lin2),
                f"parallel w8a8 {shape} linear2 stage")
    # linear1 over the codes of h: q, k and v within one bf16 step
    hc = O.bf16_to_f64(bf16_bits(_bf16_view(ws, reg["h"], (R, H))))[rows].astype(np.int8)
    sa1 = _f32_view(ws, sa1_off, R)[rows]
    u = O.w8a8_linear(hc, sa1, *l1)
    q_ref = O.rotate(O.qk_rmsnorm(u[:, :H].reshape(-1, nh, d), inp.q_norm, sh.qk_eps), cos[rows], sin[rows])
    k_ref = O.rotate(O.qk_rmsnorm(u[:, H:2 * H].reshape(-1, nh, d), inp.k_norm, sh.qk_eps), cos[rows], sin[rows])
    v_ref = u[:, 2 * H:3 * H].reshape(-1, nh, d)
    for name, got_bits, r in (("q", bf16_bits(_bf16_view(ws, reg["q"], (nh, R, d)))[:, rows].transpose(1, 0, 2), q_ref),
                              ("k", bf16_bits(_bf16_view(ws, reg["k"], (nh, R, d)))[:, rows].transpose(1, 0, 2), k_ref),
                              ("v", bf16_bits(_bf16_view(ws, reg["vt"], (nh, d, _ru(R, 8))))[:, :, rows]
                               .transpose(2, 0, 1), v_ref)):
        worst = float(np.max(np.abs(O.bf16_to_f64(got_bits) - r) / (2.0 ** -8 * np.abs(r) + 2.0 ** -20 * rms(r))))
        print(f"parallel w8a8 {shape} linear1 stage, {name}: max |err| / one bf16 step = {worst:.3f}")
        assert worst <= 1.0, name


def test_parallel_w8a8_block_deterministic():
    inp, l1, l2, sm1, sm2 = _parallel_case("512sq", True)
    a, _ = _run_parallel(inp, l1, l2, sm1, sm2)
    b, _ = _run_parallel(inp, l1, l2, sm1, sm2)
    assert np.array_equal(a, b)


# -------------------------------------------------------------------------- double-stream block

def _double_case(shape, smooth, L=None, seed=9):
    img = DI.block_inputs(shape, norm_weights=True)
    txt_w = DI.block_inputs(shape, norm_weights=True, seed=img.shape.seed + 50)
    sh = img.shape
    H, F = sh.hidden, sh.ffn
    g = np.random.default_rng(seed)
    ins = (H, H, H, F)
    sms = [[g.uniform(0.5, 2.0, size=n).astype(np.float32) for n in ins] if smooth else [None] * 4 for _ in range(2)]
    f32 = lambda u: O.bf16_to_f64(u).astype(np.float32)
    q = [[O.quantize_weight(f32(W), s) for W, s in zip((b.wqkv, b.wout, b.wup, b.wdown), sm)]
         for b, sm in zip((txt_w, img), sms)]
    return img, txt_w, q, sms


def _w8a8_dev(b, qws, sm):
    return D.W8A8BlockWeights([dev(c) for c, _ in qws], [dev(s) for _, s in qws], [opt_dev(s) for s in sm],
                              opt_dev(b.norm1), opt_dev(b.norm2), opt_dev(b.q_norm), opt_dev(b.k_norm))


def _run_double(img, txt_w, q, sms):
    sh = img.shape
    dims = dims_of(sh)
    txt = dev(img.txt) if sh.L > 0 else None
    xi = dev(img.img)
    tc, ts, ic, is_ = rope_dev(sh)
    ws = workspace(D.dit_workspace_bytes(dims, sh.L, sh.N, 8))
    wt = _w8a8_dev(txt_w, q[0], sms[0]) if sh.L > 0 else None
    D.dit_double_block_forward_w8a8(dims, wt, _w8a8_dev(img, q[1], sms[1]), txt, xi, tc, ts, ic, is_,
                                    modulation_dev(img), ws)
    D.dit_check()
    t = txt.cpu().numpy() if txt is not None else np.zeros((0, sh.hidden))
    return np.concatenate([t, xi.cpu().numpy()]).astype(np.float64), ws


@pytest.mark.parametrize("shape,smooth", [("tiny", False), ("tiny", True), ("512sq", True)])
def test_double_w8a8_block(shape, smooth):
    img, txt_w, q, sms = _double_case(shape, smooth)
    sh = img.shape
    R, H, F, nh, d, L = sh.R, sh.hidden, sh.ffn, sh.heads, sh.head_dim, sh.L
    got, ws = _run_double(img, txt_w, q, sms)
    rows = np.arange(R) if R <= 512 else _sample_rows(sh, seed=37)
    x = np.concatenate([img.txt, img.img]).astype(np.float64)
    cos, sin = O.rope_tables(O.positions(L, sh.grid_h, sh.grid_w), d)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_w8a8_rows(x, q[0], q[1], img.mod, img.mod_map, cos, sin, nh, d, L, rows=rows,
                                           norms_txt=nrm(txt_w), norms_img=nrm(img), eps=sh.eps, qk_eps=sh.qk_eps,
                                           smooth_txt=sms[0] if smooth else None, smooth_img=sms[1] if smooth else None)
    _check_w8a8(got[rows], ref, x[rows], f"double w8a8 {shape} smooth={smooth}")
    # the down linear, per stream, on the block's own codes of a and their scales: with the MLP gate
    # zeroed the block returns x_mid (its attention half; every code upstream of the down linear is
    # the same in both runs), and the full block's output must be x_mid + gate_m * W8A8(a) to float32
    import copy
    mid_in = copy.copy(img)
    mid_in.mod = img.mod.copy()
    mid_in.mod[:, 5, :] = 0.0
    x_mid, _ = _run_double(mid_in, txt_w, q, sms)
    reg = _block_regions(sh)
    sa_off = reg["end"] + 4 * _ru(max(3 * H * H, H * H, 2 * F * H, H * F) * 2)
    assert D.dit_workspace_bytes(dims_of(sh), L, sh.N, 8) == sa_off + _ru(R * 4)
    ac = O.bf16_to_f64(bf16_bits(_bf16_view(ws, reg["a"], (R, F))))[rows].astype(np.int8)
    sa = _f32_view(ws, sa_off, R)[rows]
    m = np.asarray(img.mod, np.float64)[np.asarray(img.mod_map)[rows]]
    for stream, sel in ((0, rows < L), (1, rows >= L)):
        if not sel.any():
            continue
        lin = O.w8a8_linear(ac[sel], sa[sel], *q[stream][3])
        ref_out = x_mid[rows][sel] + m[sel, 5] * lin
        _fp32_close(got[rows][sel], ref_out, np.abs(x_mid[rows][sel]) + np.abs(m[sel, 5] * lin),
                    f"double w8a8 {shape} down stage, stream {stream}")


def test_double_w8a8_no_text_rows():
    # L = 0: the image stream alone, every row quantised with the image divisors
    sh = DI.BlockShape("dw8_L0", 256, 4, 64, 768, 0, 8, 8, seed=41)
    img, txt_w, q, sms = _double_case(sh, True)
    got, _ = _run_double(img, txt_w, q, sms)
    x = img.img.astype(np.float64)
    cos, sin = O.rope_tables(O.positions(0, sh.grid_h, sh.grid_w), sh.head_dim)
    nrm = lambda a: (a.norm1, a.norm2, a.q_norm, a.k_norm)
    ref = O.double_block_forward_w8a8_rows(x, q[0], q[1], img.mod, img.mod_map, cos, sin, sh.heads, sh.head_dim, 0,
                                           norms_txt=nrm(txt_w), norms_img=nrm(img), eps=sh.eps, qk_eps=sh.qk_eps,
                                           smooth_txt=sms[0], smooth_img=sms[1])
    _check_w8a8(got, ref, x, "double w8a8 L=0")


def test_double_w8a8_block_deterministic():
    img, txt_w, q, sms = _double_case("512sq", True)
    a, _ = _run_double(img, txt_w, q, sms)
    b, _ = _run_double(img, txt_w, q, sms)
    assert np.array_equal(a, b)
