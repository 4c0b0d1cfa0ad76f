"""W8A8 block, linear by linear: each of the block's four W8A8 linears checked on the GPU's own bf16
input to that linear [klein, section 5 and its D4 / D5 entries].

The whole-block comparison in test_gpu_w8a8.py has to allow for code flips: where the GPU's bf16
activation and the oracle's differ in the last bit, a per-token int8 code may differ by one step,
and a gate loose enough for that cannot tell a flipped code from a wrong scale. Here every linear
is isolated instead. The oracle's stage function takes the GPU's own upstream activation (each
upstream stage is pinned against the oracle by the other tests), so the codes and scales must agree
bit for bit and the linear's output to float32 rounding:

* qkv: h from dit_modnorm (the block's first kernel) -> the block's q, k and transposed v, which
  are the oracle's QK-normed and rotated W8A8 product rounded once to bf16 (within one bf16 step);
* out: o from dit_attention_qknorm on the block's q, k, v -> the o codes the block left in its
  workspace (bit for bit), and the block's output with the MLP gate zeroed, x + gate_a W8A8(o)
  (within float32 rounding);
* up: h2 from dit_modnorm on that output -> the h2 codes in the workspace (bit for bit) and the
  SwiGLU output's codes and per-token scales (the same but where the last bit of a bf16 value of
  the SwiGLU output differs, float32 on the GPU against float64 here: at most one step, rarely);
* down: the a codes and scales in the workspace -> the block's output, x_mid + gate_m W8A8(a)
  (within float32 rounding).

White box: the workspace regions read here (h, q, k, vt, o, a, then the two weight slots and the
per-token scales) follow the layout of the block workspace; the sizes are checked against
dit_workspace_bytes first, and a region overwritten by a later kernel fails the bit-exact checks.
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_bits, dev, dims_of, modulation_dev, opt_dev, rms, rope_dev, workspace
from tests.test_gpu_block import _sample_rows
from tests.test_gpu_w8a8 import _w8a8_case

pytestmark = pytest.mark.gpu


def _ru(n, a=256):
    return (n + a - 1) // a * a


def _regions(sh):
    """Byte offsets of the block workspace regions of the W8A8 block (variant 4)."""
    R, H, F, nh, d = sh.R, sh.hidden, sh.ffn, sh.heads, sh.head_dim
    sizes = [("h", R * H * 2), ("q", nh * R * d * 2), ("k", nh * R * d * 2), ("vt", nh * d * _ru(R, 8) * 2),
             ("o", R * H * 2), ("a", R * F * 2)]
    off, out = 0, {}
    for name, n in sizes:
        out[name] = off
        off += _ru(n)
    slot = _ru(max(3 * H * H, H * H, 2 * F * H, H * F) * 2)
    out["sa"] = off + 2 * slot
    out["end"] = out["sa"] + _ru(R * 4)
    return out


def _bf16_view(ws, off, shape):
    n = int(np.prod(shape))
    return ws[off:off + 2 * n].view(torch.bfloat16).view(*shape)


def _f64(bits):
    return O.bf16_to_f64(bits)


def _bf16_round(x64):
    return _f64(O.bf16_rne_bits(np.asarray(x64, np.float64).astype(np.float32)))


def _run(inp, qws, sm, ws):
    sh = inp.shape
    dims = dims_of(sh)
    txt, img = dev(inp.txt), dev(inp.img)
    tc, ts, ic, is_ = rope_dev(sh)
    w = D.W8A8BlockWeights([dev(q) for q, _ in qws], [dev(s) for _, s in qws], [opt_dev(s) for s in sm],
                           opt_dev(inp.norm1), opt_dev(inp.norm2), opt_dev(inp.q_norm), opt_dev(inp.k_norm))
    D.dit_block_forward_w8a8(dims, w, txt, img, tc, ts, ic, is_, modulation_dev(inp), ws)
    D.dit_check()
    return np.concatenate([txt.cpu().numpy(), img.cpu().numpy()]).astype(np.float64)


def _fp32_close(got, ref, scale, label):
    # a few float32 roundings (integer accumulator times two scales, then the gated fma) of values of
    # magnitude `scale`: 2^-20 relative leaves a margin of 16 float32 steps
    err = np.abs(got - ref)
    bound = 2.0 ** -20 * scale + 1e-30
    worst = float(np.max(err / bound))
    print(f"{label}: max |err| / bound = {worst:.3f} (bound = 2^-20 x magnitude)")
    assert worst <= 1.0, label


@pytest.mark.parametrize("shape,smooth", [("tiny", False), ("tiny", True), ("512sq", False), ("512sq", True)])
def test_w8a8_block_each_linear_on_the_gpu_input(shape, smooth):
    inp, qws, sm = _w8a8_case(shape, smooth)
    sh = inp.shape
    R, H, nh, d, L = sh.R, sh.hidden, sh.heads, sh.head_dim, sh.L
    dims = dims_of(sh)
    reg = _regions(sh)
    assert D.dit_workspace_bytes(dims, sh.L, sh.N, 4) == reg["end"]
    rows = np.arange(R) if R <= 512 else _sample_rows(sh, seed=23)
    x_in = np.concatenate([inp.txt, inp.img]).astype(np.float64)
    mod = np.asarray(inp.mod, np.float64)[np.asarray(inp.mod_map)[rows]]
    cos, sin = O.rope_tables(O.positions(L, sh.grid_h, sh.grid_w), d)
    mdev = modulation_dev(inp)
    f32 = lambda bits: _f64(bits).astype(np.float32)

    # ---- run 1: the MLP gate zeroed, so the block's output is x_mid = x + gate_a W8A8(o)
    inp_mid = DI.block_inputs(shape, norm_weights=True)
    inp_mid.mod[:, 5, :] = 0.0
    ws = workspace(reg["end"])
    x_mid = _run(inp_mid, qws, sm, ws)

    # qkv: the block's q, k, vt against the oracle's stage on the GPU's h
    h_gpu = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    D.dit_modnorm(dims, dev(inp.txt) if L else None, dev(inp.img), opt_dev(inp.norm1), mdev, 0, h_gpu)
    D.dit_check()
    hb = bf16_bits(h_gpu)[rows]
    qh, sh_ = O.quantize_rows(f32(hb), sm[0])
    qkv = O.w8a8_linear(qh, sh_, *qws[0])
    q_ref = O.rotate(O.qk_rmsnorm(qkv[:, :H].reshape(-1, nh, d), inp.q_norm, sh.qk_eps), cos[rows], sin[rows])
    k_ref = O.rotate(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(-1, nh, d), inp.k_norm, sh.qk_eps), cos[rows], sin[rows])
    v_ref = qkv[:, 2 * H:].reshape(-1, nh, d)
    q_ws = _bf16_view(ws, reg["q"], (nh, R, d))
    k_ws = _bf16_view(ws, reg["k"], (nh, R, d))
    vt_ws = _bf16_view(ws, reg["vt"], (nh, d, _ru(R, 8)))
    for name, got_bits, ref in (("q", bf16_bits(q_ws)[:, rows, :].transpose(1, 0, 2), q_ref),
                                ("k", bf16_bits(k_ws)[:, rows, :].transpose(1, 0, 2), k_ref),
                                ("v", bf16_bits(vt_ws)[:, :, rows].transpose(2, 0, 1), v_ref)):
        got = _f64(got_bits)
        # the GPU's float32 value rounded once to bf16 against the float64 value: within one bf16
        # step of it (2^-8 relative), far below what a wrong scale, divisor or row would move it
        err = np.abs(got - ref)
        worst = float(np.max(err / (2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * rms(ref))))
        print(f"{shape} smooth={smooth} qkv stage, {name}: max |err| / one bf16 step = {worst:.3f}")
        assert worst <= 1.0, name

    # out: the o codes in the workspace are the quantisation of the GPU's own attention output
    o_gpu = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    D.dit_attention_qknorm(dims, R, q_ws, k_ws, vt_ws, opt_dev(inp.q_norm), opt_dev(inp.k_norm), o_gpu)
    D.dit_check()
    qo, so = O.quantize_rows(f32(bf16_bits(o_gpu)[rows]), sm[1])
    o_codes = _f64(bf16_bits(_bf16_view(ws, reg["o"], (R, H)))[rows])
    np.testing.assert_array_equal(o_codes, qo.astype(np.float64))
    lin1 = O.w8a8_linear(qo, so, *qws[1])
    ref_mid = x_in[rows] + mod[:, 2, :] * lin1
    _fp32_close(x_mid[rows], ref_mid, np.abs(x_in[rows]) + np.abs(mod[:, 2, :] * lin1),
                f"{shape} smooth={smooth} out stage")

    # ---- run 2: the whole block
    ws2 = workspace(reg["end"])
    out = _run(inp, qws, sm, ws2)
    # up: h2 from the GPU's x_mid; its codes in the workspace bit for bit
    xm = torch.from_numpy(x_mid.astype(np.float32)).cuda()
    h2_gpu = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    D.dit_modnorm(dims, xm[:L].contiguous() if L else None, xm[L:].contiguous(), opt_dev(inp.norm2), mdev, 1, h2_gpu)
    D.dit_check()
    qh2, sh2 = O.quantize_rows(f32(bf16_bits(h2_gpu)[rows]), sm[2])
    h2_codes = _f64(bf16_bits(_bf16_view(ws2, reg["h"], (R, H)))[rows])
    np.testing.assert_array_equal(h2_codes, qh2.astype(np.float64))
    # the SwiGLU output's codes and scales: equal but where a bf16 value's last bit differs
    a_ref = _bf16_round(O.swiglu_interleaved(O.w8a8_linear(qh2, sh2, *qws[2])))
    qa_ref, sa_ref = O.quantize_rows(a_ref.astype(np.float32), sm[3])
    a_codes = _f64(bf16_bits(_bf16_view(ws2, reg["a"], (R, sh.ffn)))[rows])
    sa_gpu = ws2[reg["sa"]:reg["sa"] + 4 * R].view(torch.float32).cpu().numpy()[rows]
    diff = np.abs(a_codes - qa_ref.astype(np.float64))
    frac = float(np.count_nonzero(diff)) / diff.size
    srel = float(np.max(np.abs(sa_gpu.astype(np.float64) - sa_ref) / np.maximum(sa_ref, 1e-30)))
    print(f"{shape} smooth={smooth} up stage: codes differing {frac:.2e} (max step {diff.max():.0f}), "
          f"scales max rel diff {srel:.2e}")
    assert diff.max() <= 1 and frac <= 1e-3 and srel <= 2.0 ** -7
    # down: the block's output from the workspace's a codes and scales
    lin3 = O.w8a8_linear(a_codes.astype(np.int8), sa_gpu, *qws[3])
    ref_out = x_mid[rows] + mod[:, 5, :] * lin3
    _fp32_close(out[rows], ref_out, np.abs(x_mid[rows]) + np.abs(mod[:, 5, :] * lin3),
                f"{shape} smooth={smooth} down stage")
