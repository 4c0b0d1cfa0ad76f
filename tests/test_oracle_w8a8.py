"""Pins of the W8A8 oracle [klein, section 5 (int8 detail); log entries D4 (quantize_weight,
quantize_rows, linear_int8) and D5 (SmoothQuant)]: the code rounding (half to even, clipping, zero
scales) on hand-picked values, the quantisation error bound, the smoothing formula's balance at
alpha = 1/2, the integer dot product against a scalar loop, and the whole W8A8 block against a
scalar brute force whose linears quantise with pure-Python arithmetic (no NumPy)."""

import struct

import numpy as np
import pytest

import oracle as O
from tests import brute
from tests.test_oracle_block import _fused, _tiny_case


def test_codes_round_half_to_even_and_clip():
    s = np.float32(0.5)
    v = np.array([[1.25, 0.75, -0.25, 0.25, 63.5, -63.75, 100.0, -1e9, 0.0]], np.float32)
    # v / s = 2.5 -> 2, 1.5 -> 2, -0.5 -> -0, 0.5 -> 0, 127 -> 127, -127.5 -> -128 -> clip -127,
    # 200 -> clip 127, huge -> clip -127, 0 -> 0
    got = O.quantize_codes(v, np.full((1, 1), s, np.float32))
    np.testing.assert_array_equal(got, [[2, 2, 0, 0, 127, -127, 127, -127, 0]])
    z = O.quantize_codes(np.array([[3.0, -2.0]], np.float32), np.zeros((1, 1), np.float32))
    np.testing.assert_array_equal(z, [[0, 0]])  # a zero scale gives zero codes


def test_rows_scale_is_absmax_over_127_and_error_is_half_a_step():
    g = np.random.default_rng(0)
    x = (g.standard_normal((9, 40)) * g.uniform(0.1, 10, size=(9, 1))).astype(np.float32)
    x[3] = 0.0  # a zero row
    q, sc = O.quantize_rows(x)
    np.testing.assert_array_equal(sc, (np.abs(x).max(axis=1) / np.float32(127)).astype(np.float32))
    assert sc[3] == 0 and not q[3].any()
    for r in range(9):
        if sc[r] == 0:
            continue
        j = np.argmax(np.abs(x[r]))
        assert abs(int(q[r, j])) == 127  # the largest element takes the largest code
        err = np.abs(x[r].astype(np.float64) - q[r].astype(np.float64) * float(sc[r]))
        assert np.all(err <= 0.5 * float(sc[r]) * (1 + 2 ** -20))


def test_weight_is_per_output_channel_with_the_fold():
    g = np.random.default_rng(1)
    w = g.standard_normal((6, 16)).astype(np.float32)
    s = np.float32(2.0) ** g.integers(-2, 3, size=16).astype(np.float32)  # exact folds
    q, sc = O.quantize_weight(w, s)
    ws = (w * s[None, :]).astype(np.float32)
    for o in range(6):
        assert sc[o] == np.float32(np.abs(ws[o]).max() / np.float32(127))
        assert abs(int(q[o, np.argmax(np.abs(ws[o]))])) == 127
    # folding then quantising equals quantising the pre-multiplied weight
    q2, sc2 = O.quantize_weight(ws)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(sc, sc2)


def test_smoothing_balances_the_ranges_at_alpha_half():
    g = np.random.default_rng(2)
    xa = g.uniform(0.1, 50, size=32)
    wa = g.uniform(0.01, 2, size=32)
    s = O.smooth_scales(xa, wa, 0.5).astype(np.float64)
    # max|X_j| / s_j = max|W_j| s_j = sqrt(max|X_j| max|W_j|): the ranges meet in the middle
    np.testing.assert_allclose(xa / s, wa * s, rtol=1e-6)
    np.testing.assert_allclose(xa / s, np.sqrt(xa * wa), rtol=1e-6)
    # alpha = 1 moves everything onto the weight, alpha = 0 nothing; zero statistics give 1
    np.testing.assert_allclose(O.smooth_scales(xa, wa, 1.0), xa.astype(np.float32), rtol=1e-6)
    np.testing.assert_allclose(O.smooth_scales(xa, wa, 0.0), (1 / wa).astype(np.float32), rtol=1e-6)
    assert O.smooth_scales(np.array([0.0, 1.0]), np.array([1.0, 0.0]), 0.5).tolist() == [1.0, 1.0]


def test_integer_dot_matches_a_scalar_loop():
    g = np.random.default_rng(3)
    qx = g.integers(-127, 128, size=(5, 33)).astype(np.int8)
    qw = g.integers(-127, 128, size=(4, 33)).astype(np.int8)
    sx = g.uniform(0.01, 1, size=5).astype(np.float32)
    sw = g.uniform(0.01, 1, size=4).astype(np.float32)
    got = O.w8a8_linear(qx, sx, qw, sw)
    for r in range(5):
        for o in range(4):
            acc = sum(int(qx[r, j]) * int(qw[o, j]) for j in range(33))
            assert got[r, o] == acc * float(sx[r]) * float(sw[o])


# ---------------------------------------------------------------------- scalar W8A8 brute force

def _f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def _bf16(v):
    """Round a float to float32, then to bfloat16 (nearest, ties to even), pure Python."""
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    keep, rest = u >> 16, u & 0xFFFF
    if rest > 0x8000 or (rest == 0x8000 and keep & 1):
        keep += 1
    return struct.unpack("<f", struct.pack("<I", (keep & 0xFFFF) << 16))[0]


def _quant_row(row, smooth=None):
    """Per-token codes and scale of one activation row (its bf16 values, float32 arithmetic)."""
    v = [_bf16(a) for a in row]
    if smooth is not None:
        v = [_f32(a / s) for a, s in zip(v, smooth)]
    amax = max(abs(a) for a in v)
    sc = _f32(amax / 127.0)
    codes = [0 if sc == 0 else max(-127, min(127, round(_f32(a / sc)))) for a in v]
    return codes, sc


def _quant_matrix(W, smooth=None):
    """Per-output-channel codes and scales of a weight (rows = output channels), fold included."""
    out = []
    for row in W:
        v = [_f32(a) for a in row]
        if smooth is not None:
            v = [_f32(a * s) for a, s in zip(v, smooth)]
        amax = max(abs(a) for a in v)
        sc = _f32(amax / 127.0)
        out.append(([0 if sc == 0 else max(-127, min(127, round(_f32(a / sc)))) for a in v], sc))
    return out


@pytest.mark.parametrize("seed,use_smooth", [(0, False), (1, True)])
def test_w8a8_block_matches_scalar_brute_force(seed, use_smooth):
    c = _tiny_case(seed + 20)
    eps, qk_eps = 1e-3, 1e-2
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    g = np.random.default_rng(seed + 40)
    smooth = None
    if use_smooth:
        smooth = [g.uniform(0.5, 2.0, size=n).astype(np.float32) for n in (H, H, H, F)]
    # quantised weights: per output row, so splitting Q/K/V and gate/up keeps every row's scale
    mats = {k: c[k].astype(np.float32) for k in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
    sm_of = {"Wq": 0, "Wk": 0, "Wv": 0, "Wo": 1, "Wg": 2, "Wu": 2, "Wd": 3}
    quant = {k: _quant_matrix(mats[k].tolist(), None if smooth is None else smooth[sm_of[k]].tolist())
             for k in mats}

    def linear_for(name):
        qrows = quant[name]
        sm = None if smooth is None else smooth[sm_of[name]].tolist()

        def lin(_W, row):
            codes, sc = _quant_row(row, sm)
            return [sum(a * b for a, b in zip(codes, qc)) * sc * sw for qc, sw in qrows]
        return lin

    # brute.block calls linear(W, row) for each matrix; pick the quantised form by identity
    def linear(W, row):
        for k in mats:
            if W is brute_mats[k]:
                return linear_for(k)(W, row)
        raise AssertionError("unknown weight")

    brute_mats = {k: mats[k].tolist() for k in mats}
    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(6)] for r in range(len(c["x"]))]
    yb = np.array(brute.block([list(r) for r in c["x"]], brute_mats["Wq"], brute_mats["Wk"], brute_mats["Wv"],
                              brute_mats["Wo"], brute_mats["Wg"], brute_mats["Wu"], brute_mats["Wd"], mod_rows,
                              c["cos"].tolist(), c["sin"].tolist(), c["heads"], c["d"], eps, qk_eps,
                              linear=linear))
    # the oracle on the fused weights, quantised by quantize_weight
    Wqkv, Wo, Wup, Wd = _fused(c)
    qws = [O.quantize_weight(W.astype(np.float32), None if smooth is None else smooth[i])
           for i, W in enumerate((Wqkv, Wo, Wup, Wd))]
    y = O.block_forward_w8a8_rows(c["x"], qws, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"],
                                  eps=eps, qk_eps=qk_eps, smooth=smooth)
    np.testing.assert_allclose(y, yb, rtol=1e-9, atol=1e-9)
    # and it is a perturbation of the float block, not the float block
    yf = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"],
                              eps=eps, qk_eps=qk_eps)
    rel = np.abs(y - yf).max() / np.sqrt(np.mean(yf ** 2))
    assert 1e-5 < rel < 0.1, rel


# ------------------------------------------------------------ parallel and double-stream W8A8 blocks

def _quantised_linear(qrows, sm):
    """linear(W, row) of a quantised weight (rows of (codes, scale)): per-token codes of the row."""
    def lin(_W, row):
        codes, sc = _quant_row(row, sm)
        return [sum(a * b for a, b in zip(codes, qc)) * sc * sw for qc, sw in qrows]
    return lin


@pytest.mark.parametrize("seed,use_smooth", [(0, False), (1, True)])
def test_parallel_w8a8_block_matches_scalar_brute_force(seed, use_smooth):
    # linear1 = [Wqkv ; Wup] over h; linear2 = [Wout | Wdown] over the joined row [o | a], one code
    # row and one scale per output channel over all H + F inputs [klein, section 5: single linear1
    # and linear2]
    from tests.test_oracle_parallel import _case
    c = _case(seed + 30)
    eps, qk_eps = 0.5, 1e-2
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    g = np.random.default_rng(seed + 50)
    sm1 = g.uniform(0.5, 2.0, size=H).astype(np.float32) if use_smooth else None
    sm2 = g.uniform(0.5, 2.0, size=H + F).astype(np.float32) if use_smooth else None
    lin1 = {k: _quant_matrix(c[k].astype(np.float32).tolist(), None if sm1 is None else sm1.tolist())
            for k in ("Wq", "Wk", "Wv", "Wg", "Wu")}
    W2 = np.concatenate([c["Wo"], c["Wd"]], axis=1).astype(np.float32)
    lin2 = _quant_matrix(W2.tolist(), None if sm2 is None else sm2.tolist())
    mats = {k: c[k].tolist() for k in lin1}

    def linear(W, row):
        for k in mats:
            if W is mats[k]:
                return _quantised_linear(lin1[k], None if sm1 is None else sm1.tolist())(W, row)
        raise AssertionError("unknown weight")

    def linear2(o, a):
        return _quantised_linear(lin2, None if sm2 is None else sm2.tolist())(None, list(o) + list(a))

    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(3)] for r in range(len(c["x"]))]
    yb = np.array(brute.parallel_block([list(r) for r in c["x"]], mats["Wq"], mats["Wk"], mats["Wv"],
                                       c["Wo"].tolist(), mats["Wg"], mats["Wu"], c["Wd"].tolist(), mod_rows,
                                       c["cos"].tolist(), c["sin"].tolist(), c["heads"], c["d"], eps, qk_eps,
                                       linear=linear, linear2=linear2))
    Wqkv, _, Wup, _ = _fused(c)
    q1 = O.quantize_weight(np.concatenate([Wqkv, Wup], axis=0).astype(np.float32), sm1)
    q2 = O.quantize_weight(W2, sm2)
    y = O.parallel_block_forward_w8a8_rows(c["x"], q1, q2, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                           c["d"], eps=eps, qk_eps=qk_eps, smooth1=sm1, smooth2=sm2)
    np.testing.assert_allclose(y, yb, rtol=1e-9, atol=1e-9)
    # a perturbation of the float parallel block, not the float block
    yf = O.parallel_block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                       c["d"], eps=eps, qk_eps=qk_eps)
    rel = np.abs(y - yf).max() / np.sqrt(np.mean(yf ** 2))
    assert 1e-5 < rel < 0.1, rel


def test_parallel_w8a8_linear2_is_one_joint_quantisation():
    # quantising [o | a] and [Wout | Wdown] as one row each is not the sum of two separately
    # quantised linears (different per-token and per-channel scales): the planted mistake is caught
    from tests.test_oracle_parallel import _case
    c = _case(7)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wqkv, _, Wup, _ = _fused(c)
    q1 = O.quantize_weight(np.concatenate([Wqkv, Wup], axis=0).astype(np.float32))
    W2 = np.concatenate([c["Wo"], c["Wd"]], axis=1).astype(np.float32)
    y = O.parallel_block_forward_w8a8_rows(c["x"], q1, O.quantize_weight(W2), c["mod"], c["mod_map"], c["cos"],
                                           c["sin"], c["heads"], c["d"])
    # the mistaken form: linear2 as two W8A8 linears added
    qo, qd = O.quantize_weight(c["Wo"].astype(np.float32)), O.quantize_weight(c["Wd"].astype(np.float32))
    x = c["x"]
    m = c["mod"][c["mod_map"]]
    h = O.modulated_layernorm(x, None, m[:, 0], m[:, 1], 1e-6)
    u = O.w8a8_linear_f(h, *q1)
    nh, d = c["heads"], c["d"]
    R = x.shape[0]
    q = O.rotate(O.qk_rmsnorm(u[:, :H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    k = O.rotate(O.qk_rmsnorm(u[:, H:2 * H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    o = O.attention(q, k, u[:, 2 * H:3 * H].reshape(R, nh, d))
    a = O.swiglu_interleaved(u[:, 3 * H:])
    wrong = x + m[:, 2] * (O.w8a8_linear_f(o, *qo) + O.w8a8_linear_f(a, *qd))
    assert np.abs(wrong - y).max() > 1e-4 * np.abs(y).max()


@pytest.mark.parametrize("seed,L,use_smooth", [(0, 2, False), (1, 3, True), (2, 0, True)])
def test_double_w8a8_block_matches_scalar_brute_force(seed, L, use_smooth):
    # each stream's four linears quantised with its own divisors [klein, section 5: double img / txt
    # qkv, proj, mlp.0, mlp.2]
    from tests.test_oracle_double import _stream
    c = _tiny_case(seed + 60, L=L)
    eps, qk_eps = 1e-3, 1e-2
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    g = np.random.default_rng(seed + 70)
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    ins = (H, H, H, F)
    sm_t = [g.uniform(0.5, 2.0, size=n).astype(np.float32) for n in ins] if use_smooth else None
    sm_i = [g.uniform(0.5, 2.0, size=n).astype(np.float32) for n in ins] if use_smooth else None
    sm_of = {"Wq": 0, "Wk": 0, "Wv": 0, "Wo": 1, "Wg": 2, "Wu": 2, "Wd": 3}
    order = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")
    brute_t = [Wt[k].astype(np.float32).tolist() for k in order]
    brute_i = [Wi[k].astype(np.float32).tolist() for k in order]
    table = []
    for W, sm, mats in ((Wt, sm_t, brute_t), (Wi, sm_i, brute_i)):
        for k, mat in zip(order, mats):
            s = None if sm is None else sm[sm_of[k]].tolist()
            table.append((mat, _quantised_linear(_quant_matrix(W[k].astype(np.float32).tolist(), s), s)))

    def linear(W, row):
        for mat, lin in table:
            if W is mat:
                return lin(W, row)
        raise AssertionError("unknown weight")

    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(6)] for r in range(len(c["x"]))]
    yb = np.array(brute.double_block([list(r) for r in c["x"]], L, brute_t, brute_i, mod_rows, c["cos"].tolist(),
                                     c["sin"].tolist(), c["heads"], c["d"], eps, qk_eps, linear=linear))
    qt = [O.quantize_weight(W.astype(np.float32), None if sm_t is None else sm_t[i]) for i, W in enumerate(_fused(Wt))]
    qi = [O.quantize_weight(W.astype(np.float32), None if sm_i is None else sm_i[i]) for i, W in enumerate(_fused(Wi))]
    y = O.double_block_forward_w8a8_rows(c["x"], qt, qi, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                         c["d"], L, eps=eps, qk_eps=qk_eps, smooth_txt=sm_t, smooth_img=sm_i)
    np.testing.assert_allclose(y, yb, rtol=1e-9, atol=1e-9)


def test_double_w8a8_with_shared_weights_is_the_sequential_w8a8_block():
    c = _tiny_case(9, L=3, gh=3, gw=3)
    g = np.random.default_rng(11)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    sm = [g.uniform(0.5, 2.0, size=n).astype(np.float32) for n in (H, H, H, F)]
    qws = [O.quantize_weight(W.astype(np.float32), sm[i]) for i, W in enumerate(_fused(c))]
    seq = O.block_forward_w8a8_rows(c["x"], qws, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"],
                                    smooth=sm)
    dbl = O.double_block_forward_w8a8_rows(c["x"], qws, qws, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                           c["d"], 3, smooth_txt=sm, smooth_img=sm)
    np.testing.assert_array_equal(dbl, seq)
