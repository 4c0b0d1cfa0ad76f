"""Pins of the oracle's block forward: closed forms, invariants and scalar brute force."""

import math

import numpy as np
import pytest

import oracle as O
from tests import brute


def _tiny_case(seed=0, H=8, heads=2, d=4, F=6, L=2, gh=2, gw=2, M=None):
    g = np.random.default_rng(seed)
    R = L + gh * gw
    x = g.standard_normal((R, H))
    Wq, Wk, Wv = (0.3 * g.standard_normal((H, H)) for _ in range(3))
    Wo = 0.3 * g.standard_normal((H, H))
    Wg, Wu = 0.3 * g.standard_normal((F, H)), 0.3 * g.standard_normal((F, H))
    Wd = 0.3 * g.standard_normal((H, F))
    M = R if M is None else M
    mod = 0.3 * g.standard_normal((M, 6, H))
    mod_map = (np.arange(R) % M).astype(np.int32)
    pos = O.positions(L, gh, gw)
    # head_dim 4 is not one of the contract's widths: give it a hand-made table with distinct angles
    ang = g.uniform(-3, 3, size=(R, d // 2))
    cos, sin = np.cos(ang), np.sin(ang)
    return dict(x=x, Wq=Wq, Wk=Wk, Wv=Wv, Wo=Wo, Wg=Wg, Wu=Wu, Wd=Wd, mod=mod, mod_map=mod_map,
                cos=cos, sin=sin, heads=heads, d=d, pos=pos)


def _fused(c):
    F = c["Wg"].shape[0]
    H = c["Wg"].shape[1]
    Wup = np.empty((2 * F, H))
    Wup[0::2] = c["Wg"]   # gate j at row 2j
    Wup[1::2] = c["Wu"]   # up j at row 2j + 1
    Wqkv = np.concatenate([c["Wq"], c["Wk"], c["Wv"]], axis=0)  # all-Q, all-K, all-V
    return (Wqkv, c["Wo"], Wup, c["Wd"])


def _brute(c, eps, qk_eps, **kw):
    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(6)] for r in range(len(c["x"]))]
    y = brute.block([list(r) for r in c["x"]], c["Wq"].tolist(), c["Wk"].tolist(), c["Wv"].tolist(),
                    c["Wo"].tolist(), c["Wg"].tolist(), c["Wu"].tolist(), c["Wd"].tolist(), mod_rows,
                    c["cos"].tolist(), c["sin"].tolist(), c["heads"], c["d"], eps, qk_eps, **kw)
    return np.array(y)


@pytest.mark.parametrize("seed,M", [(0, None), (1, 2), (2, 1)])
def test_block_matches_scalar_brute_force(seed, M):
    c = _tiny_case(seed, M=M)
    eps, qk_eps = 1e-3, 1e-2  # large enough that dropping either changes the result
    y = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                             c["heads"], c["d"], eps=eps, qk_eps=qk_eps)
    yb = _brute(c, eps, qk_eps)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_block_norm_weights_match_brute_force():
    c = _tiny_case(5)
    g = np.random.default_rng(9)
    H, d = c["x"].shape[1], c["d"]
    n1, n2 = 1 + 0.2 * g.standard_normal(H), 1 + 0.2 * g.standard_normal(H)
    qn, kn = 1 + 0.2 * g.standard_normal(d), 1 + 0.2 * g.standard_normal(d)
    y = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                             c["heads"], c["d"], norm1=n1, norm2=n2, q_norm=qn, k_norm=kn,
                             eps=1e-6, qk_eps=1e-6)
    yb = _brute(c, 1e-6, 1e-6, norm1=list(n1), norm2=list(n2), qn=list(qn), kn=list(kn))
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    c = _tiny_case(3, L=3, gh=3, gw=3)
    full = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                                c["heads"], c["d"])
    rows = np.array([0, 4, 11, 7])
    part = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                                c["heads"], c["d"], rows=rows)
    np.testing.assert_array_equal(part, full[rows])


def test_zero_gates_leave_residual_bitwise():
    c = _tiny_case(4)
    c["mod"][:, 2, :] = 0.0
    c["mod"][:, 5, :] = 0.0
    y = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                             c["heads"], c["d"])
    assert np.array_equal(y, c["x"])


def test_gate_linearity_of_each_branch():
    # x_out - x is gate_a * attn + gate_m * mlp(x + gate_a * attn): with gate_m = 0 the update is
    # exactly proportional to gate_a when gate_a is a constant multiple.
    c = _tiny_case(6)
    c["mod"][:, 5, :] = 0.0
    c["mod"][:, 2, :] = 1.0
    y1 = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    c["mod"][:, 2, :] = 0.5
    y2 = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    np.testing.assert_allclose(y2 - c["x"], 0.5 * (y1 - c["x"]), rtol=1e-12, atol=1e-14)


def test_gate_rows_of_up_zero_silence_mlp():
    # Only the up rows (2j+1) nonzero: gate = 0, silu(0) = 0, so the MLP adds nothing.
    c = _tiny_case(7)
    c["Wg"][:] = 0.0
    W = _fused(c)
    c2 = dict(c)
    c2["mod"] = c["mod"].copy()
    c2["mod"][:, 5, :] = 0.0  # gate_m = 0: MLP disabled by the gate instead
    y = O.block_forward_rows(c["x"], W, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    y_nomlp = O.block_forward_rows(c["x"], W, c2["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    np.testing.assert_array_equal(y, y_nomlp)


def test_swiglu_pairs_one_hot():
    # u = [g0, u0, g1, u1, ...]: a_j = silu(g_j) * u_j, pairs taken from rows 2j and 2j+1 (gluRows)
    u = np.array([[0.5, 2.0, -1.0, 3.0, 0.0, 7.0]])
    a = O.swiglu_interleaved(u)
    s = lambda z: z / (1 + math.exp(-z))
    assert np.allclose(a, [[s(0.5) * 2.0, s(-1.0) * 3.0, 0.0]], rtol=0, atol=1e-15)


def test_glu_rows_golden():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "gizai_glu_rows.txt")
    line = [l for l in open(path) if l.startswith("packed_rows")][0].split()[1:]
    F = 3
    gate = np.arange(F) * 10.0 + 1.0      # gate j marked 1, 11, 21
    up = np.arange(F) * 10.0 + 5.0        # up j marked 5, 15, 25
    names = {}
    for j in range(F):
        names[f"gate{j}"] = gate[j]
        names[f"up{j}"] = up[j]
    packed = np.array([names[n] for n in line])
    # the oracle reads gate from even rows and up from odd rows: with silu replaced by identity
    # on these markers, a_j pairs gate j with up j
    assert np.array_equal(packed[0::2], gate) and np.array_equal(packed[1::2], up)


def test_identity_out_projection_passes_attention_through():
    # Wout = I, gate_a = 1, gate_m = 0: x_out - x equals the attention output o exactly.
    c = _tiny_case(8)
    H = c["x"].shape[1]
    c["Wo"] = np.eye(H)
    c["mod"][:, 2, :] = 1.0
    c["mod"][:, 5, :] = 0.0
    W = _fused(c)
    y = O.block_forward_rows(c["x"], W, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    sa, ca = c["mod"][c["mod_map"], 0], c["mod"][c["mod_map"], 1]
    h = O.modulated_rmsnorm(c["x"], None, sa, ca, 1e-6)
    R = len(h)
    q = (h @ c["Wq"].T).reshape(R, c["heads"], c["d"])
    k = (h @ c["Wk"].T).reshape(R, c["heads"], c["d"])
    v = (h @ c["Wv"].T).reshape(R, c["heads"], c["d"])
    q = O.rope_apply(O.qk_rmsnorm(q, None, 1e-6), c["cos"], c["sin"])
    k = O.rope_apply(O.qk_rmsnorm(k, None, 1e-6), c["cos"], c["sin"])
    np.testing.assert_allclose(y - c["x"], O.attention(q, k, v), rtol=0, atol=1e-13)
