"""Pins of the oracle's parallel (single-stream) block [gizai:dit, Block.parallel]: scalar brute
force, closed forms of the modulated LayerNorm, invariants, and a planted mistake."""

import numpy as np
import pytest

import oracle as O
import oracle.dit as OD
from tests import brute
from tests.test_oracle_block import _fused, _tiny_case


def _case(seed, M=None, **kw):
    c = _tiny_case(seed, M=M, **kw)
    g = np.random.default_rng(100 + seed)
    c["mod"] = 0.3 * g.standard_normal((c["mod"].shape[0], 3, c["x"].shape[1]))
    return c


def _oracle(c, eps, qk_eps, **kw):
    return O.parallel_block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"],
                                         c["heads"], c["d"], eps=eps, qk_eps=qk_eps, **kw)


def _brute(c, eps, qk_eps, **kw):
    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(3)] for r in range(len(c["x"]))]
    y = brute.parallel_block([list(r) for r in c["x"]], c["Wq"].tolist(), c["Wk"].tolist(), c["Wv"].tolist(),
                             c["Wo"].tolist(), c["Wg"].tolist(), c["Wu"].tolist(), c["Wd"].tolist(), mod_rows,
                             c["cos"].tolist(), c["sin"].tolist(), c["heads"], c["d"], eps, qk_eps, **kw)
    return np.array(y)


@pytest.mark.parametrize("seed,M", [(0, None), (1, 2), (2, 1)])
def test_parallel_block_matches_scalar_brute_force(seed, M):
    c = _case(seed, M=M)
    eps, qk_eps = 0.5, 1e-2  # large enough that dropping either changes the result
    np.testing.assert_allclose(_oracle(c, eps, qk_eps), _brute(c, eps, qk_eps), rtol=1e-12, atol=1e-12)


def test_parallel_block_norm_weights_match_brute_force():
    c = _case(5)
    g = np.random.default_rng(9)
    H, d = c["x"].shape[1], c["d"]
    w, qn, kn = (1 + 0.2 * g.standard_normal(n) for n in (H, d, d))
    y = _oracle(c, 1e-6, 1e-6, norm=w, q_norm=qn, k_norm=kn)
    yb = _brute(c, 1e-6, 1e-6, norm=list(w), qn=list(qn), kn=list(kn))
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_modulated_layernorm_closed_forms():
    H, eps = 8, 0.25
    shift, scale = np.linspace(-1, 1, H), np.linspace(0.5, -0.5, H)
    # a constant row has no deviation: the norm is the shift alone, whatever the constant and eps
    np.testing.assert_array_equal(O.modulated_layernorm(np.full((1, H), 3.7), None, shift, scale, eps)[0], shift)
    # mu +/- delta alternating: variance delta^2, so each value is +/- delta / sqrt(delta^2 + eps)
    mu, delta = 2.0, 0.6
    x = mu + delta * np.array([1, -1] * (H // 2), dtype=np.float64)
    ref = np.array([1, -1] * (H // 2)) * delta / np.sqrt(delta ** 2 + eps) * (1 + scale) + shift
    np.testing.assert_allclose(O.modulated_layernorm(x[None], None, shift, scale, eps)[0], ref, rtol=1e-15,
                               atol=1e-15)
    # unlike the RMS norm, a LayerNorm does not see a constant added to the row
    g = np.random.default_rng(1)
    y = g.standard_normal((3, H))
    np.testing.assert_allclose(O.modulated_layernorm(y + 5.0, None, shift, scale, eps),
                               O.modulated_layernorm(y, None, shift, scale, eps), rtol=1e-12, atol=1e-12)
    assert not np.allclose(O.modulated_rmsnorm(y + 5.0, None, shift, scale, eps),
                           O.modulated_rmsnorm(y, None, shift, scale, eps))


def test_zero_gate_is_identity_and_gate_is_linear():
    c = _case(3)
    c["mod"][:, 2, :] = 0.0
    np.testing.assert_array_equal(_oracle(c, 1e-6, 1e-6), c["x"])
    c = _case(4)
    y1 = _oracle(c, 1e-6, 1e-6) - c["x"]
    c["mod"][:, 2, :] *= 2.5
    y2 = _oracle(c, 1e-6, 1e-6) - c["x"]
    np.testing.assert_allclose(y2, 2.5 * y1, rtol=1e-12, atol=1e-13)


def test_zero_up_weights_leave_the_attention_branch():
    # Wup = 0 gives u = 0 and silu(0) * 0 = 0: the output is x + gate * (o Wout^T), o the attention of
    # the LayerNorm'd rows, composed here from the pinned pieces
    c = _case(6)
    c["Wg"][:] = 0.0
    c["Wu"][:] = 0.0
    eps, qk_eps = 1e-6, 1e-6
    R, H = c["x"].shape
    nh, d = c["heads"], c["d"]
    m = c["mod"][c["mod_map"]]
    h = O.modulated_layernorm(c["x"], None, m[:, 0], m[:, 1], eps)
    q = O.rope_apply(O.qk_rmsnorm((h @ c["Wq"].T).reshape(R, nh, d), None, qk_eps), c["cos"], c["sin"])
    k = O.rope_apply(O.qk_rmsnorm((h @ c["Wk"].T).reshape(R, nh, d), None, qk_eps), c["cos"], c["sin"])
    v = (h @ c["Wv"].T).reshape(R, nh, d)
    ref = c["x"] + m[:, 2] * (O.attention(q, k, v) @ c["Wo"].T)
    np.testing.assert_allclose(_oracle(c, eps, qk_eps), ref, rtol=1e-12, atol=1e-12)


def test_parallel_sampled_rows_equal_full_rows():
    c = _case(7, L=3, gh=3, gw=3)
    full = _oracle(c, 1e-6, 1e-6)
    rows = np.array([0, 4, 11, 7])
    part = _oracle(c, 1e-6, 1e-6, rows=rows)
    np.testing.assert_array_equal(part, full[rows])


def test_planted_rmsnorm_for_layernorm_fails_the_brute_force_pin(monkeypatch):
    c = _case(8)
    c["x"] = c["x"] + 1.5  # rows with a clear mean, where the two norms differ
    yb = _brute(c, 1e-6, 1e-6)
    monkeypatch.setattr(OD, "modulated_layernorm", O.modulated_rmsnorm)
    y = _oracle(c, 1e-6, 1e-6)
    assert not np.allclose(y, yb, rtol=1e-6, atol=1e-6)
