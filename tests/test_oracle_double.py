"""Pins of the oracle's double-stream block: scalar brute force with per-stream weights, reduction
to the (pinned) sequential block when both streams share their weights, and stream separation."""

import numpy as np
import pytest

import oracle as O
from tests import brute
from tests.test_oracle_block import _fused, _tiny_case


def _stream(g, H, F):
    Wq, Wk, Wv = (0.3 * g.standard_normal((H, H)) for _ in range(3))
    return dict(Wq=Wq, Wk=Wk, Wv=Wv, Wo=0.3 * g.standard_normal((H, H)), Wg=0.3 * g.standard_normal((F, H)),
                Wu=0.3 * g.standard_normal((F, H)), Wd=0.3 * g.standard_normal((H, F)))


def _oracle(c, Wt, Wi, L, eps=1e-6, qk_eps=1e-6, **kw):
    return O.double_block_forward_rows(c["x"], _fused(Wt), _fused(Wi), c["mod"], c["mod_map"], c["cos"], c["sin"],
                                       c["heads"], c["d"], L, eps=eps, qk_eps=qk_eps, **kw)


def _brute(c, Wt, Wi, L, eps, qk_eps, **kw):
    mod_rows = [[list(c["mod"][c["mod_map"][r], i]) for i in range(6)] for r in range(len(c["x"]))]
    order = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")
    y = brute.double_block([list(r) for r in c["x"]], L, [Wt[k].tolist() for k in order],
                           [Wi[k].tolist() for k in order], mod_rows, c["cos"].tolist(), c["sin"].tolist(),
                           c["heads"], c["d"], eps, qk_eps, **kw)
    return np.array(y)


@pytest.mark.parametrize("seed,L,M", [(0, 2, None), (1, 3, 2), (2, 1, 1), (3, 0, None)])
def test_double_block_matches_scalar_brute_force(seed, L, M):
    c = _tiny_case(seed, L=L, M=M)
    g = np.random.default_rng(200 + seed)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    eps, qk_eps = 1e-3, 1e-2
    np.testing.assert_allclose(_oracle(c, Wt, Wi, L, eps, qk_eps), _brute(c, Wt, Wi, L, eps, qk_eps),
                               rtol=1e-12, atol=1e-12)


def test_double_block_norm_weights_match_brute_force():
    c = _tiny_case(5, L=2)
    g = np.random.default_rng(9)
    H, d, F = c["x"].shape[1], c["d"], c["Wg"].shape[0]
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    nt = tuple(1 + 0.2 * g.standard_normal(n) for n in (H, H, d, d))
    ni = tuple(1 + 0.2 * g.standard_normal(n) for n in (H, H, d, d))
    y = _oracle(c, Wt, Wi, 2, norms_txt=nt, norms_img=ni)
    yb = _brute(c, Wt, Wi, 2, 1e-6, 1e-6, norms_t=[list(a) for a in nt], norms_i=[list(a) for a in ni])
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_shared_weights_reduce_to_the_sequential_block():
    c = _tiny_case(6, L=3, gh=3, gw=3)
    W = {k: c[k] for k in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
    seq = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    np.testing.assert_allclose(_oracle(c, W, W, 3), seq, rtol=1e-13, atol=1e-13)


def test_streams_are_separate():
    # the joint attention mixes all rows, but the MLP acts row by row after it: changing only the
    # text stream's down weights moves the text rows and leaves the image rows bit for bit
    c = _tiny_case(7, L=2)
    g = np.random.default_rng(17)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    y1 = _oracle(c, Wt, Wi, 2)
    Wt2 = dict(Wt)
    Wt2["Wd"] = Wt["Wd"] * 1.5
    y2 = _oracle(c, Wt2, Wi, 2)
    np.testing.assert_array_equal(y1[2:], y2[2:])
    assert not np.allclose(y1[:2], y2[:2])


def test_double_sampled_rows_equal_full_rows():
    c = _tiny_case(8, L=3, gh=3, gw=3)
    g = np.random.default_rng(3)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    full = _oracle(c, Wt, Wi, 3)
    rows = np.array([0, 2, 4, 11, 7])
    np.testing.assert_array_equal(_oracle(c, Wt, Wi, 3, rows=rows), full[rows])
