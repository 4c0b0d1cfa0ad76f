"""Pins of the sandwich block's post-norms [gizai:dit, POST_ATTN, POST_MLP]: scalar brute force,
invariance of each normed branch to a positive scaling of its linear (eps = 0), and linearity in the
post-norm weight."""

import numpy as np
import pytest

import oracle as O
from tests import brute
from tests.test_oracle_block import _brute, _fused, _tiny_case


def _run(c, W, eps=1e-3, **kw):
    return O.block_forward_rows(c["x"], W, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"],
                                eps=eps, qk_eps=1e-2, **kw)


@pytest.mark.parametrize("seed,M", [(0, None), (1, 2)])
def test_sandwich_matches_scalar_brute_force(seed, M):
    c = _tiny_case(seed, M=M)
    g = np.random.default_rng(50 + seed)
    H = c["x"].shape[1]
    pa, pm = 1 + 0.3 * g.standard_normal(H), 1 + 0.3 * g.standard_normal(H)
    y = _run(c, _fused(c), post_attn=pa, post_mlp=pm)
    yb = _brute(c, 1e-3, 1e-2, post_attn=list(pa), post_mlp=list(pm))
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)
    assert not np.allclose(y, _run(c, _fused(c)))


def test_normed_branches_ignore_the_scale_of_their_linear():
    c = _tiny_case(3)
    H = c["x"].shape[1]
    W = _fused(c)
    ones = np.ones(H)
    base = _run(c, W, eps=0.0, post_attn=ones, post_mlp=ones)
    scaled = (W[0], 3.0 * W[1], W[2], 0.25 * W[3])
    np.testing.assert_allclose(_run(c, scaled, eps=0.0, post_attn=ones, post_mlp=ones), base, rtol=1e-12,
                               atol=1e-12)
    assert not np.allclose(_run(c, scaled, eps=0.0), _run(c, W, eps=0.0))  # without the norms it matters


def test_post_weight_scales_the_branch():
    c = _tiny_case(4)
    H = c["x"].shape[1]
    g = np.random.default_rng(2)
    pa = 1 + 0.3 * g.standard_normal(H)
    W = _fused(c)
    # zero MLP gate isolates the attention branch, which is linear in the post weight
    c["mod"][:, 5, :] = 0.0
    d1 = _run(c, W, post_attn=pa) - c["x"]
    d2 = _run(c, W, post_attn=2.0 * pa) - c["x"]
    np.testing.assert_allclose(d2, 2.0 * d1, rtol=1e-12, atol=1e-13)


def test_parallel_sandwich_matches_scalar_brute_force():
    # each branch normed with its own weight, then the one gate over their sum
    from tests.test_oracle_parallel import _case, _oracle, _brute
    c = _case(21)
    H = c["x"].shape[1]
    g = np.random.default_rng(22)
    pa, pm = 1 + 0.3 * g.standard_normal(H), 1 + 0.3 * g.standard_normal(H)
    eps, qk_eps = 1e-3, 1e-2
    for post_attn, post_mlp in ((pa, pm), (pa, None), (None, pm)):
        y = _oracle(c, eps, qk_eps, post_attn=post_attn, post_mlp=post_mlp)
        yb = _brute(c, eps, qk_eps, post_attn=None if post_attn is None else list(post_attn),
                    post_mlp=None if post_mlp is None else list(post_mlp))
        np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)
    # a normed branch ignores a positive scaling of its linear (eps = 0), as in the sequential block
    W = list(_fused(c))
    y1 = O.parallel_block_forward_rows(c["x"], tuple(W), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                       c["d"], eps=0.0, post_attn=pa, post_mlp=pm)
    W[1] = 3.0 * W[1]
    W[3] = 0.5 * W[3]
    y2 = O.parallel_block_forward_rows(c["x"], tuple(W), c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                       c["d"], eps=0.0, post_attn=pa, post_mlp=pm)
    np.testing.assert_allclose(y1, y2, rtol=1e-12, atol=1e-12)


def test_double_sandwich_matches_scalar_brute_force():
    from tests.test_oracle_double import _brute, _oracle, _stream
    c = _tiny_case(23, L=2)
    g = np.random.default_rng(24)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wt, Wi = _stream(g, H, F), _stream(g, H, F)
    pt = (1 + 0.3 * g.standard_normal(H), 1 + 0.3 * g.standard_normal(H))
    pi = (1 + 0.3 * g.standard_normal(H), None)
    y = _oracle(c, Wt, Wi, 2, 1e-3, 1e-2, post_txt=pt, post_img=pi)
    yb = _brute(c, Wt, Wi, 2, 1e-3, 1e-2, post_t=[list(pt[0]), list(pt[1])], post_i=[list(pi[0]), None])
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)
    # the image stream's post weights change the image rows and leave the text rows bit for bit
    y2 = _oracle(c, Wt, Wi, 2, 1e-3, 1e-2, post_txt=pt, post_img=(None, None))
    assert not np.allclose(y[2:], y2[2:])
    np.testing.assert_array_equal(y[:2], y2[:2])
