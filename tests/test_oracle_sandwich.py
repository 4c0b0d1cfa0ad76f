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
