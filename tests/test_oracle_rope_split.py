"""Pins of the split-halves partial rotation [gizai:dit, prepOf, HEAD]: it is the (pinned) adjacent-
pair rotation seen through a fixed reordering of each head's values; zero angles leave heads
unchanged bit for bit; the last quarter is never touched; pair norms are kept. Through a whole
block, split-halves tables equal adjacent-pair tables on q/k weight columns reordered the same way."""

import numpy as np
import pytest

import oracle as O
from tests.test_oracle_block import _fused, _tiny_case


def _perm(d):
    # head value order that makes split-halves pairs adjacent: [0, h, 1, h+1, ..., h-1, 2h-1, 2h, ..., d-1]
    h = 3 * d // 8
    order = []
    for i in range(h):
        order += [i, i + h]
    return np.array(order + list(range(2 * h, d)))


def _expand(cos, sin, d):
    # adjacent-pair tables for the reordered head: the split tables, then angle 0 for the tail pairs
    R, h = cos.shape
    tail = (d - 2 * h) // 2
    return (np.concatenate([cos, np.ones((R, tail))], axis=1), np.concatenate([sin, np.zeros((R, tail))], axis=1))


@pytest.mark.parametrize("d", [64, 128, 32])
def test_split_is_pair_rotation_of_reordered_head(d):
    g = np.random.default_rng(d)
    R, nh, h = 7, 3, 3 * d // 8
    t = g.standard_normal((R, nh, d))
    ang = g.uniform(-4, 4, size=(R, h))
    cos, sin = np.cos(ang), np.sin(ang)
    P = _perm(d)
    c2, s2 = _expand(cos, sin, d)
    via_pairs = np.empty_like(t)
    via_pairs[..., P] = O.rope_apply(t[..., P], c2, s2)
    np.testing.assert_allclose(O.rope_apply_split(t, cos, sin), via_pairs, rtol=0, atol=1e-14)
    np.testing.assert_allclose(O.rotate(t, cos, sin), via_pairs, rtol=0, atol=1e-14)


def test_split_zero_angle_tail_and_norms():
    g = np.random.default_rng(1)
    d, h = 128, 48
    t = g.standard_normal((5, 2, d))
    np.testing.assert_array_equal(O.rope_apply_split(t, np.ones((5, h)), np.zeros((5, h))), t)
    ang = g.uniform(-3, 3, size=(5, h))
    y = O.rope_apply_split(t, np.cos(ang), np.sin(ang))
    np.testing.assert_array_equal(y[..., 2 * h:], t[..., 2 * h:])
    np.testing.assert_allclose(y[..., :h] ** 2 + y[..., h:2 * h] ** 2, t[..., :h] ** 2 + t[..., h:2 * h] ** 2,
                               rtol=1e-13)
    with pytest.raises(ValueError):
        O.rotate(t, np.ones((5, 40)), np.zeros((5, 40)))


def test_block_with_split_tables_is_block_with_reordered_qk_columns():
    c = _tiny_case(11, H=16, heads=2, d=8, F=6)
    g = np.random.default_rng(5)
    R, H, d, nh = c["x"].shape[0], 16, 8, 2
    h = 3 * d // 8
    ang = g.uniform(-3, 3, size=(R, h))
    cos, sin = np.cos(ang), np.sin(ang)
    qn, kn = 1 + 0.2 * g.standard_normal(d), 1 + 0.2 * g.standard_normal(d)
    y_split = O.block_forward_rows(c["x"], _fused(c), c["mod"], c["mod_map"], cos, sin, nh, d,
                                   q_norm=qn, k_norm=kn)
    P = _perm(d)
    cols = np.concatenate([n * d + P for n in range(nh)])
    c2 = dict(c)
    c2["Wq"], c2["Wk"] = c["Wq"][cols], c["Wk"][cols]
    ce, se = _expand(cos, sin, d)
    y_pairs = O.block_forward_rows(c["x"], _fused(c2), c["mod"], c["mod_map"], ce, se, nh, d,
                                   q_norm=qn[P], k_norm=kn[P])
    np.testing.assert_allclose(y_split, y_pairs, rtol=1e-12, atol=1e-12)
