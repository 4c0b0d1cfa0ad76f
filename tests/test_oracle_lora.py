"""Pins of the LoRA adapter [gizai:dit, withLora, loraOf, weightAt]: the adapter beside the linear and
the merged weight are the same map (checked element by element on integer matrices, where float64
sums are exact), a zero B or A leaves the linear, rank-one closed form, and the block with adapters
equals the block with merged weights while both differ from the plain block."""

import numpy as np
import pytest

import oracle as O
from tests.test_oracle_block import _fused, _tiny_case


def test_adapter_equals_merged_weight_exactly_on_integers():
    g = np.random.default_rng(0)
    x = g.integers(-5, 6, size=(7, 12)).astype(np.float64)
    W = g.integers(-5, 6, size=(9, 12)).astype(np.float64)
    A = g.integers(-3, 4, size=(4, 12)).astype(np.float64)
    B = g.integers(-3, 4, size=(9, 4)).astype(np.float64)
    ref = np.array([[sum(x[r, i] * (W[o, i] + sum(B[o, j] * A[j, i] for j in range(4))) for i in range(12))
                     for o in range(9)] for r in range(7)])
    np.testing.assert_array_equal(O.lora_linear(x, W, A, B), ref)
    np.testing.assert_array_equal(x @ O.lora_merge(W, A, B).T, ref)


def test_zero_factor_and_rank_one():
    g = np.random.default_rng(1)
    x, W = g.standard_normal((5, 8)), g.standard_normal((6, 8))
    A, B = g.standard_normal((3, 8)), g.standard_normal((6, 3))
    np.testing.assert_array_equal(O.lora_linear(x, W, A, np.zeros_like(B)), x @ W.T)
    np.testing.assert_array_equal(O.lora_linear(x, W, np.zeros_like(A), B), x @ W.T)
    a, b = g.standard_normal(8), g.standard_normal(6)
    y = O.lora_linear(x, W, a[None, :], b[:, None])
    np.testing.assert_allclose(y, x @ W.T + np.outer(x @ a, b), rtol=1e-13, atol=1e-13)


def test_block_with_adapters_is_block_with_merged_weights():
    c = _tiny_case(12)
    g = np.random.default_rng(3)
    W = _fused(c)
    rank = 4
    ad = [(0.3 * g.standard_normal((rank, w.shape[1])), 0.3 * g.standard_normal((w.shape[0], rank))) for w in W]
    merged = tuple(O.lora_merge(w, a, b) for w, (a, b) in zip(W, ad))
    y_lora = O.block_forward_rows(c["x"], merged, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    y_plain = O.block_forward_rows(c["x"], W, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"], c["d"])
    assert not np.allclose(y_lora, y_plain)
    # the same block with the adapters applied beside each linear, written out step by step
    x = c["x"]
    R, H = x.shape
    nh, d = c["heads"], c["d"]
    m = c["mod"][c["mod_map"]]
    h = O.modulated_rmsnorm(x, None, m[:, 0], m[:, 1], 1e-6)
    qkv = O.lora_linear(h, W[0], *ad[0])
    q = O.rotate(O.qk_rmsnorm(qkv[:, :H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    k = O.rotate(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    o = O.attention(q, k, qkv[:, 2 * H:].reshape(R, nh, d))
    x1 = x + m[:, 2] * O.lora_linear(o, W[1], *ad[1])
    h2 = O.modulated_rmsnorm(x1, None, m[:, 3], m[:, 4], 1e-6)
    a = O.swiglu_interleaved(O.lora_linear(h2, W[2], *ad[2]))
    y = x1 + m[:, 5] * O.lora_linear(a, W[3], *ad[3])
    np.testing.assert_allclose(y_lora, y, rtol=1e-12, atol=1e-12)


def test_parallel_block_with_adapters_is_the_block_with_merged_weights():
    # the parallel block's four linears with adapters beside them, written out step by step, equals
    # the parallel block on W + B A [gizai:dit, Block.parallel; withLora, loraOf, weightAt]
    from tests.test_oracle_parallel import _case
    c = _case(13)
    g = np.random.default_rng(5)
    W = _fused(c)
    ad = [(0.3 * g.standard_normal((3, w.shape[1])), 0.3 * g.standard_normal((w.shape[0], 3))) for w in W]
    merged = tuple(O.lora_merge(w, a, b) for w, (a, b) in zip(W, ad))
    y_merged = O.parallel_block_forward_rows(c["x"], merged, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                             c["d"])
    x = c["x"]
    R, H = x.shape
    nh, d = c["heads"], c["d"]
    m = c["mod"][c["mod_map"]]
    h = O.modulated_layernorm(x, None, m[:, 0], m[:, 1], 1e-6)
    qkv = O.lora_linear(h, W[0], *ad[0])
    q = O.rotate(O.qk_rmsnorm(qkv[:, :H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    k = O.rotate(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(R, nh, d), None, 1e-6), c["cos"], c["sin"])
    o = O.attention(q, k, qkv[:, 2 * H:].reshape(R, nh, d))
    a = O.swiglu_interleaved(O.lora_linear(h, W[2], *ad[2]))
    y = x + m[:, 2] * (O.lora_linear(o, W[1], *ad[1]) + O.lora_linear(a, W[3], *ad[3]))
    np.testing.assert_allclose(y_merged, y, rtol=1e-12, atol=1e-12)
    assert not np.allclose(y_merged, O.parallel_block_forward_rows(c["x"], W, c["mod"], c["mod_map"], c["cos"],
                                                                   c["sin"], c["heads"], c["d"]))


def test_double_block_with_per_stream_adapters_is_the_block_with_merged_weights():
    # each stream's linears with that stream's adapters = the double block on each stream's W + B A
    from tests.test_oracle_double import _stream
    c = _tiny_case(14, L=2)
    g = np.random.default_rng(6)
    H, F = c["x"].shape[1], c["Wg"].shape[0]
    Wt, Wi = _fused(_stream(g, H, F)), _fused(_stream(g, H, F))
    adt = [(0.3 * g.standard_normal((2, w.shape[1])), 0.3 * g.standard_normal((w.shape[0], 2))) for w in Wt]
    adi = [(0.3 * g.standard_normal((2, w.shape[1])), 0.3 * g.standard_normal((w.shape[0], 2))) for w in Wi]
    mt = tuple(O.lora_merge(w, a, b) for w, (a, b) in zip(Wt, adt))
    mi = tuple(O.lora_merge(w, a, b) for w, (a, b) in zip(Wi, adi))
    y_merged = O.double_block_forward_rows(c["x"], mt, mi, c["mod"], c["mod_map"], c["cos"], c["sin"], c["heads"],
                                           c["d"], 2)
    x = c["x"]
    R, H = x.shape
    nh, d = c["heads"], c["d"]
    m = c["mod"][c["mod_map"]]
    q, k, v = np.empty((R, nh, d)), np.empty((R, nh, d)), np.empty((R, nh, d))
    streams = ((np.arange(0, 2), Wt, adt), (np.arange(2, R), Wi, adi))
    for idx, W, ad in streams:
        h = O.modulated_rmsnorm(x[idx], None, m[idx, 0], m[idx, 1], 1e-6)
        qkv = O.lora_linear(h, W[0], *ad[0])
        q[idx] = O.rotate(O.qk_rmsnorm(qkv[:, :H].reshape(-1, nh, d), None, 1e-6), c["cos"][idx], c["sin"][idx])
        k[idx] = O.rotate(O.qk_rmsnorm(qkv[:, H:2 * H].reshape(-1, nh, d), None, 1e-6), c["cos"][idx], c["sin"][idx])
        v[idx] = qkv[:, 2 * H:].reshape(-1, nh, d)
    o = O.attention(q, k, v)
    y = np.empty_like(x)
    for idx, W, ad in streams:
        x1 = x[idx] + m[idx, 2] * O.lora_linear(o[idx], W[1], *ad[1])
        h2 = O.modulated_rmsnorm(x1, None, m[idx, 3], m[idx, 4], 1e-6)
        a = O.swiglu_interleaved(O.lora_linear(h2, W[2], *ad[2]))
        y[idx] = x1 + m[idx, 5] * O.lora_linear(a, W[3], *ad[3])
    np.testing.assert_allclose(y_merged, y, rtol=1e-12, atol=1e-12)
