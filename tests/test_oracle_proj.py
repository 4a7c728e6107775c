"""Pins of the oracle's dense projections and of its bf16 rounding.

The layer's inputs q|k|v, z, a, b come out of an input projection of the
hidden state and its output goes through an output projection (the hybrid
models of "Serving large language models on our own stack", section
"Qwen3.5-35B-A3B from a real GGUF").  Each pin checks a value the mathematics
fixes independently of the oracle's code: an identity weight, one-hot rows,
a product worked by hand, the nearest-even rule on constructed ties, and the
column order of the split into the layer's buffers.
"""
import numpy as np
import pytest
import torch

import oracle


def test_linear_identity_weight_returns_input():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 7))
    assert np.array_equal(oracle.linear(x, np.eye(7)), x)


def test_linear_one_hot_rows_pick_input_columns():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 6))
    pick = [3, 0, 5, 5, 1, 2, 4, 0, 3]          # output feature n reads input feature pick[n]
    w = np.zeros((len(pick), 6))
    w[np.arange(len(pick)), pick] = 1.0
    y = oracle.linear(x, w)
    assert y.shape == (4, len(pick))
    for n, f in enumerate(pick):
        assert np.array_equal(y[:, n], x[:, f])


def test_linear_hand_computed_2x3():
    # x [2][2], w [3][2] (output by input): y[m][n] = sum_k x[m][k] w[n][k]
    x = np.array([[1.0, 2.0], [3.0, 4.0]])
    w = np.array([[2.0, -1.0], [0.0, 3.0], [1.0, 1.0]])
    #   row 0: (1*2 + 2*-1, 1*0 + 2*3, 1*1 + 2*1) = (0, 6, 3)
    #   row 1: (3*2 + 4*-1, 3*0 + 4*3, 3*1 + 4*1) = (2, 12, 7)
    assert np.array_equal(oracle.linear(x, w), np.array([[0.0, 6.0, 3.0], [2.0, 12.0, 7.0]]))


def test_linear_is_linear_in_both_operands():
    rng = np.random.default_rng(2)
    x1, x2 = rng.standard_normal((3, 9)), rng.standard_normal((3, 9))
    w1, w2 = rng.standard_normal((4, 9)), rng.standard_normal((4, 9))
    np.testing.assert_allclose(oracle.linear(x1 + x2, w1), oracle.linear(x1, w1) + oracle.linear(x2, w1),
                               atol=1e-12)
    np.testing.assert_allclose(oracle.linear(x1, w1 - w2), oracle.linear(x1, w1) - oracle.linear(x1, w2),
                               atol=1e-12)


def test_round_bf16_nearest_even_on_constructed_ties():
    u = 2.0 ** -7                                  # bf16 spacing in [1, 2)
    cases = {
        1.0: 1.0,
        1.0 + u / 2: 1.0,                          # tie, 1.0 is even
        1.0 + 3 * u / 2: 1.0 + 2 * u,              # tie, 1 + 2u is even
        1.0 + u / 2 + 2.0 ** -20: 1.0 + u,         # just above the tie
        1.0 + u / 2 - 2.0 ** -20: 1.0,             # just below
        -(1.0 + 3 * u / 2): -(1.0 + 2 * u),        # sign symmetric
        0.0: 0.0,
        2.0 ** -100 * (1 + u / 2): 2.0 ** -100,    # the rule holds at any exponent
        3.0 * 2.0 ** 60: 3.0 * 2.0 ** 60,          # exactly representable
        255.5: 256.0,                              # 8 significant bits: 255.5 -> tie -> 256 (even)
        254.5: 254.0,
    }
    got = oracle.round_bf16(np.array(list(cases)))
    assert np.array_equal(got, np.array(list(cases.values())))


def test_round_bf16_agrees_with_float32_to_bfloat16_conversion():
    # for values that are already fp32 the rounding is torch's fp32 -> bf16
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), want)


def test_in_proj_splits_columns_in_the_documented_order():
    # hidden = 1: w_in's row n is the number n + 1, so output feature n of a
    # token with x = 1 is n + 1 -- the split must hand feature n to the
    # documented place: Cc conv channels, then z head-major, then a, then b
    h_k, h_v, d_k, d_v = 1, 2, 4, 3
    Cc, Cv = 2 * h_k * d_k + h_v * d_v, h_v * d_v
    N = Cc + Cv + 2 * h_v
    w = (np.arange(N, dtype=np.float64) + 1.0).reshape(N, 1)
    qkv, z, a, b = oracle.in_proj(np.ones((2, 1)), w, h_k=h_k, h_v=h_v, d_k=d_k, d_v=d_v)
    assert qkv.shape == (2, Cc) and z.shape == (2, h_v, d_v) and a.shape == (2, h_v) and b.shape == (2, h_v)
    assert np.array_equal(qkv[1], np.arange(Cc) + 1.0)
    assert np.array_equal(z[1], (Cc + np.arange(Cv) + 1.0).reshape(h_v, d_v))
    assert np.array_equal(a[1], Cc + Cv + np.arange(h_v) + 1.0)
    assert np.array_equal(b[1], Cc + Cv + h_v + np.arange(h_v) + 1.0)


def test_in_proj_rounds_to_bf16():
    x = np.array([[1.0, 2.0 ** -8]])                 # 1 + 2^-8 is a tie between 1 and 1 + 2^-7
    w = np.ones((2 * 4 + 4 + 4 + 2, 2))              # h_k = h_v = 1, d = 4 (Cc 12, z 4, a 1, b 1): each feature is 1 + 2^-8
    qkv, z, a, b = oracle.in_proj(x, w, h_k=1, h_v=1, d_k=4, d_v=4)
    for t in (qkv, z, a, b):
        assert np.all(t == 1.0)


def test_out_proj_reads_heads_in_row_major_order():
    T, h_v, d_v = 3, 2, 4
    o = np.arange(T * h_v * d_v, dtype=np.float64).reshape(T, h_v, d_v)
    w = np.zeros((2, h_v * d_v))
    w[0, 1 * d_v + 2] = 1.0                          # output 0 reads head 1, component 2
    w[1, 0 * d_v + 3] = -2.0                         # output 1 reads head 0, component 3, times -2
    y = oracle.out_proj(o, w)
    assert np.array_equal(y[:, 0], o[:, 1, 2])
    assert np.array_equal(y[:, 1], -2.0 * o[:, 0, 3])


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 2), (7, 2, 9)])
def test_linear_matches_sum_of_rank_one_terms(shape):
    # a second formulation: x w^T = sum_k (column k of x)(column k of w)^T
    M, N, K = shape
    rng = np.random.default_rng(4)
    x, w = rng.standard_normal((M, K)), rng.standard_normal((N, K))
    ref = sum(np.outer(x[:, k], w[:, k]) for k in range(K))
    np.testing.assert_allclose(oracle.linear(x, w), ref, atol=1e-12)
