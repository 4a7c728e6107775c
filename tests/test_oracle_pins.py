"""Pins of the fp64 oracle against closed forms, invariants and brute force.

None of these re-types the oracle's formulas: each checks a value the
mathematics fixes independently (a special case with a known answer, an
identity, a second formulation of the same recurrence, a hand-expanded step
with the numbers written out).  The source pages print no worked example of
the layer, so there is no page value to pin against.
"""
import math

import numpy as np
import pytest

import oracle

TOL = 1e-12


# ---- scalar pieces ------------------------------------------------------------

def test_softplus_closed_forms():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    for x in (-30.0, -3.0, -0.1, 0.7, 5.0, 40.0):
        # softplus(x) - softplus(-x) = x for every x
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, abs=1e-13)
    # far tails: softplus(x) -> x, softplus(-x) -> e^{-x}
    assert oracle.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    # softplus(ln 3) = ln 4
    assert oracle.softplus(math.log(3.0)) == pytest.approx(math.log(4.0), abs=1e-15)


def test_sigmoid_and_silu_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(math.log(3.0)) == pytest.approx(0.75, abs=1e-15)
    for x in (-7.0, -1.3, 0.2, 4.4):
        assert oracle.sigmoid(x) + oracle.sigmoid(-x) == pytest.approx(1.0, abs=1e-15)
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-14)
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), abs=1e-15)


def test_gates_closed_forms():
    # A_log = 0 and a + dt_bias = 0: g = -softplus(0) = -ln 2, so exp(g) = 1/2
    g, beta = oracle.gates(0.0, 0.0, 0.0, 0.0)
    assert g == pytest.approx(-math.log(2.0), abs=1e-15)
    assert math.exp(g) == pytest.approx(0.5, abs=1e-15)
    assert beta == 0.5
    # A_log = ln 2 doubles the log-decay: exp(g) = 1/4
    g, _ = oracle.gates(0.0, 0.0, math.log(2.0), 0.0)
    assert math.exp(g) == pytest.approx(0.25, abs=1e-15)
    # dt_bias shifts a: (a=1, dt=-1) equals (a=0, dt=0); a = ln 3 gives g = -ln 4
    assert oracle.gates(1.0, 0.0, 0.0, -1.0)[0] == pytest.approx(-math.log(2.0), abs=1e-15)
    assert oracle.gates(0.5, 0.0, 0.0, math.log(3.0) - 0.5)[0] == pytest.approx(
        -math.log(4.0), abs=1e-15)
    # b = ln 3 gives beta = 3/4; the decay is always <= 0 and falls with a
    assert oracle.gates(0.0, math.log(3.0), 0.0, 0.0)[1] == pytest.approx(0.75, abs=1e-15)
    gs = [oracle.gates(a, 0.0, 0.3, 0.0)[0] for a in (-5.0, -1.0, 0.0, 2.0, 9.0)]
    assert all(x < 0 for x in gs) and all(x > y for x, y in zip(gs, gs[1:]))


# ---- conv ------------------------------------------------------------------------

def _rng(seed=0):
    return np.random.default_rng(seed)


def test_conv_identity_tap_gives_silu():
    r = _rng(1)
    x = r.standard_normal((9, 5))
    state = r.standard_normal((3, 5))
    w = np.tile([0.0, 0.0, 0.0, 1.0], (5, 1))
    y, st = oracle.conv_silu(x, w, state)
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(st, x[-3:])


def test_conv_oldest_tap_reads_state_rows_in_order():
    # w = [1, 0, 0, 0] picks x_{t-3}: tokens 0, 1, 2 must see state rows 0, 1, 2
    r = _rng(2)
    x = r.standard_normal((6, 4))
    state = r.standard_normal((3, 4))
    w = np.tile([1.0, 0.0, 0.0, 0.0], (4, 1))
    y, _ = oracle.conv_silu(x, w, state)
    src = np.concatenate([state, x[:3]])
    np.testing.assert_allclose(y, src / (1 + np.exp(-src)), rtol=0, atol=1e-15)


def test_conv_box_filter_is_moving_sum():
    r = _rng(3)
    x = r.standard_normal((7, 3))
    state = r.standard_normal((3, 3))
    w = np.ones((3, 4))
    y, _ = oracle.conv_silu(x, w, state)
    full = np.concatenate([state, x])
    for t in range(7):
        s = full[t:t + 4].sum(axis=0)      # x_{t-3} .. x_t
        np.testing.assert_allclose(y[t], s / (1 + np.exp(-s)), rtol=0, atol=1e-14)


def test_conv_state_carry_identity():
    # conv over (prefix || x) equals conv over x started from the prefix's
    # last three rows, and the carried rows are the last three raw inputs
    r = _rng(4)
    pre = r.standard_normal((5, 6))
    x = r.standard_normal((4, 6))
    w = r.standard_normal((6, 4))
    y_all, st_all = oracle.conv_silu(np.concatenate([pre, x]), w, None)
    _, st_pre = oracle.conv_silu(pre, w, None)
    y_tail, st_tail = oracle.conv_silu(x, w, st_pre)
    np.testing.assert_allclose(y_tail, y_all[5:], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(st_tail, st_all)
    np.testing.assert_array_equal(st_pre, pre[-3:])


@pytest.mark.parametrize("T", [0, 1, 2])
def test_conv_short_sequence_mixes_state(T):
    r = _rng(5 + T)
    x = r.standard_normal((T, 3))
    state = r.standard_normal((3, 3))
    _, st = oracle.conv_silu(x, np.ones((3, 4)), state)
    np.testing.assert_array_equal(st, np.concatenate([state, x])[-3:])


# ---- norms -----------------------------------------------------------------------

def test_l2norm_closed_form():
    out = oracle.l2norm(np.array([3.0, 4.0]), 0.0, 1.0)
    np.testing.assert_allclose(out, [0.6, 0.8], rtol=0, atol=1e-15)
    out = oracle.l2norm(np.array([3.0, 4.0]), 0.0, 1.0 / math.sqrt(2.0))
    np.testing.assert_allclose(out, [0.6 / math.sqrt(2), 0.8 / math.sqrt(2)], atol=1e-15)
    v = _rng(6).standard_normal(128)
    n = oracle.l2norm(v, 1e-6, 1.0)
    ss = float(v @ v)
    assert float(n @ n) == pytest.approx(ss / (ss + 1e-6), abs=1e-14)
    np.testing.assert_array_equal(oracle.l2norm(np.zeros(8), 1e-6, 1.0), np.zeros(8))


def test_gated_rmsnorm_closed_forms():
    # o = (1, -1): mean(o^2) = 1, so with eps = 0 the norm leaves o unchanged;
    # z = ln 3 on both gives silu = 0.75 ln 3; w = (2, 1/2)
    out = oracle.gated_rmsnorm(np.array([1.0, -1.0]), np.array([math.log(3)] * 2),
                               np.array([2.0, 0.5]), 0.0)
    s = 0.75 * math.log(3.0)
    np.testing.assert_allclose(out, [2.0 * s, -0.5 * s], rtol=0, atol=1e-15)
    r = _rng(7)
    o, z, w = r.standard_normal(16), r.standard_normal(16), r.standard_normal(16)
    np.testing.assert_array_equal(oracle.gated_rmsnorm(o, np.zeros(16), w, 1e-6), 0.0)
    # scale invariance in o (eps = 0)
    np.testing.assert_allclose(oracle.gated_rmsnorm(3.7 * o, z, w, 0.0),
                               oracle.gated_rmsnorm(o, z, w, 0.0), rtol=0, atol=1e-14)
    # normalise first, then gate: the gate does not enter the mean
    base = oracle.gated_rmsnorm(o, np.full(16, 30.0), np.ones(16), 0.0)
    np.testing.assert_allclose(base, o / math.sqrt(np.mean(o * o)) * 30.0, atol=1e-12)


# ---- the recurrence --------------------------------------------------------------

def _unit_rows(r, T, d):
    x = r.standard_normal((T, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _case(seed, T, d_k, d_v, slow=False):
    r = _rng(seed)
    q = _unit_rows(r, T, d_k) / math.sqrt(d_k)
    k = _unit_rows(r, T, d_k)
    v = r.standard_normal((T, d_v))
    if slow:
        g = np.log(r.uniform(0.9, 1.0, T))
        beta = r.uniform(0.0, 0.3, T)
    else:
        g = -np.exp(r.uniform(0, math.log(16), T)) * np.log1p(np.exp(r.standard_normal(T)))
        beta = 1 / (1 + np.exp(-r.standard_normal(T)))
    S0 = r.standard_normal((d_v, d_k)) * math.sqrt(0.1)
    return q, k, v, g, beta, S0


def test_hand_expanded_first_step_from_zero():
    # d_k = 2, d_v = 3 (non-square, so a transposed state fails).
    # S0 = 0: S1 = beta v k^T and o1 = beta (k.q) v, whatever g is.
    k = np.array([[0.6, 0.8]])
    q = np.array([[1.0, 0.0]])
    v = np.array([[1.0, 2.0, -4.0]])
    o, S = oracle.recurrence_seq(q, k, v, np.array([-0.7]), np.array([0.5]))
    np.testing.assert_allclose(S, [[0.3, 0.4], [0.6, 0.8], [-1.2, -1.6]], atol=1e-15)
    np.testing.assert_allclose(o, [[0.3, 0.6, -1.2]], atol=1e-15)


def test_hand_expanded_two_steps():
    # S0 = [[1, 0], [0, 1], [2, 2]] (d_v = 3, d_k = 2).
    # step 1: g = ln(1/2), beta = 1, k = (1, 0), v = (3, 5, 7), q = (0, 1)
    #   decayed S = [[.5, 0], [0, .5], [1, 1]];  S k = (.5, 0, 1)
    #   u = v - S k = (2.5, 5, 6);  S1 = S + u k^T = [[3, 0], [5, .5], [7, 1]]
    #   o1 = S1 q = (0, .5, 1)
    # step 2: g = 0, beta = 1/2, k = (0, 1), v = (1, 1, 1), q = (1, 1)
    #   S k = (0, .5, 1);  u = (1/2)(1 - Sk) = (.5, .25, 0)
    #   S2 = [[3, .5], [5, .75], [7, 1]];  o2 = (3.5, 5.75, 8)
    S0 = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 2.0]])
    q = np.array([[0.0, 1.0], [1.0, 1.0]])
    k = np.array([[1.0, 0.0], [0.0, 1.0]])
    v = np.array([[3.0, 5.0, 7.0], [1.0, 1.0, 1.0]])
    g = np.array([math.log(0.5), 0.0])
    beta = np.array([1.0, 0.5])
    for fn in (oracle.recurrence_seq, oracle.recurrence_products,
               lambda *a: oracle.recurrence_chunked(*a, chunk=2)):
        o, S = fn(q, k, v, g, beta, S0)
        np.testing.assert_allclose(o, [[0.0, 0.5, 1.0], [3.5, 5.75, 8.0]], atol=1e-15)
        np.testing.assert_allclose(S, [[3.0, 0.5], [5.0, 0.75], [7.0, 1.0]], atol=1e-15)


@pytest.mark.parametrize("slow", [False, True])
def test_output_from_the_state_before_the_token_equals_the_oracle(slow):
    # The decode kernels take o_t from the state before token t:
    #   u = beta (v - e^g S k),  o = e^g (S q) + u (k . q)
    # which is S' q with S' = e^g S + u k^T, the oracle's order.  Checked on 8
    # tokens, d_k = 6, d_v = 5, against the oracle's outputs and states.
    T = 8
    q, k, v, g, beta, S0 = _case(17, T, 6, 5, slow=slow)
    o_ref, _ = oracle.recurrence_seq(q, k, v, g, beta, S0)
    S = S0.copy()
    for t in range(T):
        d = math.exp(g[t])
        u = beta[t] * (v[t] - d * (S @ k[t]))
        o = d * (S @ q[t]) + u * float(k[t] @ q[t])
        np.testing.assert_allclose(o, o_ref[t], rtol=0, atol=1e-12)
        _, S = oracle.recurrence_seq(q[: t + 1], k[: t + 1], v[: t + 1], g[: t + 1],
                                     beta[: t + 1], S0)


def test_beta0_g0_leaves_state_bitwise():
    q, k, v, _, _, S0 = _case(11, 10, 8, 6)
    o, S = oracle.recurrence_seq(q, k, v, np.zeros(10), np.zeros(10), S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0.T, rtol=0, atol=1e-15)


def test_beta1_overwrites_key_direction():
    # beta = 1 with a unit key: S_t k_t = v_t exactly, and any direction
    # orthogonal to k_t keeps exp(g) S_{t-1}
    r = _rng(12)
    d_k, d_v = 6, 5
    S = r.standard_normal((d_v, d_k))
    for t in range(5):
        k = _unit_rows(r, 1, d_k)
        v = r.standard_normal((1, d_v))
        g = -abs(r.standard_normal())
        x = r.standard_normal(d_k)
        x -= (x @ k[0]) * k[0]                       # x orthogonal to k
        _, S1 = oracle.recurrence_seq(np.zeros((1, d_k)), k, v, np.array([g]),
                                      np.array([1.0]), S)
        np.testing.assert_allclose(S1 @ k[0], v[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(S1 @ x, math.exp(g) * (S @ x), rtol=0, atol=1e-13)
        S = S1


def test_full_decay_resets_state():
    q, k, v, _, beta, S0 = _case(13, 1, 8, 4)
    o, S = oracle.recurrence_seq(q, k, v, np.array([-1e3]), beta, S0)
    np.testing.assert_allclose(S, beta[0] * np.outer(v[0], k[0]), rtol=0, atol=1e-15)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
@pytest.mark.parametrize("slow", [False, True])
def test_products_form_equals_sequential(T, slow):
    q, k, v, g, beta, S0 = _case(20 + T, T, 5, 3, slow)
    o1, S1 = oracle.recurrence_seq(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrence_products(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=TOL)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("slow", [False, True])
def test_chunked_equals_sequential(C, slow):
    T = 150                                       # several chunks and a ragged tail
    q, k, v, g, beta, S0 = _case(30 + C, T, 16, 12, slow)
    o1, S1 = oracle.recurrence_seq(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrence_chunked(q, k, v, g, beta, S0, chunk=C)
    scale = max(1.0, np.abs(o1).max())
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL * scale)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=TOL * max(1.0, np.abs(S1).max()))


def test_chunked_survives_decay_underflow():
    # a 64-token chunk whose cumulative log-decay is about -6000: every
    # exp(gamma_i - gamma_j) must be formed from a difference, never a product
    T = 64
    q, k, v, _, beta, S0 = _case(40, T, 8, 8)
    g = np.full(T, -100.0)
    o1, S1 = oracle.recurrence_seq(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrence_chunked(q, k, v, g, beta, S0, chunk=64)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(S2))
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=TOL)
