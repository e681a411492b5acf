"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (decay on the value
columns instead of the key rows, reading the state before the write, a dropped
or misplaced beta, a wrong sign in the residual, a transposed state, a lost
scale, state leaking between packed sequences, an ignored initial state) makes
at least one of them fail.  Shapes use d_k != d_v wherever a transposition
could otherwise go unnoticed.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _unit_rows(rng, *shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_problem(rng, T, H, dk, dv, decay=0.05):
    q = _unit_rows(rng, T, H, dk)
    k = _unit_rows(rng, T, H, dk)
    v = rng.standard_normal((T, H, dv))
    la = -decay * np.log1p(np.exp(rng.standard_normal((T, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, la, beta


# ---------------------------------------------------------------- worked example
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


def test_hand_worked_example():
    """Two tokens, d_k = d_v = 2, worked by hand in the fixture from the update
    rule of "Day 19, linear attention & KDA", section 3."""
    g = _read_golden("hand_worked_dk2_dv2_T2.txt")
    q = g["q"].reshape(2, 1, 2)
    k = g["k"].reshape(2, 1, 2)
    v = g["v"].reshape(2, 1, 2)
    la = np.log(g["alpha"]).reshape(2, 1, 2)
    beta = g["beta"].reshape(2, 1)
    o, fs, _ = oracle.prefill(q, k, v, la, beta)
    np.testing.assert_allclose(o.reshape(-1) * math.sqrt(2.0), g["o_times_sqrt2"], atol=1e-14)
    np.testing.assert_allclose(fs.reshape(-1), g["final_state"], atol=1e-14)


# ---------------------------------------------------------------- exact rationals
def _fraction_recurrence(q, k, v, alpha, beta):
    """Product form (I - beta k k^T) Diag(alpha) S + beta k v^T ("K3 attention,
    three-piece set", KDA paragraph on the (I - beta k k^T) factor), in exact
    rational arithmetic.  Returns S_t^T q_t (unscaled) per token and the final S."""
    T, dk = len(k), len(k[0])
    dv = len(v[0])
    S = [[Fraction(0)] * dv for _ in range(dk)]
    outs = []
    for t in range(T):
        D = [[alpha[t][i] * S[i][j] for j in range(dv)] for i in range(dk)]
        P = [[(Fraction(1) if i == a else Fraction(0)) - beta[t] * k[t][i] * k[t][a]
              for a in range(dk)] for i in range(dk)]
        S = [[sum(P[i][a] * D[a][j] for a in range(dk)) + beta[t] * k[t][i] * v[t][j]
              for j in range(dv)] for i in range(dk)]
        outs.append([sum(S[i][j] * q[t][i] for i in range(dk)) for j in range(dv)])
    return outs, S


def test_brute_force_exact_rationals():
    """Tiny problem with rational alpha, beta, k, v, q (k not normalised, d_k != d_v)
    evaluated exactly; the oracle must agree to double rounding."""
    rng = np.random.default_rng(7)
    T, dk, dv = 5, 3, 2
    fr = lambda a, b: Fraction(int(a), int(b))
    alpha = [[fr(rng.integers(1, 8), 8) for _ in range(dk)] for _ in range(T)]
    beta = [fr(rng.integers(0, 5), 4) for _ in range(T)]
    k = [[fr(rng.integers(-4, 5), 4) for _ in range(dk)] for _ in range(T)]
    v = [[fr(rng.integers(-6, 7), 3) for _ in range(dv)] for _ in range(T)]
    q = [[fr(rng.integers(-4, 5), 2) for _ in range(dk)] for _ in range(T)]
    outs, S = _fraction_recurrence(q, k, v, alpha, beta)
    f = lambda m: np.array([[float(x) for x in row] for row in m])
    o, fs, _ = oracle.prefill(f(q)[:, None], f(k)[:, None], f(v)[:, None],
                              np.log(f(alpha))[:, None], f([[b] for b in beta]), )
    np.testing.assert_allclose(o[:, 0] * math.sqrt(dk), f(outs), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fs[0, 0], f(S), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- closed forms
def test_beta_zero_is_pure_decay():
    """beta = 0 writes nothing: S_T = Diag(prod alpha) S_0, and each output reads the
    decayed initial state.  Decay must act on key rows (index i of S)."""
    rng = np.random.default_rng(1)
    T, H, dk, dv = 9, 2, 5, 3
    q, k, v, la, _ = _rand_problem(rng, T, H, dk, dv, decay=0.3)
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    o, fs, _ = oracle.prefill(q, k, v, la, beta, init_state=S0)
    g = np.cumsum(la, axis=0)  # [T, H, dk]
    for h in range(H):
        np.testing.assert_allclose(fs[0, h], np.exp(g[-1, h])[:, None] * S0[0, h], rtol=1e-13)
        for t in range(T):
            St = np.exp(g[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h] / math.sqrt(dk), rtol=1e-12,
                                       atol=1e-15)


def test_exact_retrieval_any_alpha_any_state():
    """beta = 1 and |k| = 1: the write cancels the prediction, so S_t^T k_t = v_t for any
    decay and any prior state.  Querying with q_t = k_t therefore returns v_t/sqrt(d_k):
    this fails if the read happened before the write, if the decay came after the
    write, or if the residual had the wrong sign."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 12, 3, 6, 4
    _, k, v, la, _ = _rand_problem(rng, T, H, dk, dv, decay=0.5)
    S0 = rng.standard_normal((1, H, dk, dv))
    o, _, _ = oracle.prefill(k.copy(), k, v, la, np.ones((T, H)), init_state=S0)
    np.testing.assert_allclose(o * math.sqrt(dk), v, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_store_exactly():
    """alpha = 1, beta = 1, S_0 = 0, orthonormal keys: S_m = sum_s k_s v_s^T (the
    linear-attention state of "Day 19", quiz Q2), and q = k_s reads back v_s."""
    rng = np.random.default_rng(3)
    dk, dv, m = 8, 5, 6
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Q[:, :m].T.copy()[:, None, :]  # [m, 1, dk]
    v = rng.standard_normal((m, 1, dv))
    zeros = np.zeros((m, 1, dk))
    _, fs, _ = oracle.prefill(k, k, v, zeros, np.ones((m, 1)))
    np.testing.assert_allclose(fs[0, 0], sum(np.outer(k[s, 0], v[s, 0]) for s in range(m)),
                               atol=1e-13)
    state = fs.copy()
    for s in range(m):  # read with a decode step that writes nothing (beta = 0)
        st = state.copy()
        o, _ = oracle.decode_step(k[s][None], k[s][None], v[s][None], zeros[s][None],
                                  np.zeros((1, 1)), st)
        np.testing.assert_allclose(o[0, 0] * math.sqrt(dk), v[s, 0], atol=1e-12)


def test_same_key_overwrites():
    """Delta rule overwrites instead of accumulating ("From 124M to 2.8T", chapter 3):
    writing v1 then v2 under the same key with beta = 1 leaves v2 retrievable and no
    trace of v1 along that key."""
    dk, dv = 4, 3
    k = np.array([0.5, 0.5, 0.5, 0.5])
    ks = np.stack([k, k])[:, None]
    vs = np.array([[1.0, 2.0, 3.0], [-4.0, 0.5, 7.0]])[:, None]
    _, fs, _ = oracle.prefill(ks, ks, vs, np.zeros((2, 1, dk)), np.ones((2, 1)))
    np.testing.assert_allclose(fs[0, 0].T @ k, vs[1, 0], atol=1e-14)
    np.testing.assert_allclose(fs[0, 0], np.outer(k, vs[1, 0]), atol=1e-14)


@pytest.mark.parametrize("b", [0.25, 0.5, 0.9])
def test_repeated_write_converges_geometrically(b):
    """alpha = 1, the same unit key and value written m times with strength b from a zero
    state: the prediction along k after m writes is (1 - (1-b)^m) v.  A beta applied to
    v but not to the prediction would give a different sequence."""
    dk, dv, m = 3, 2, 7
    k = np.array([2.0, -1.0, 2.0]) / 3.0
    v = np.array([1.5, -2.0])
    ks = np.tile(k, (m, 1))[:, None]
    vs = np.tile(v, (m, 1))[:, None]
    o, _, _ = oracle.prefill(ks, ks, vs, np.zeros((m, 1, dk)), np.full((m, 1), b))
    for t in range(m):
        np.testing.assert_allclose(o[t, 0] * math.sqrt(dk), (1 - (1 - b) ** (t + 1)) * v,
                                   rtol=1e-13)


def test_alpha_one_matches_deltanet_code():
    """With alpha = 1 KDA is DeltaNet.  "From 124M to 2.8T", chapter 3, gives DeltaNet in
    row-vector form: v_old = k @ S; u = beta (v - v_old); S = S + k^T u; o = q @ S.
    Written here per token with numpy (output scale 1/sqrt(d_k) added)."""
    rng = np.random.default_rng(4)
    T, dk, dv = 20, 6, 4
    q, k, v, _, beta = _rand_problem(rng, T, 1, dk, dv)
    S = np.zeros((dk, dv))
    o_ref = np.zeros((T, dv))
    for t in range(T):
        kt = k[t, 0][None, :]
        u = beta[t, 0] * (v[t, 0][None, :] - kt @ S)
        S = S + kt.T @ u
        o_ref[t] = (q[t, 0][None, :] @ S)[0] / math.sqrt(dk)
    o, fs, _ = oracle.prefill(q, k, v, np.zeros((T, 1, dk)), beta)
    np.testing.assert_allclose(o[:, 0], o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fs[0, 0], S, rtol=1e-12, atol=1e-14)


def test_scalar_alpha_is_gated_deltanet_decay_first():
    """alpha_i = a_t for every channel: KDA reduces to the scalar-gate delta rule with the
    decay applied before the prediction, S_t = a_t (I - beta k k^T) S_{t-1} + beta k v^T."""
    rng = np.random.default_rng(5)
    T, dk, dv = 25, 5, 7
    q, k, v, _, beta = _rand_problem(rng, T, 1, dk, dv)
    a = np.exp(-0.3 * rng.random(T))
    S = rng.standard_normal((dk, dv))
    S0 = S.copy()
    o_ref = np.zeros((T, dv))
    for t in range(T):
        kt = k[t, 0]
        S = a[t] * (np.eye(dk) - beta[t, 0] * np.outer(kt, kt)) @ S + beta[t, 0] * np.outer(kt, v[t, 0])
        o_ref[t] = S.T @ q[t, 0] / math.sqrt(dk)
    la = np.repeat(np.log(a)[:, None, None], dk, axis=2)
    o, fs, _ = oracle.prefill(q, k, v, la, beta, init_state=S0[None, None])
    np.testing.assert_allclose(o[:, 0], o_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(fs[0, 0], S, rtol=1e-11, atol=1e-13)


def test_gdn_page_code_order_differs():
    """"From 124M to 2.8T", chapter 3, writes Gated DeltaNet with the prediction taken on
    the UNdecayed state (v_old = k @ S, then S = alpha*S + k^T u).  That is a different
    recurrence from the decay-first order of the KDA update, and the oracle must NOT
    match it whenever decay and writes interact.  This records the discrepancy instead
    of adopting the page's order silently."""
    rng = np.random.default_rng(6)
    T, dk, dv = 10, 4, 3
    q, k, v, _, beta = _rand_problem(rng, T, 1, dk, dv)
    a = np.full(T, 0.5)
    S = np.zeros((dk, dv))
    for t in range(T):
        kt = k[t, 0][None, :]
        u = beta[t, 0] * (v[t, 0][None, :] - kt @ S)
        S = a[t] * S + kt.T @ u
    la = np.full((T, 1, dk), math.log(0.5))
    _, fs, _ = oracle.prefill(q, k, v, la, beta)
    assert np.linalg.norm(fs[0, 0] - S) > 1e-3 * np.linalg.norm(S)


def test_linear_in_initial_state_and_values():
    rng = np.random.default_rng(8)
    T, H, dk, dv = 30, 2, 6, 5
    q, k, v1, la, beta = _rand_problem(rng, T, H, dk, dv, decay=0.2)
    v2 = rng.standard_normal(v1.shape)
    S1 = rng.standard_normal((1, H, dk, dv))
    S2 = rng.standard_normal((1, H, dk, dv))
    a, b = 0.7, -1.3
    o1, f1, _ = oracle.prefill(q, k, v1, la, beta, init_state=S1)
    o2, f2, _ = oracle.prefill(q, k, v2, la, beta, init_state=S2)
    o3, f3, _ = oracle.prefill(q, k, a * v1 + b * v2, la, beta, init_state=a * S1 + b * S2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(f3, a * f1 + b * f2, atol=1e-12)


def test_value_columns_are_independent():
    """Permuting the value channels of V and S_0 permutes those of o and S_T."""
    rng = np.random.default_rng(9)
    T, H, dk, dv = 17, 2, 4, 6
    q, k, v, la, beta = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    perm = rng.permutation(dv)
    o, fs, _ = oracle.prefill(q, k, v, la, beta, init_state=S0)
    op, fsp, _ = oracle.prefill(q, k, v[:, :, perm], la, beta, init_state=S0[..., perm])
    np.testing.assert_allclose(op, o[:, :, perm], atol=1e-14)
    np.testing.assert_allclose(fsp, fs[..., perm], atol=1e-14)


def test_state_norm_bound():
    """|beta| <= 1, alpha <= 1, |k| = 1: (I - beta k k^T) Diag(alpha) has spectral norm
    <= 1, so |S_t|_2 <= |S_{t-1}|_2 + beta |v_t| at every token."""
    rng = np.random.default_rng(10)
    T, dk, dv = 40, 6, 6
    q, k, v, la, beta = _rand_problem(rng, T, 1, dk, dv, decay=0.1)
    state = rng.standard_normal((1, 1, dk, dv))
    for t in range(T):
        prev = np.linalg.norm(state[0, 0], 2)
        oracle.decode_step(q[t][None], k[t][None], v[t][None], la[t][None], beta[t][None],
                           state)
        assert np.linalg.norm(state[0, 0], 2) <= prev + beta[t, 0] * np.linalg.norm(v[t, 0]) + 1e-12


# ---------------------------------------------------------------- composition
def test_packed_sequences_equal_separate_calls_and_empty_sequence():
    rng = np.random.default_rng(11)
    lens = [7, 0, 13, 1]
    T, H, dk, dv = sum(lens), 2, 5, 3
    q, k, v, la, beta = _rand_problem(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, fs, _ = oracle.prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        on, fn, _ = oracle.prefill(q[t0:t1], k[t0:t1], v[t0:t1], la[t0:t1], beta[t0:t1],
                                   init_state=S0[n:n + 1])
        np.testing.assert_array_equal(o[t0:t1], on)
        np.testing.assert_array_equal(fs[n], fn[0])
    np.testing.assert_array_equal(fs[1], S0[1])  # zero-length sequence keeps its state


def test_split_prefill_and_decode_continue_the_recurrence():
    rng = np.random.default_rng(12)
    T, H, dk, dv = 24, 2, 4, 5
    q, k, v, la, beta = _rand_problem(rng, T, H, dk, dv)
    o, fs, _ = oracle.prefill(q, k, v, la, beta)
    o1, f1, _ = oracle.prefill(q[:10], k[:10], v[:10], la[:10], beta[:10])
    o2, f2, _ = oracle.prefill(q[10:20], k[10:20], v[10:20], la[10:20], beta[10:20],
                               init_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o[:20], atol=1e-13)
    state = f2.copy()
    for t in range(20, T):
        od, _ = oracle.decode_step(q[t][None], k[t][None], v[t][None], la[t][None],
                                   beta[t][None], state)
        np.testing.assert_allclose(od[0], o[t], atol=1e-13)
    np.testing.assert_allclose(state, fs, atol=1e-13)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(13)
    q, k, v, la, beta = _rand_problem(rng, 50, 8, 6, 6)
    o1, f1, n1 = oracle.prefill(q, k, v, la, beta, nthreads=1)
    o4, f4, n4 = oracle.prefill(q, k, v, la, beta, nthreads=4)
    assert n1 == 1 and n4 == 4
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(f1, f4)


# ---------------------------------------------------------------- q / k L2 normalisation
def test_l2_normalize_worked_rows_and_the_floor():
    """Rows over the last axis: (3, 4) -> (0.6, 0.8) (a 3-4-5 triangle), a zero row stays
    zero, and a row shorter than the floor is divided by the floor, not by its norm."""
    x = np.array([[[3.0, 4.0, 0.0], [0.0, 0.0, 0.0]], [[1e-13, 0.0, 0.0], [0.0, -2.0, 0.0]]])
    y = oracle.l2_normalize(x)
    assert y.shape == x.shape
    np.testing.assert_allclose(y[0, 0], [0.6, 0.8, 0.0], rtol=0, atol=1e-15)
    assert np.all(y[0, 1] == 0.0)
    np.testing.assert_allclose(y[1, 0], [0.1, 0.0, 0.0], rtol=1e-12)
    np.testing.assert_array_equal(y[1, 1], [0.0, -1.0, 0.0])


def test_l2_normalize_gives_unit_rows_in_the_same_direction():
    """Every row of a [T, H, d] array comes out with norm 1 and the same direction (its
    cosine with the input row is 1); scaling a row by c > 0 changes nothing."""
    rng = np.random.default_rng(7)
    x = 3.0 * rng.standard_normal((5, 3, 16))
    y = oracle.l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    cos = np.sum(x * y, axis=-1) / np.linalg.norm(x, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.l2_normalize(x * 17.5), y, rtol=1e-14, atol=1e-16)
