"""The chunkwise form the CUDA prefill uses equals the token recurrence.

The pages name the chunkwise method (WY representation + UT transform) but omit
its algebra; ``chunked_reference.py`` derives it.  These tests check it against
the oracle on tiny inputs, with chunk sizes 1 (brute force), 4, 16 and 64,
ragged tails, strong decay and packed sequences, and record the rounding budget
that decides which products may use bf16 operands.
"""
import numpy as np
import pytest

import oracle
from chunked_reference import bf16_round, chunked_prefill, folded_unit, tf32_round


def _problem(seed, lens, H, dk, dv, decay):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q = rng.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    la = -decay * np.log1p(np.exp(rng.standard_normal((T, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.1 * rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    return q, k, v, la, beta, cu, S0


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("decay", [0.05, 1.0])
def test_chunked_equals_recurrence(C, decay):
    q, k, v, la, beta, cu, S0 = _problem(20 + C, [150, 0, 64, 37], 2, 16, 12, decay)
    o_ref, f_ref, _ = oracle.prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0)
    o, f = chunked_prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0, C=C)
    scale_o = np.abs(o_ref).max()
    np.testing.assert_allclose(o, o_ref, atol=1e-12 * max(scale_o, 1.0))
    np.testing.assert_allclose(f, f_ref, atol=1e-12 * max(np.abs(f_ref).max(), 1.0))


def test_chunked_full_head_dimension():
    q, k, v, la, beta, cu, S0 = _problem(31, [200], 1, 64, 64, 0.05)
    o_ref, f_ref, _ = oracle.prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0)
    o, f = chunked_prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0, C=64)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, atol=1e-12)


def test_rounding_budget_of_the_state_chain():
    """At d = 128 over 4096 tokens, rounding every product operand to bf16 puts the
    final state ~3e-3 (relative Frobenius) from the oracle: above a 1e-3 budget.
    Keeping the operands that produce u and the state (T diag(beta), V, K*Gamma, the
    state, u and K*gamma_C/Gamma) at tf32 precision and the rest at bf16 brings it to
    ~5e-4.  This is why the tensor-core prefill runs that chain as tf32 products."""
    rng = np.random.default_rng(0)
    T, dk = 2048, 128
    q = rng.standard_normal((T, 1, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, 1, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q, k = bf16_round(q), bf16_round(k)
    v = bf16_round(rng.standard_normal((T, 1, dk)))
    la = (-0.05 * np.log1p(np.exp(rng.standard_normal((T, 1, dk))))).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((T, 1))))).astype(np.float32)
    _, f_ref, _ = oracle.prefill(q, k, v, la, beta)
    rel = lambda f: np.linalg.norm(f - f_ref) / np.linalg.norm(f_ref)
    _, f_bf16 = chunked_prefill(q, k, v, la, beta, rnd=bf16_round, state_rnd=bf16_round)
    _, f_mixed = chunked_prefill(q, k, v, la, beta, rnd=bf16_round, state_rnd=tf32_round)
    assert rel(f_bf16) > 1.5e-3
    assert rel(f_mixed) < 7e-4


@pytest.mark.parametrize("decay", [0.05, 1.0])
def test_folded_form_equals_recurrence(decay):
    """The four-matrix form (S <- Diag(gamma) S + P V + N S, o = Q' S + P2 V) is the
    same recurrence: exact arithmetic matches the oracle on ragged, decayed chunks."""
    q, k, v, la, beta, cu, S0 = _problem(40, [150], 1, 16, 12, decay)
    o_ref, f_ref, _ = oracle.prefill(q, k, v, la, beta, cu_seqlens=cu, init_state=S0)
    o, f = folded_unit(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0], C=64)
    np.testing.assert_allclose(o, o_ref[:, 0], atol=1e-12 * max(np.abs(o_ref).max(), 1.0))
    np.testing.assert_allclose(f, f_ref[0, 0], atol=1e-12 * max(np.abs(f_ref).max(), 1.0))


def test_rounding_budget_of_the_folded_form():
    """The two-kernel prefill's rounding points (bf16 N, Q', W and state operand;
    fp16 P, P2, V; P from bf16 high/low splits of Kd and T') stay well inside the
    bar at d = 128 over 2048 tokens, where all-bf16 operands would not."""
    rng = np.random.default_rng(0)
    T, dk = 2048, 128
    q = rng.standard_normal((T, 1, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, 1, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q, k = bf16_round(q), bf16_round(k)
    v = bf16_round(rng.standard_normal((T, 1, dk)))
    la = (-0.05 * np.log1p(np.exp(rng.standard_normal((T, 1, dk))))).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((T, 1))))).astype(np.float32)
    o_ref, f_ref, _ = oracle.prefill(q, k, v, la, beta)
    o, f = folded_unit(q[:, 0], k[:, 0], v[:, 0], la[:, 0].astype(np.float64), beta[:, 0].astype(np.float64),
                       kernel_rounding=True)
    assert np.linalg.norm(f - f_ref[0, 0]) / np.linalg.norm(f_ref[0, 0]) < 7e-4
    assert np.abs(o - o_ref[:, 0]).max() < 2e-3

