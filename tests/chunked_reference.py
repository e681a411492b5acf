"""Chunkwise restatement of the KDA recurrence (test-only, numpy, float64).

The pages say that real deployments do not loop token by token but run a
chunkwise-parallel form (WY representation plus UT transform) and omit the
algebra ("K3 attention, three-piece set", KDA engineering-details paragraph;
"From 124M to 2.8T", chapter 3, intra-chunk parallel / inter-chunk serial).
This module writes that algebra out so the tests can check it against the
token-by-token oracle BEFORE any kernel relies on it.

For one chunk of rows r = 0..C-1 starting from state S0 (d_k x d_v), with
g_r = sum_{s<=r} log alpha_s (a vector over key channels) and gamma_r = e^{g_r}:

  S_r  = Diag(gamma_r) S0 + sum_{s<=r} (k_s * gamma_r / gamma_s) u_s^T
  A    = strict-lower( diag(beta) (K*Gamma) (K/Gamma)^T )
  (I + A) U = diag(beta) V - diag(beta) (K*Gamma) S0          (UT transform)
  U    = T diag(beta) V - T diag(beta) (K*Gamma) S0 = U~ - W S0 (WY factors)
  O    = scale [ (Q*Gamma) S0 + lower( (Q*Gamma)(K/Gamma)^T ) U ]
  S_C  = Diag(gamma_{C-1}) S0 + (K * gamma_{C-1} / Gamma)^T U

``rnd`` lets a test round the matrix-product operands (e.g. to bf16) at the
points where a tensor-core implementation would, to predict rounding error.
"""
from __future__ import annotations

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (via float32, ties to even)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def tf32_round(x: np.ndarray) -> np.ndarray:
    """Round to 10 explicit mantissa bits (ties to even)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0xFFF + ((u >> 13) & 1)) >> 13 << 13
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def f16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest IEEE fp16 (10 explicit mantissa bits, ties to even)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


def _ident(x):
    return x


def chunked_unit(q, k, v, log_alpha, beta, S0=None, C=64, rnd=None, state_rnd=None):
    """One (sequence, head) unit.  q, k, log_alpha: [T, dk]; v: [T, dv]; beta: [T].

    Rounding points (identity when None):
      rnd       -- operands of the products that only shape the output and the
                   k-k interaction matrix: Q*Gamma, K*Gamma and K/Gamma in A and
                   (Q*Gamma)(K/Gamma)^T, and that masked matrix itself;
      state_rnd -- operands of the chain that produces u and the state:
                   T' = (I+A)^-1 diag(beta), K*Gamma and V as multiplied by T',
                   W, the state, u and K*gamma_C/Gamma (defaults to rnd).
    beta is folded into the columns of the inverse: U~ = T' V, W = T' (K*Gamma).
    Returns (o [T, dv], S_final)."""
    rnd = rnd or _ident
    state_rnd = state_rnd or rnd
    T, dk = q.shape
    dv = v.shape[1]
    scale = 1.0 / np.sqrt(dk)
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        n = c1 - c0
        qc, kc, vc = q[c0:c1], k[c0:c1], v[c0:c1]
        bc = beta[c0:c1]
        g = np.cumsum(log_alpha[c0:c1], axis=0)
        Qg = rnd(scale * qc * np.exp(g))
        Kg = kc * np.exp(g)
        Kgi = rnd(kc * np.exp(-g))
        Kd = state_rnd(kc * np.exp(g[-1] - g))
        A = bc[:, None] * np.tril(rnd(Kg) @ Kgi.T, -1)
        Aqk = rnd(np.tril(Qg @ Kgi.T, 0))
        Tb = state_rnd(np.linalg.solve(np.eye(n) + A, np.eye(n)) * bc[None, :])
        W = state_rnd(Tb @ state_rnd(Kg))
        Ut = Tb @ state_rnd(vc)
        Sr = state_rnd(S)
        U = Ut - W @ Sr
        Ur = state_rnd(U)
        o[c0:c1] = Qg @ Sr + Aqk @ Ur
        S = np.exp(g[-1])[:, None] * S + Kd.T @ Ur
    return o, S


def chunked_prefill(q, k, v, log_alpha, beta, cu_seqlens=None, init_state=None, C=64, rnd=None,
                    state_rnd=None):
    """Packed sequences, all heads.  Shapes as the oracle's prefill.
    Returns (o [T, H, dv], final_state [N, H, dk, dv])."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    log_alpha = np.asarray(log_alpha, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    o = np.zeros((T, H, dv))
    fs = np.zeros((N, H, dk, dv))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S0 = None if init_state is None else init_state[n, h]
            if t1 == t0:
                fs[n, h] = 0.0 if S0 is None else S0
                continue
            o[t0:t1, h], fs[n, h] = chunked_unit(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h],
                                                 log_alpha[t0:t1, h], beta[t0:t1, h], S0, C,
                                                 rnd, state_rnd)
    return o, fs


def folded_unit(q, k, v, log_alpha, beta, S0=None, C=64, kernel_rounding=False):
    """The same chunk update folded into four matrices per chunk, the form the
    two-kernel tensor-core prefill uses.  Substituting U = U~ - W S0 into the
    output and state lines above gives, with Kd = K*gamma_C/Gamma:

      S_C = Diag(gamma_C) S0 + P V + N S0      P  = Kd^T T',  N = -Kd^T W
      O   = Q' S0 + P2 V                       Q' = scale Q*Gamma - Aqk W,  P2 = Aqk T'

    (T' = (I + A)^-1 diag(beta); Aqk as above).  With kernel_rounding the operands
    are rounded where the kernels round them: bf16 Q*Gamma, K*Gamma, K/Gamma, Aqk,
    W, N, Q' and the state operand of N S0 and Q' S0; T' and Kd each split into a
    bf16 high part and a bf16 low part, P formed from hi.hi + hi.lo + lo.hi; fp16
    P, P2 and V; W and P2 use the high part of T'; the state itself stays fp32.
    Returns (o [T, dv], S_final)."""
    B = bf16_round if kernel_rounding else _ident
    F = f16_round if kernel_rounding else _ident
    T, dk = q.shape
    dv = v.shape[1]
    scale = 1.0 / np.sqrt(dk)
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        n = c1 - c0
        qc, kc, vc, bc = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        g = np.cumsum(log_alpha[c0:c1], axis=0)
        Kg, Ki, Qg = B(kc * np.exp(g)), B(kc * np.exp(-g)), B(scale * qc * np.exp(g))
        A = bc[:, None] * np.tril(Kg @ Ki.T, -1)
        Aqk = B(np.tril(Qg @ Ki.T, 0))
        Tp = np.linalg.solve(np.eye(n) + A, np.eye(n)) * bc[None, :]
        Kd = kc * np.exp(g[-1] - g)
        th, kh = B(Tp), B(Kd)
        tl, kl = B(Tp - th), B(Kd - kh)
        W = B(th @ Kg)
        if kernel_rounding:
            P = F(kh.T @ th + kh.T @ tl + kl.T @ th)
        else:
            P = Kd.T @ Tp
        N = B(-(kh.T @ W))
        Qp = B(Qg - Aqk @ W)
        P2 = F(Aqk @ th)
        Vr, Sr = F(vc), B(S)
        o[c0:c1] = Qp @ Sr + P2 @ Vr
        S = np.exp(g[-1])[:, None] * S + N @ Sr + P @ Vr
    return o, S
