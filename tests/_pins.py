"""Independent NumPy evaluations used to pin the fp64 oracle.

Nothing here imports the oracle or the CUDA package; each function reaches
the KDA result by a different route than the oracle's token loop, so that a
plausible slip in the oracle (a dropped term, a wrong sign, decay applied
after the write, the output read from the pre-update state, a transposed
operand) shows up as a disagreement.

All functions work on ONE head: q, k, log_alpha [T, Dk]; v [T, Dv];
beta [T]; S0 [Dk, Dv].
"""
from __future__ import annotations

import math

import numpy as np


def dense_brute_force(q, k, v, log_alpha, beta, S0):
    """Transition-matrix form of the recurrence.

    A_t = (I - beta_t k_t k_t^T) Diag(alpha_t) is formed as a dense Dk x Dk
    matrix, and the state after t tokens is assembled as

        S_t = A_t ... A_1 S0 + sum_{i<=t} (A_t ... A_{i+1}) beta_i k_i v_i^T

    with every transition product multiplied out explicitly (O(T^2 Dk^3)).
    Returns (o [T, Dv], S_T).
    """
    T, Dk = q.shape
    I = np.eye(Dk)
    A = [(I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(log_alpha[t])) for t in range(T)]
    o = np.zeros((T, v.shape[1]))
    S = S0
    for t in range(T):
        P = I.copy()                      # A_t ... A_1
        for s in range(t, -1, -1):
            P = P @ A[s]
        S = P @ S0
        for i in range(t + 1):
            Pi = I.copy()                 # A_t ... A_{i+1}
            for s in range(t, i, -1):
                Pi = Pi @ A[s]
            S = S + Pi @ (beta[i] * np.outer(k[i], v[i]))
        o[t] = S.T @ q[t]
    return o, S


def decay_products(log_alpha):
    """G[t, i, :] = prod_{s=i+1..t} alpha_s for i <= t (0 above the diagonal),
    built by running products of alpha (not by exponentiating cumulative sums)."""
    T, Dk = log_alpha.shape
    alpha = np.exp(log_alpha)
    G = np.zeros((T, T, Dk))
    for i in range(T):
        p = np.ones(Dk)
        G[i, i] = p
        for t in range(i + 1, T):
            p = p * alpha[t]
            G[t, i] = p
    return G


def gated_linear_attention(q, k, v, log_alpha):
    """Causal linear attention with per-channel decay and no delta term:
    o_t = sum_{i<=t} (q_t * prod_{s=i+1..t} alpha_s) . k_i  v_i.
    With alpha == 1 this is the masked product tril(Q K^T) V."""
    G = decay_products(log_alpha)
    scores = np.einsum("td,tid,id->ti", q, G, k)
    return scores @ v


def inverse_forward_substitution(L):
    """(I + L)^{-1} for strictly lower-triangular L, row by row."""
    C = L.shape[0]
    Tm = np.zeros((C, C))
    for t in range(C):
        row = np.zeros(C)
        row[t] = 1.0
        for i in range(t):
            row -= L[t, i] * Tm[i]
        Tm[t] = row
    return Tm


def inverse_neumann(L):
    """(I + L)^{-1} = prod_{m=0}^{ceil(log2 C)-1} (I + (-L)^{2^m}), exact because
    L is strictly lower triangular and hence nilpotent (N^C = 0)."""
    C = L.shape[0]
    I = np.eye(C)
    N = -L
    Tm = I.copy()
    P = N.copy()
    for _ in range(max(1, math.ceil(math.log2(C))) if C > 1 else 0):
        Tm = Tm @ (I + P)
        P = P @ P
    return Tm


def chunked_wy(q, k, v, log_alpha, beta, S0, C, inverse="forward"):
    """Chunkwise evaluation of the recurrence (the form the GPU kernels use).

    Within a chunk, with g_t the chunk-local cumulative log decay,
      Kt = k * exp(g_t), Kb = k * exp(-g_t), Qt = q * exp(g_t),
      Kh = k * exp(g_C - g_t),
      L  = strict_lower(diag(beta) Kt Kb^T),  A = lower_incl(Qt Kb^T),
      U  = (I + L)^{-1} diag(beta) (V - Kt S),
      O  = Qt S + A U,   S <- Diag(exp(g_C)) S + Kh^T U.
    Returns (o [T, Dv], S_T, flops) where flops counts the eight C x C x D
    and six C x D x D multiply-adds of this schedule (inverse excluded).
    """
    T, Dk = q.shape
    Dv = v.shape[1]
    S = S0.copy()
    o = np.zeros((T, Dv))
    flops = 0
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        n = c1 - c0
        g = np.cumsum(log_alpha[c0:c1], axis=0)
        Kt = k[c0:c1] * np.exp(g)
        Kb = k[c0:c1] * np.exp(-g)
        Qt = q[c0:c1] * np.exp(g)
        Kh = k[c0:c1] * np.exp(g[-1] - g)
        b = beta[c0:c1]
        L = np.tril(b[:, None] * (Kt @ Kb.T), -1)
        A = np.tril(Qt @ Kb.T)
        flops += 2 * (2 * n * n * Dk)
        Tm = inverse_forward_substitution(L) if inverse == "forward" else inverse_neumann(L)
        X = b[:, None] * (v[c0:c1] - Kt @ S)
        U = Tm @ X
        O = Qt @ S + A @ U
        flops += 2 * n * Dk * Dv * 2 + 2 * n * n * Dv * 2
        S = np.exp(g[-1])[:, None] * S + Kh.T @ U
        flops += 2 * n * Dk * Dv
        o[c0:c1] = O
    return o, S, flops
