"""Independent float64 forms of the operator, used only to pin the oracle.

TEST INFRASTRUCTURE. Each form here is a different association order of the
same operator, written from the identities the pages prove. None of them
shares code with ``la_oracle.c``, so a wrong sign, index or term in either
one shows up as a disagreement. All arrays are for ONE sequence-head:
q,k [T,dk], v [T,dv], gates [T,dk] (gla) or [T] (gdn).
"""
from __future__ import annotations

import numpy as np


def elu1(x: np.ndarray) -> np.ndarray:
    """phi(x) = elu(x) + 1 with alpha = 1 (section 11.2 of the Hyena chapter)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def causal_mask(T: int) -> np.ndarray:
    """L_tj = 1 for j <= t (the diagonal included), else 0."""
    return np.tril(np.ones((T, T), dtype=np.float64))


def norm_masked_parallel(q, k, v):
    """Normalized elu+1 attention as one masked product.

    "Linear attention and Hyena", section 11.2 and Exercise 11.4:
    num = (L o (Q_phi K_phi^T)) V and den = (L o (Q_phi K_phi^T)) 1, with L
    causal including the diagonal. The final state is S_T = K_phi^T V and
    z_T = K_phi^T 1. Returns (o, S_T, z_T, den).
    """
    Qp, Kp = elu1(q), elu1(k)
    A = causal_mask(q.shape[0]) * (Qp @ Kp.T)
    num = A @ v
    den = A.sum(axis=1)
    return num / den[:, None], Kp.T @ v, Kp.sum(axis=0), den


def norm_decay_masked_parallel(q, k, v, gamma: float):
    """Normalized elu+1 attention with one fixed decay, as one masked product.

    "Linear attention and recurrent memory", Fixed decay versus an
    input-dependent gate, and its Pitfalls (the parallel form weights the
    pair (t, i) by gamma^(t-i), in the numerator and the normalizer alike):
    A_ti = gamma^(t-i) phi(q_t) . phi(k_i) for i <= t, num = A V, den = A 1.
    The final state is S_T = sum_i gamma^(T-1-i) phi(k_i) v_i^T and z_T the
    same sum of phi(k_i). Returns (o, S_T, z_T, den).
    """
    Qp, Kp = elu1(q), elu1(k)
    T = q.shape[0]
    t = np.arange(T, dtype=np.float64)
    W = np.where(t[:, None] >= t[None, :], float(gamma) ** np.maximum(t[:, None] - t[None, :], 0.0), 0.0)
    A = W * (Qp @ Kp.T)
    den = A.sum(axis=1)
    w_end = float(gamma) ** (T - 1 - t)
    return (A @ v) / den[:, None], (Kp * w_end[:, None]).T @ v, (Kp * w_end[:, None]).sum(axis=0), den


def gla_masked(q, k, v, gamma, identity_phi: bool = False):
    """Per-channel gated attention as a masked sum.

    "Linear attention and Hyena", section 11.3 and Exercise 11.5:
    y_t = sum_{j<=t} v_j sum_c phi(q_t)_c exp(G_tc - G_jc) phi(k_j)_c with
    G_t = sum_{i<=t} log gamma_i over the whole sequence. The final state is
    S_T[c,:] = sum_j exp(G_Tc - G_jc) phi(k_j)_c v_j. Returns (y, S_T).
    """
    f = (lambda x: np.asarray(x, np.float64)) if identity_phi else elu1
    Qp, Kp = f(q), f(k)
    G = np.cumsum(np.log(np.asarray(gamma, np.float64)), axis=0)   # [T,dk]
    T = q.shape[0]
    D = np.exp(G[:, None, :] - G[None, :, :])                       # [t,j,c]
    D *= causal_mask(T)[:, :, None]
    scores = np.einsum("tc,tjc,jc->tj", Qp, D, Kp)
    y = scores @ v
    S_T = (np.exp(G[-1][None, :] - G) * Kp).T @ v
    return y, S_T


def gla_factorized(q, k, v, gamma):
    """The "secondary" rescaling of section 11.3 (tiny T only).

    q~_t = phi(q_t) * e^{G_t}, k~_j = phi(k_j) * e^{-G_j}; then
    y = (L o (Q~ K~^T)) V. Overflows for long sequences by construction.
    """
    G = np.cumsum(np.log(np.asarray(gamma, np.float64)), axis=0)
    Qt = elu1(q) * np.exp(G)
    Kt = elu1(k) * np.exp(-G)
    return (causal_mask(q.shape[0]) * (Qt @ Kt.T)) @ v


def retnet_toeplitz(q, k, v, gamma: float):
    """Constant gate: the Toeplitz mask L_tj = gamma^(t-j) (section 11.3)."""
    T = q.shape[0]
    lag = np.arange(T)[:, None] - np.arange(T)[None, :]
    L = np.where(lag >= 0, float(gamma) ** np.maximum(lag, 0), 0.0)
    return (L * (elu1(q) @ elu1(k).T)) @ v


def additive_regrouped(q, k, v):
    """Plain additive memory read as a regrouped sum.

    "Beyond attention", section 18.1: sum_{j<=t} (q_t . k_j) v_j, which the
    page regroups into S_t q_t with S_t = sum_j v_j k_j^T.
    """
    return (causal_mask(q.shape[0]) * (q @ k.T)) @ v


def gdn_literal(q, k, v, g, beta, S0=None):
    """Gated delta rule in the product form of "Beyond attention", 18.2.

    S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t,
    with the identity matrix and the outer products formed explicitly.
    """
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    I = np.eye(dk)
    o = np.empty((T, dv))
    for t in range(T):
        kt = k[t][:, None]
        S = g[t] * S @ (I - beta[t] * (kt @ kt.T)) + beta[t] * np.outer(v[t], k[t])
        o[t] = S @ q[t]
    return o, S


def gdn_unrolled(q, k, v, g, beta, S0=None):
    """Brute-force unrolled gated delta rule (tiny T only).

    With A_i = g_i (I - beta_i k_i k_i^T), unrolling S_t = S_{t-1} A_t +
    beta_t v_t k_t^T gives S_t = S_0 A_1...A_t + sum_j beta_j v_j k_j^T
    A_{j+1}...A_t. Every product is rebuilt from scratch for every t.
    """
    T, dk = q.shape
    dv = v.shape[1]
    S0 = np.zeros((dv, dk)) if S0 is None else np.asarray(S0, dtype=np.float64)
    A = [g[i] * (np.eye(dk) - beta[i] * np.outer(k[i], k[i])) for i in range(T)]

    def prod(lo, hi):            # A_lo @ ... @ A_hi (inclusive, 0-based)
        P = np.eye(dk)
        for i in range(lo, hi + 1):
            P = P @ A[i]
        return P

    o = np.empty((T, dv))
    S = S0
    for t in range(T):
        S = S0 @ prod(0, t)
        for j in range(t + 1):
            S = S + beta[j] * np.outer(v[j], k[j]) @ prod(j + 1, t)
        o[t] = S @ q[t]
    return o, S


def kda_literal(q, k, v, alpha, beta, S0=None):
    """Gated delta rule with a diagonal decay, in product form.

    "Linear attention and recurrent memory", From fixed decay to KDA's gated
    delta write, with the decay per key channel:
    S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
    o_t = S_t q_t, every matrix formed explicitly. alpha [T, dk].
    """
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    I = np.eye(dk)
    o = np.empty((T, dv))
    for t in range(T):
        kt = k[t][:, None]
        S = S @ np.diag(alpha[t]) @ (I - beta[t] * (kt @ kt.T)) + beta[t] * np.outer(v[t], k[t])
        o[t] = S @ q[t]
    return o, S


def kda_unrolled(q, k, v, alpha, beta, S0=None):
    """Brute-force unrolled diagonal-decay delta rule (tiny T only).

    With A_i = Diag(alpha_i) (I - beta_i k_i k_i^T): S_t = S_0 A_1...A_t +
    sum_j beta_j v_j k_j^T A_{j+1}...A_t, every product rebuilt for every t.
    """
    T, dk = q.shape
    dv = v.shape[1]
    S0 = np.zeros((dv, dk)) if S0 is None else np.asarray(S0, dtype=np.float64)
    A = [np.diag(alpha[i]) @ (np.eye(dk) - beta[i] * np.outer(k[i], k[i])) for i in range(T)]

    def prod(lo, hi):
        P = np.eye(dk)
        for i in range(lo, hi + 1):
            P = P @ A[i]
        return P

    o = np.empty((T, dv))
    S = S0
    for t in range(T):
        S = S0 @ prod(0, t)
        for j in range(t + 1):
            S = S + beta[j] * np.outer(v[j], k[j]) @ prod(j + 1, t)
        o[t] = S @ q[t]
    return o, S
