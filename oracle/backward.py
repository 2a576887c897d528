"""Float64 gradients of the normalized elu+1 recurrence (with and without a
fixed decay), of the per-channel gated recurrence and of the gated delta rule
(scalar or per-channel decay), as test infrastructure.

TEST INFRASTRUCTURE, like the rest of ``oracle``: only ``tests/`` and
``bench.py``'s CPU legs use it.

The pages define the forward operator only ("Transformers are RNNs" as
summarized in "Beyond — Linear attention and recurrent memory": phi = elu + 1,
S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t), o_t = S_t^T
phi(q_t) / phi(q_t)^T z_t, update first) and name chunked training without
giving gradients. This module applies the chain rule to that recurrence, token
by token, in plain float64:

    f_t = phi(k_t), p_t = phi(q_t), num_t = S_t^T p_t, den_t = p_t . z_t
    dnum_t = do_t / den_t,  dden_t = -(do_t . num_t) / den_t^2
    dp_t   = S_t dnum_t + z_t dden_t
    GS_t   = dS_T + sum_{tau >= t} p_tau dnum_tau^T   (gradient reaching f_t v_t^T)
    Gz_t   = dz_T + sum_{tau >= t} p_tau dden_tau
    df_t   = GS_t v_t + Gz_t,  dv_t = GS_t^T f_t
    dq_t   = dp_t * phi'(q_t),  dk_t = df_t * phi'(k_t),  phi'(x) = 1 (x > 0), e^x (x <= 0)
    dS_0   = GS_0,  dz_0 = Gz_0

``tests/test_oracle_pins.py`` pins every output against central finite
differences of the C forward oracle (``oracle.run``), which shares no
arithmetic with this module; ``tests/test_backward_mutations.py`` plants
mistakes in copies of each function and checks that those pins catch them.
``gla_backward`` and ``delta_backward`` state their own chain rules.
"""
from __future__ import annotations

import numpy as np


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


def norm_backward(q, k, v, do, state_in=None, dstate_out=None):
    """Gradients of the normalized recurrence.

    q, k [B,H,T,dk]; v, do [B,H,T,dv]; state_in, dstate_out [B,H,dk*dv+dk]
    (S [dk,dv] then z [dk]) or None (zero state / no gradient on the final
    state). Returns (dq, dk, dv, dstate_in) in float64.
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    ss = dk * dv + dk
    sin = np.zeros((B, H, ss)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, ss)
    dso = np.zeros((B, H, ss)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, ss)
    f, p = _phi(k), _phi(q)
    # forward, keeping every state (update first)
    S = np.empty((B, H, T, dk, dv))
    z = np.empty((B, H, T, dk))
    s_prev = sin[..., :dk * dv].reshape(B, H, dk, dv).copy()
    z_prev = sin[..., dk * dv:].copy()
    for t in range(T):
        s_prev = s_prev + f[:, :, t, :, None] * v[:, :, t, None, :]
        z_prev = z_prev + f[:, :, t]
        S[:, :, t] = s_prev
        z[:, :, t] = z_prev
    num = np.einsum("bhtkv,bhtk->bhtv", S, p)
    den = np.einsum("bhtk,bhtk->bht", z, p)
    # reverse
    GS = dso[..., :dk * dv].reshape(B, H, dk, dv).copy()
    Gz = dso[..., dk * dv:].copy()
    dq = np.empty_like(q)
    dkk = np.empty_like(k)
    dvv = np.empty_like(v)
    for t in range(T - 1, -1, -1):
        dnum = do[:, :, t] / den[:, :, t, None]
        dden = -np.einsum("bhv,bhv->bh", do[:, :, t], num[:, :, t]) / den[:, :, t] ** 2
        dp = np.einsum("bhkv,bhv->bhk", S[:, :, t], dnum) + z[:, :, t] * dden[..., None]
        GS = GS + p[:, :, t, :, None] * dnum[:, :, None, :]
        Gz = Gz + p[:, :, t] * dden[..., None]
        df = np.einsum("bhkv,bhv->bhk", GS, v[:, :, t]) + Gz
        dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", GS, f[:, :, t])
        dq[:, :, t] = dp * _dphi(q[:, :, t])
        dkk[:, :, t] = df * _dphi(k[:, :, t])
    dsin = np.concatenate([GS.reshape(B, H, dk * dv), Gz], axis=-1)
    return dq, dkk, dvv, dsin


def norm_decay_backward(q, k, v, gamma, do, state_in=None, dstate_out=None):
    """Gradients of the normalized recurrence with a fixed decay per
    sequence-head (S_t = gamma S_{t-1} + phi(k_t) v_t^T, z likewise; the
    normalized variant with one gamma in (0, 1] per (b,h), as
    "Beyond — Linear attention and recurrent memory" states for a fixed
    decay). With G_t, g_t the whole gradients reaching S_t, z_t:

        G_t = p_t dnum_t^T + gamma G_{t+1},   g_t = p_t dden_t + gamma g_{t+1}
        (G_{T-1} and g_{T-1} also take dS_T, dz_T)
        df_t = G_t v_t + g_t,  dv_t = G_t^T f_t,  dp_t = S_t dnum_t + z_t dden_t
        dS_0 = gamma G_0,  dz_0 = gamma g_0
        dgamma = sum_t <G_t, S_{t-1}> + <g_t, z_{t-1}>

    gamma [B,H]; the rest as ``norm_backward``. Returns (dq, dk, dv,
    dstate_in, dgamma) in float64.
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    gm = np.asarray(gamma, np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    ss = dk * dv + dk
    sin = np.zeros((B, H, ss)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, ss)
    dso = np.zeros((B, H, ss)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, ss)
    f, p = _phi(k), _phi(q)
    S = np.empty((B, H, T + 1, dk, dv))   # S[:, :, t + 1] is the state after token t
    z = np.empty((B, H, T + 1, dk))
    S[:, :, 0] = sin[..., :dk * dv].reshape(B, H, dk, dv)
    z[:, :, 0] = sin[..., dk * dv:]
    for t in range(T):
        S[:, :, t + 1] = gm[..., None, None] * S[:, :, t] + f[:, :, t, :, None] * v[:, :, t, None, :]
        z[:, :, t + 1] = gm[..., None] * z[:, :, t] + f[:, :, t]
    num = np.einsum("bhtkv,bhtk->bhtv", S[:, :, 1:], p)
    den = np.einsum("bhtk,bhtk->bht", z[:, :, 1:], p)
    G = dso[..., :dk * dv].reshape(B, H, dk, dv).copy()   # gradient arriving from after token t
    g = dso[..., dk * dv:].copy()
    dq = np.empty_like(q)
    dkk = np.empty_like(k)
    dvv = np.empty_like(v)
    dgam = np.zeros((B, H))
    for t in range(T - 1, -1, -1):
        dnum = do[:, :, t] / den[:, :, t, None]
        dden = -np.einsum("bhv,bhv->bh", do[:, :, t], num[:, :, t]) / den[:, :, t] ** 2
        G = G + p[:, :, t, :, None] * dnum[:, :, None, :]
        g = g + p[:, :, t] * dden[..., None]
        dp = np.einsum("bhkv,bhv->bhk", S[:, :, t + 1], dnum) + z[:, :, t + 1] * dden[..., None]
        df = np.einsum("bhkv,bhv->bhk", G, v[:, :, t]) + g
        dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", G, f[:, :, t])
        dq[:, :, t] = dp * _dphi(q[:, :, t])
        dkk[:, :, t] = df * _dphi(k[:, :, t])
        dgam += np.einsum("bhkv,bhkv->bh", G, S[:, :, t]) + np.einsum("bhk,bhk->bh", g, z[:, :, t])
        G = gm[..., None, None] * G   # through S_t = gamma S_{t-1} + ...
        g = gm[..., None] * g
    dsin = np.concatenate([G.reshape(B, H, dk * dv), g], axis=-1)
    return dq, dkk, dvv, dsin, dgam


def norm_backward_chunked(q, k, v, do, C=64, state_in=None, dstate_out=None):
    """The same gradients as ``norm_backward``, by chunks of C tokens: the
    form a tensor-core backward computes. Per chunk c (Q, K the feature-mapped
    tiles, S_in, z_in the state entering it, P = L o Q K^T):

        num = P V + Q S_in,  den = P 1 + Q z_in
        dnum = dO / den,  dden = -rowsum(dO o num) / den^2
        dP = L o (dnum V^T + dden 1^T)
        dQ = dP K + dnum S_in^T + dden z_in^T
        dK = dP^T Q + V G^T + 1 g^T,   dV = P^T dnum + K G

    where G, g are the gradients of the state and normalizer after the chunk
    (the final-state cotangent plus Q^T dnum and Q^T dden of every later
    chunk), carried from the last chunk to the first; the initial state
    receives G, g after chunk 0 has added its own. dq = dQ o phi'(q),
    dk = dK o phi'(k).
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    ss = dk * dv + dk
    sin = np.zeros((B, H, ss)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, ss)
    dso = np.zeros((B, H, ss)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, ss)
    Qf, Kf = _phi(q), _phi(k)
    nch = (T + C - 1) // C
    # states entering every chunk (forward, by chunks)
    S_in = np.empty((B, H, nch, dk, dv))
    z_in = np.empty((B, H, nch, dk))
    S = sin[..., :dk * dv].reshape(B, H, dk, dv).copy()
    z = sin[..., dk * dv:].copy()
    for c in range(nch):
        sl = slice(c * C, min(T, (c + 1) * C))
        S_in[:, :, c], z_in[:, :, c] = S, z
        S = S + np.einsum("bhtk,bhtv->bhkv", Kf[:, :, sl], v[:, :, sl])
        z = z + Kf[:, :, sl].sum(axis=2)
    G = dso[..., :dk * dv].reshape(B, H, dk, dv).copy()
    g = dso[..., dk * dv:].copy()
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    for c in range(nch - 1, -1, -1):
        sl = slice(c * C, min(T, (c + 1) * C))
        Q, K, V, dO = Qf[:, :, sl], Kf[:, :, sl], v[:, :, sl], do[:, :, sl]
        n = Q.shape[2]
        L = np.tril(np.ones((n, n)))
        P = L * np.einsum("bhtk,bhjk->bhtj", Q, K)
        num = np.einsum("bhtj,bhjv->bhtv", P, V) + np.einsum("bhtk,bhkv->bhtv", Q, S_in[:, :, c])
        den = P.sum(-1) + np.einsum("bhtk,bhk->bht", Q, z_in[:, :, c])
        dnum = dO / den[..., None]
        dden = -np.einsum("bhtv,bhtv->bht", dO, num) / den ** 2
        dP = L * (np.einsum("bhtv,bhjv->bhtj", dnum, V) + dden[..., None])
        dQ = (np.einsum("bhtj,bhjk->bhtk", dP, K) + np.einsum("bhtv,bhkv->bhtk", dnum, S_in[:, :, c])
              + dden[..., None] * z_in[:, :, c][:, :, None, :])
        dK = np.einsum("bhtj,bhtk->bhjk", dP, Q) + np.einsum("bhjv,bhkv->bhjk", V, G) + g[:, :, None, :]
        dV = np.einsum("bhtj,bhtv->bhjv", P, dnum) + np.einsum("bhjk,bhkv->bhjv", K, G)
        dq[:, :, sl] = dQ * _dphi(q[:, :, sl])
        dkk[:, :, sl] = dK * _dphi(k[:, :, sl])
        dvv[:, :, sl] = dV
        # the state entering this chunk also reaches this chunk's outputs
        G = G + np.einsum("bhtk,bhtv->bhkv", Q, dnum)
        g = g + np.einsum("bhtk,bht->bhk", Q, dden)
    dsin = np.concatenate([G.reshape(B, H, dk * dv), g], axis=-1)
    return dq, dkk, dvv, dsin


def delta_backward(q, k, v, decay, beta, do, state_in=None, dstate_out=None):
    """Gradients of the gated delta rule, scalar or per-channel decay.

    The forward operator is the gated delta rule with the decay applied to
    the state before the error is taken ("Beyond attention" §18.2 for a
    scalar gate; "Linear attention and recurrent memory", from fixed decay to
    KDA, for a decay per key channel), S in R^{dv x dk}:

        S~_t = S_{t-1} Diag(a_t)      (a_t = g_t 1 for the scalar gate)
        u_t  = beta_t (v_t - S~_t k_t),   S_t = S~_t + u_t k_t^T,   o_t = S_t q_t

    The pages give no gradients. By the chain rule, with D_t the whole
    gradient reaching S_t (the final-state cotangent, then carried back) and
    every term taken at token t:

        D_t  += do_t q_t^T,                  dq_t = S_t^T do_t
        du    = D_t k_t
        dv_t  = beta_t du,                   dbeta_t = (v_t - S~_t k_t) . du
        dk_t  = D_t^T u_t - beta_t S~_t^T du
        dS~   = D_t - beta_t du k_t^T
        D_{t-1} = dS~ Diag(a_t)
        da_t  = column sums of dS~ o S_{t-1}   (their total for a scalar g_t)

    and dstate_in = D_0. q, k [B,H,T,dk]; v, do [B,H,T,dv]; decay [B,H,T]
    (scalar gate g) or [B,H,T,dk] (per-channel alpha); beta [B,H,T];
    state_in, dstate_out [B,H,dv*dk] (S row-major) or None. Returns
    (dq, dk, dv, ddecay, dbeta, dstate_in) in float64, ddecay shaped like
    decay.

    ``tests/test_oracle_pins.py`` pins every output against central finite
    differences of the C forward oracle (``oracle.run``), which shares no
    arithmetic with this module.
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    a = np.asarray(decay, np.float64)
    bt = np.asarray(beta, np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    per_channel = a.ndim == 4
    av = a if per_channel else np.broadcast_to(a[..., None], (B, H, T, dk))
    sin = np.zeros((B, H, dv, dk)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, dv, dk)
    # forward, keeping every state: S[:, :, t + 1] is the state after token t
    S = np.empty((B, H, T + 1, dv, dk))
    S[:, :, 0] = sin
    for t in range(T):
        st = S[:, :, t] * av[:, :, t, None, :]
        u = bt[:, :, t, None] * (v[:, :, t] - np.einsum("bhvk,bhk->bhv", st, k[:, :, t]))
        S[:, :, t + 1] = st + u[..., None] * k[:, :, t, None, :]
    D = np.zeros((B, H, dv, dk)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, dv, dk).copy()
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    da = np.empty((B, H, T, dk))
    db = np.empty((B, H, T))
    for t in range(T - 1, -1, -1):
        kt, qt = k[:, :, t], q[:, :, t]
        D = D + do[:, :, t, :, None] * qt[:, :, None, :]
        dq[:, :, t] = np.einsum("bhvk,bhv->bhk", S[:, :, t + 1], do[:, :, t])
        st = S[:, :, t] * av[:, :, t, None, :]
        err = v[:, :, t] - np.einsum("bhvk,bhk->bhv", st, kt)
        u = bt[:, :, t, None] * err
        du = np.einsum("bhvk,bhk->bhv", D, kt)
        dvv[:, :, t] = bt[:, :, t, None] * du
        db[:, :, t] = np.einsum("bhv,bhv->bh", err, du)
        dkk[:, :, t] = (np.einsum("bhvk,bhv->bhk", D, u)
                        - bt[:, :, t, None] * np.einsum("bhvk,bhv->bhk", st, du))
        dst = D - bt[:, :, t, None, None] * du[..., None] * kt[:, :, None, :]
        da[:, :, t] = np.einsum("bhvk,bhvk->bhk", dst, S[:, :, t])
        D = dst * av[:, :, t, None, :]
    dgate = da if per_channel else da.sum(axis=-1)
    return dq, dkk, dvv, dgate, db, D.reshape(B, H, dv * dk)


def delta_backward_chunked(q, k, v, g, beta, do, C=64, state_in=None, dstate_out=None):
    """The same gradients as ``delta_backward`` for a scalar gate, by chunks
    of C tokens: the form a chunkwise backward computes. Inside a chunk
    (rows r, s; b_r = sum of log g up to r, gam_r = e^{b_r}, gam_C and b_C
    those of its last token, lam_s = gam_C / gam_s, E_rs = e^{b_r - b_s}) the
    forward is the WY/UT chunk form of the rule ("Beyond attention" §18.2):

        A  = strictly lower (diag(beta) o E o K K^T),   Ti = (I + A)^{-1}
        W  = Ti diag(beta gam) K,   Ut = Ti diag(beta) V,   U = Ut - W S_0^T
        P  = lower (E o Q K^T),     O  = diag(gam) Q S_0^T + P U
        S_C = gam_C S_0 + U^T diag(lam) K

    so that, across chunks, both the state and its gradient follow one linear
    map X <- gam_C X - (X A'^T) B' + C'^T D' per chunk:
    forward S with (A', B', C', D') = (W, lam K, Ut, lam K), backward dS (from
    the last chunk) with (K, lam W, dO, Qh), Qh = diag(gam) Q - P W. With S_0
    and dS_C (the gradient reaching the chunk's last state) known, the chain
    rule through those four lines gives, per chunk:

        dU  = P^T dO + diag(lam) K dS_C^T,    dW = -dU S_0
        dRv = Ti^T dU,   dRk = Ti^T dW,       dA = -(dRv Ut^T + dRk W^T)  (strictly lower)
        dV  = diag(beta) dRv
        dP  = lower (dO U^T)
        dQ  = diag(gam) dO S_0 + (dP o E) K
        dK  = (dP o E)^T Q + diag(beta gam) dRk + F K + F^T K + diag(lam) U dS_C,
              F = diag(beta) (dA o E)
        dbeta_r = dRv_r . v_r + gam_r dRk_r . k_r + sum_s (dA o E o K K^T)_rs
        db_r    = gam_r dO_r . (S_0 q_r) + beta_r gam_r dRk_r . k_r
                  + rows minus columns of (dP o P) and of (dA o A)
                  (+ at the last token: gam_C <dS_C, S_0> + sum_s c_s, and
                  - c_s at s, c_s = lam_s (U dS_C)_s . k_s)
        dlog g_t = sum_{r >= t} db_r (inside the chunk),   dg = dlog g / g

    Padded rows of a ragged last chunk have k = q = v = do = 0, beta = 0 and
    g = 1, which leaves every real row unchanged. q, k [B,H,T,dk]; v, do
    [B,H,T,dv]; g, beta [B,H,T]; states [B,H,dv*dk] or None. Returns
    (dq, dk, dv, dg, dbeta, dstate_in) in float64.
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    g = np.asarray(g, np.float64)
    bt = np.asarray(beta, np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    nch = (T + C - 1) // C
    Tp = nch * C
    pad = lambda a, fill=0.0: np.concatenate(
        [a, np.full(a.shape[:2] + (Tp - T,) + a.shape[3:], fill)], axis=2) if Tp > T else a
    Q, K, V, dO = (pad(a).reshape(B, H, nch, C, -1) for a in (q, k, v, do))
    lg = pad(np.log(g)).reshape(B, H, nch, C)
    be = pad(bt).reshape(B, H, nch, C)
    ein = np.einsum
    # per chunk, independent of the state
    b = np.cumsum(lg, axis=-1)
    gam = np.exp(b)
    gC = gam[..., -1]
    lam = np.exp(b[..., -1:] - b)
    E = np.exp(b[..., :, None] - b[..., None, :])
    lower = np.tril(np.ones((C, C)))
    strict = np.tril(np.ones((C, C)), -1)
    KK = ein("...rk,...sk->...rs", K, K)
    A = strict * be[..., :, None] * E * KK
    Ti = np.linalg.inv(np.eye(C) + A)
    W = ein("...rs,...sk->...rk", Ti, (be * gam)[..., None] * K)
    Ut = ein("...rs,...sv->...rv", Ti, be[..., None] * V)
    P = lower * E * ein("...rk,...sk->...rs", Q, K)
    Qh = gam[..., None] * Q - ein("...rs,...sk->...rk", P, W)
    lK, lW = lam[..., None] * K, lam[..., None] * W

    def chain(X, c, a_, b_, c_, d_):
        # X <- gam_C X - (X a_^T) b_ + c_^T d_   for chunk c
        Y = ein("bhik,bhrk->bhir", X, a_[:, :, c])
        return (gC[:, :, c, None, None] * X - ein("bhir,bhrk->bhik", Y, b_[:, :, c])
                + ein("bhri,bhrk->bhik", c_[:, :, c], d_[:, :, c]))

    S0 = np.empty((B, H, nch, dv, dk))
    X = np.zeros((B, H, dv, dk)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, dv, dk)
    for c in range(nch):
        S0[:, :, c] = X
        X = chain(X, c, W, lK, Ut, lK)
    dSC = np.empty((B, H, nch, dv, dk))
    X = np.zeros((B, H, dv, dk)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, dv, dk)
    for c in range(nch - 1, -1, -1):
        dSC[:, :, c] = X
        X = chain(X, c, K, lW, dO, Qh)
    dstate_in = X.reshape(B, H, dv * dk)
    # per chunk, with S_0 and dS_C
    U = Ut - ein("...rk,...ik->...ri", W, S0)
    dU = ein("...rs,...ri->...si", P, dO) + lam[..., None] * ein("...rk,...ik->...ri", K, dSC)
    dWm = -ein("...ri,...ik->...rk", dU, S0)
    dRv = ein("...sr,...si->...ri", Ti, dU)
    dRk = ein("...sr,...sk->...rk", Ti, dWm)
    dA = -strict * (ein("...ri,...si->...rs", dRv, Ut) + ein("...rk,...sk->...rs", dRk, W))
    dP = lower * ein("...ri,...si->...rs", dO, U)
    dPE = dP * E
    F = be[..., :, None] * dA * E
    dS0q = ein("...ri,...ik->...rk", dO, S0)            # dO S_0
    dQ = gam[..., None] * dS0q + ein("...rs,...sk->...rk", dPE, K)
    US = ein("...ri,...ik->...rk", U, dSC)               # U dS_C
    dK = (ein("...rs,...rk->...sk", dPE, Q) + (be * gam)[..., None] * dRk
          + ein("...rs,...sk->...rk", F, K) + ein("...rs,...rk->...sk", F, K) + lam[..., None] * US)
    dV = be[..., None] * dRv
    rk = ein("...rk,...rk->...r", dRk, K)
    dbeta = ein("...rv,...rv->...r", dRv, V) + gam * rk + (dA * E * KK).sum(-1)
    dPP, dAA = dP * P, dA * A
    db = (gam * ein("...rk,...rk->...r", dS0q, Q) + be * gam * rk
          + dPP.sum(-1) - dPP.sum(-2) + dAA.sum(-1) - dAA.sum(-2))
    cs = lam * ein("...rk,...rk->...r", US, K)
    db = db - cs
    db[..., -1] += gC * ein("...ik,...ik->...", dSC, S0) + cs.sum(-1)
    dlg = np.flip(np.cumsum(np.flip(db, -1), -1), -1)
    unpad = lambda a: a.reshape((B, H, Tp) + a.shape[4:])[:, :, :T]
    dg = unpad(dlg) / g
    return unpad(dQ), unpad(dK), unpad(dV), dg, unpad(dbeta), dstate_in


def gla_backward(q, k, v, gamma, do, state_in=None, dstate_out=None, identity_phi=False):
    """Gradients of the per-channel gated recurrence (GLA / RetNet family,
    "Linear attention and Hyena" §11.3), S in R^{dk x dv}:

        S_t = diag(gamma_t) S_{t-1} + f_t v_t^T,   o_t = S_t^T p_t,
        f = phi(k), p = phi(q) (the identity under identity_phi)

    The pages give no gradients. By the chain rule, with D the whole gradient
    reaching S_t (the final-state cotangent, then carried back):

        D += p_t do_t^T,          dp_t = S_t do_t
        df_t = D v_t,             dv_t = D^T f_t
        dgamma_t = rowsums of D o S_{t-1}  (one per key channel)
        D <- diag(gamma_t) D;     dstate_in = D after token 0
        dq = dp o phi'(q), dk = df o phi'(k)

    q, k [B,H,T,dk]; v, do [B,H,T,dv]; gamma [B,H,T,dk]; state_in,
    dstate_out [B,H,dk*dv] (S row-major) or None. Returns (dq, dk, dv,
    dgamma, dstate_in) in float64.
    """
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    gm = np.asarray(gamma, np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if identity_phi:
        f, p = k, q
        dfk, dpq = np.ones_like(k), np.ones_like(q)
    else:
        f, p = _phi(k), _phi(q)
        dfk, dpq = _dphi(k), _dphi(q)
    sin = np.zeros((B, H, dk, dv)) if state_in is None else np.asarray(state_in, np.float64).reshape(B, H, dk, dv)
    S = np.empty((B, H, T + 1, dk, dv))   # S[:, :, t + 1] is the state after token t
    S[:, :, 0] = sin
    for t in range(T):
        S[:, :, t + 1] = gm[:, :, t, :, None] * S[:, :, t] + f[:, :, t, :, None] * v[:, :, t, None, :]
    D = np.zeros((B, H, dk, dv)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, dk, dv).copy()
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dg = np.empty((B, H, T, dk))
    for t in range(T - 1, -1, -1):
        D = D + p[:, :, t, :, None] * do[:, :, t, None, :]
        dq[:, :, t] = np.einsum("bhkv,bhv->bhk", S[:, :, t + 1], do[:, :, t]) * dpq[:, :, t]
        dkk[:, :, t] = np.einsum("bhkv,bhv->bhk", D, v[:, :, t]) * dfk[:, :, t]
        dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", D, f[:, :, t])
        dg[:, :, t] = np.einsum("bhkv,bhkv->bhk", D, S[:, :, t])
        D = gm[:, :, t, :, None] * D
    return dq, dkk, dvv, dg, D.reshape(B, H, dk * dv)
