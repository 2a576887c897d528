"""Pins of the float64 oracle against what the pages and the mathematics fix.

Every test here runs on the CPU. Each compares the C recurrence with
something independent of it: a printed worked example, a closed form, or a
different association order proved equal on the pages.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def one(variant, q, k, v, gate=None, beta=None, state=None, **kw):
    """Run the oracle on a single sequence-head; arrays [T, d]."""
    ex = lambda a: None if a is None else np.asarray(a, np.float64)[None, None]
    st = None if state is None else np.asarray(state, np.float64).reshape(1, 1, -1)
    r = oracle.run(variant, ex(q), ex(k), ex(v), ex(gate), ex(beta), st, **kw)
    den = None if r.den is None else r.den[0, 0]
    return r.o[0, 0], r.state[0, 0], den


def rng(seed):
    return np.random.default_rng(seed)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ---------------------------------------------------------------- (a) norm

@pytest.mark.parametrize("T", [64, 512])
def test_norm_recurrent_equals_masked_parallel(T):
    # "Linear attention and Hyena" 11.2: the two forms agree to machine
    # precision in float64 (5.6e-16 at T=64, 2e-16 at T=512 printed).
    r = rng(T)
    q, k, v = (r.standard_normal((T, 16)) for _ in range(3))
    o, st, den = one("norm", q, k, v)
    o_p, S_p, z_p, den_p = forms.norm_masked_parallel(q, k, v)
    S, z = oracle.split_norm_state(st, 16, 16)
    assert np.max(np.abs(o - o_p)) <= 1e-12
    assert np.max(np.abs(den - den_p) / den_p) <= 1e-12
    assert np.max(np.abs(S - S_p)) <= 1e-12 * max(1.0, np.max(np.abs(S_p)))
    assert np.max(np.abs(z - z_p)) <= 1e-12 * np.max(z_p)


def test_norm_feature_map_closed_form():
    # phi = elu+1: phi(-ln 2) = 1/2 on the exp branch, phi(1) = 2 on the
    # linear branch. With d_k = d_v = 1 the output is a phi-weighted mean:
    # o_2 = (1/2 * 1 + 2 * 0) / (1/2 + 2) = 0.2 exactly; o_1 = v_1.
    q = np.array([[0.3], [-0.7]])
    k = np.array([[-math.log(2.0)], [1.0]])
    v = np.array([[1.0], [0.0]])
    o, st, den = one("norm", q, k, v)
    assert o[0, 0] == pytest.approx(1.0, abs=1e-15)
    assert o[1, 0] == pytest.approx(0.2, abs=1e-15)
    # den_2 = phi(q_2) * (phi(k_1) + phi(k_2)) = e^{-0.7} * 2.5
    assert den[1] == pytest.approx(math.exp(-0.7) * 2.5, rel=1e-15)
    assert st[0] == pytest.approx(0.5, abs=1e-15) and st[1] == pytest.approx(2.5, abs=1e-15)


def test_norm_first_token_and_prefix_mean():
    r = rng(1)
    T, d = 20, 8
    q, v = r.standard_normal((T, d)), r.standard_normal((T, d))
    k = np.tile(r.standard_normal((1, d)), (T, 1))          # identical keys
    o, _, _ = one("norm", q, k, v)
    assert np.allclose(o[0], v[0], atol=1e-15, rtol=0)       # token attends to itself
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(o - prefix_mean)) <= 1e-13


def test_norm_output_in_value_hull():
    r = rng(2)
    T, d = 100, 8
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    o, _, _ = one("norm", q, k, v)
    lo = np.minimum.accumulate(v, axis=0)
    hi = np.maximum.accumulate(v, axis=0)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


@pytest.mark.parametrize("variant", ["norm", "norm_decay", "gla", "gdn", "kda"])
def test_causality(variant):
    # Changing tokens after t leaves outputs up to t bit-identical.
    r = rng(3)
    T, d, t0 = 40, 8, 17
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    gate = beta = None
    if variant == "norm_decay":
        gate = 0.9
    if variant == "gla":
        gate = sigmoid(r.standard_normal((T, d)) + 2)
    if variant == "gdn":
        k = unit(k)
        gate, beta = sigmoid(r.standard_normal(T) + 3), sigmoid(r.standard_normal(T))
    if variant == "kda":
        k = unit(k)
        gate, beta = sigmoid(r.standard_normal((T, d)) + 3), sigmoid(r.standard_normal(T))
    o1, _, _ = one(variant, q, k, v, gate, beta)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[t0 + 1:] += 5.0
    k2[t0 + 1:] = -k2[t0 + 1:]
    v2[t0 + 1:] *= 3.0
    g2 = None if gate is None else np.array(gate, np.float64)
    if g2 is not None and g2.ndim > 0:
        g2[t0 + 1:] = 0.5
    o2, _, _ = one(variant, q2, k2, v2, g2, beta)
    assert np.array_equal(o1[: t0 + 1], o2[: t0 + 1])
    assert not np.array_equal(o1[t0 + 1:], o2[t0 + 1:])


# ------------------------------------------------------- (a') norm with decay

@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.995])
@pytest.mark.parametrize("T", [64, 200])
def test_norm_decay_recurrent_equals_masked_parallel(gamma, T):
    # "Linear attention and recurrent memory", Fixed decay and its Pitfalls:
    # the recurrence and the parallel form weighted by gamma^(t-i) agree,
    # numerator and normalizer alike.
    r = rng(int(T + 1000 * gamma))
    q, k, v = r.standard_normal((T, 16)), r.standard_normal((T, 16)), r.standard_normal((T, 12))
    o, st, den = one("norm_decay", q, k, v, gamma)
    o_p, S_p, z_p, den_p = forms.norm_decay_masked_parallel(q, k, v, gamma)
    S, z = oracle.split_norm_state(st, 16, 12)
    assert np.max(np.abs(o - o_p)) <= 1e-12 * max(1.0, np.max(np.abs(o_p)))
    assert np.max(np.abs(den - den_p) / den_p) <= 1e-12
    assert np.max(np.abs(S - S_p)) <= 1e-12 * max(1.0, np.max(np.abs(S_p)))
    assert np.max(np.abs(z - z_p)) <= 1e-12 * np.max(z_p)


def test_norm_decay_one_is_undecayed():
    # gamma = 1 is the undecayed form (the module's own reference check).
    r = rng(41)
    T = 90
    q, k, v = (r.standard_normal((T, 8)) for _ in range(3))
    o1, st1, den1 = one("norm_decay", q, k, v, 1.0)
    o0, st0, den0 = one("norm", q, k, v)
    assert np.max(np.abs(o1 - o0)) <= 1e-13 * max(1.0, np.max(np.abs(o0)))
    assert np.max(np.abs(st1 - st0)) <= 1e-13 * max(1.0, np.max(np.abs(st0)))
    assert np.max(np.abs(den1 - den0) / den0) <= 1e-13


def test_norm_decay_constant_key_closed_form():
    # One key repeated: every score phi(q_t).phi(k) is the same c_t, so
    # o_t = sum_i gamma^(t-i) v_i / sum_i gamma^(t-i), den_t = c_t (1 - gamma^(t+1)) / (1 - gamma),
    # z_T = phi(k) (1 - gamma^T) / (1 - gamma).
    r = rng(42)
    T, d, gamma = 30, 6, 0.8
    k = np.tile(r.standard_normal(d), (T, 1))
    q, v = r.standard_normal((T, d)), r.standard_normal((T, 3))
    o, st, den = one("norm_decay", q, k, v, gamma)
    t = np.arange(T)
    W = np.where(t[:, None] >= t[None, :], gamma ** np.maximum(t[:, None] - t[None, :], 0), 0.0)
    expect = (W @ v) / W.sum(axis=1, keepdims=True)
    assert np.max(np.abs(o - expect)) <= 1e-13
    c = forms.elu1(q) @ forms.elu1(k[0])
    assert np.max(np.abs(den - c * (1 - gamma ** (t + 1)) / (1 - gamma)) / den) <= 1e-13
    _, z = oracle.split_norm_state(st, d, 3)
    assert np.max(np.abs(z - forms.elu1(k[0]) * (1 - gamma ** T) / (1 - gamma))) <= 1e-13 * np.max(z)


# ----------------------------------------------------------------- (b) gla

@pytest.mark.parametrize("identity_phi", [False, True])
def test_gla_recurrent_equals_masked(identity_phi):
    # "Linear attention and Hyena" 11.3 / Exercise 11.5 (2.8e-14 printed for
    # their data-dependent gate).
    r = rng(4)
    T, dk, dv = 64, 16, 8
    q, k, v = r.standard_normal((T, dk)), r.standard_normal((T, dk)), r.standard_normal((T, dv))
    gamma = sigmoid(r.standard_normal((T, dk)) + 1.5)
    o, S, _ = one("gla", q, k, v, gamma, identity_phi=identity_phi)
    y, S_T = forms.gla_masked(q, k, v, gamma, identity_phi=identity_phi)
    scale = max(1.0, np.max(np.abs(y)))
    assert np.max(np.abs(o - y)) <= 1e-12 * scale
    assert np.max(np.abs(S.reshape(dk, dv) - S_T)) <= 1e-12 * max(1.0, np.max(np.abs(S_T)))


def test_gla_constant_gate_is_toeplitz():
    r = rng(5)
    T, d = 48, 8
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    gam = 0.9
    o, _, _ = one("gla", q, k, v, np.full((T, d), gam))
    ref = forms.retnet_toeplitz(q, k, v, gam)
    assert np.max(np.abs(o - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gla_unit_gate_is_norm_numerator():
    # gamma = 1 reduces the gated state to the undecayed one, so the gla
    # output equals the normalized output times its denominator.
    r = rng(6)
    T, d = 50, 8
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    o_g, S_g, _ = one("gla", q, k, v, np.ones((T, d)))
    o_n, st_n, den = one("norm", q, k, v)
    assert np.max(np.abs(o_g - o_n * den[:, None])) <= 1e-12 * np.max(np.abs(o_g))
    assert np.max(np.abs(S_g - st_n[: d * d])) <= 1e-12 * np.max(np.abs(S_g))


def test_gla_factorized_rescaling_tiny():
    r = rng(7)
    T, d = 12, 6
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    gamma = sigmoid(r.standard_normal((T, d)) + 1)
    o, _, _ = one("gla", q, k, v, gamma)
    ref = forms.gla_factorized(q, k, v, gamma)
    assert np.max(np.abs(o - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gla_gate_timing_closed_form():
    # gamma_t decays the state BEFORE token t's write: o_2 = phi(q_2)(gamma_2
    # phi(k_1) v_1 + phi(k_2) v_2); gamma_1 only touches the zero state.
    q = np.array([[0.0], [0.5]])
    k = np.array([[1.0], [-1.0]])
    v = np.array([[2.0], [3.0]])
    gamma = np.array([[0.25], [0.5]])
    o, S, _ = one("gla", q, k, v, gamma)
    phi_k1, phi_k2, phi_q2 = 2.0, math.exp(-1.0), 1.5
    assert o[0, 0] == pytest.approx(1.0 * phi_k1 * 2.0, rel=1e-15)
    expect = phi_q2 * (0.5 * phi_k1 * 2.0 + phi_k2 * 3.0)
    assert o[1, 0] == pytest.approx(expect, rel=1e-15)


def test_additive_memory_regrouped_sum():
    # "Beyond attention" 18.1 and its browser lab: for 50 random keys and
    # values, the regrouped sum equals the state recurrence S = sum v k^T.
    r = rng(8)
    T, d = 50, 32
    q, k, v = (r.standard_normal((T, d)) for _ in range(3))
    o, _, _ = one("gla", q, k, v, np.ones((T, d)), identity_phi=True)
    ref = forms.additive_regrouped(q, k, v)
    assert np.max(np.abs(o - ref)) <= 1e-12 * np.max(np.abs(ref))


# ----------------------------------------------------------------- (c) gdn

def _writes(case):
    ks = np.array([w[0] for w in case["writes"]], np.float64)
    vs = np.array([[w[1]] for w in case["writes"]], np.float64)
    T = len(ks)
    return ks, vs, np.ones(T), np.ones(T)


def test_gdn_two_key_example_golden():
    with open(os.path.join(GOLDEN, "two_key_delta.json")) as f:
        case = json.load(f)["cases"][0]
    ks, vs, g, b = _writes(case)
    q = np.array([[0.0, 1.0], [0.0, 1.0], [0.0, 1.0]])     # read the orthogonal key
    o, S, _ = one("gdn", q, ks, vs, g, b)
    assert S.tolist() == case["final_state"]               # exact: [5, 3]
    assert o[2, 0] == 3.0                                   # orthogonal association kept


def test_gdn_repeated_key_overwrites():
    with open(os.path.join(GOLDEN, "two_key_delta.json")) as f:
        case = json.load(f)["cases"][1]
    ks, vs, g, b = _writes(case)
    q = np.array([[1.0, 0.0]] * 3)
    o, S, _ = one("gdn", q, ks, vs, g, b)
    assert o[1, 0] == case["recall_after_second_write"]
    assert S.tolist() == case["final_state"]


def test_gdn_beta_one_unit_key_recalls_exactly():
    # With beta_t = 1 and |k_t| = 1 the write leaves S_t k_t = v_t for any
    # gate (the delta term removes what the decayed state returns for k_t).
    r = rng(9)
    T, dk, dv = 30, 16, 8
    q = unit(r.standard_normal((T, dk)))
    k = unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    g = sigmoid(r.standard_normal(T) + 1)
    o, _, _ = one("gdn", k, k, v, g, np.ones(T))              # read with q = k_t
    assert np.max(np.abs(o - v)) <= 1e-13


def test_gdn_equals_product_form():
    # The concept-page form (error against the decayed state) equals
    # g S (I - beta k k^T) + beta v k^T of "Beyond attention" 18.2.
    r = rng(10)
    T, dk, dv = 40, 12, 10
    q, k, v = r.standard_normal((T, dk)), unit(r.standard_normal((T, dk))), r.standard_normal((T, dv))
    g, b = sigmoid(r.standard_normal(T) + 2), sigmoid(r.standard_normal(T))
    S0 = r.standard_normal((dv, dk)) * 0.3
    o, S, _ = one("gdn", q, k, v, g, b, state=S0)
    o_l, S_l = forms.gdn_literal(q, k, v, g, b, S0)
    assert np.max(np.abs(o - o_l)) <= 1e-12 * np.max(np.abs(o_l))
    assert np.max(np.abs(S.reshape(dv, dk) - S_l)) <= 1e-12 * np.max(np.abs(S_l))


def test_gdn_gate_one_is_gradient_step():
    # g = 1: S_t = S_{t-1} - beta (S_{t-1} k - v) k^T ("Beyond attention" 18.2).
    r = rng(11)
    dk, dv = 8, 5
    S0 = r.standard_normal((dv, dk))
    k = unit(r.standard_normal((1, dk)))
    v, q = r.standard_normal((1, dv)), r.standard_normal((1, dk))
    beta = 0.37
    _, S, _ = one("gdn", q, k, v, np.ones(1), np.array([beta]), state=S0)
    expect = S0 - beta * np.outer(S0 @ k[0] - v[0], k[0])
    assert np.max(np.abs(S.reshape(dv, dk) - expect)) <= 1e-15 * 10


def test_gdn_beta_zero_is_pure_decay():
    r = rng(12)
    T, dk, dv = 10, 6, 4
    S0 = r.standard_normal((dv, dk))
    q, k, v = r.standard_normal((T, dk)), unit(r.standard_normal((T, dk))), r.standard_normal((T, dv))
    g = sigmoid(r.standard_normal(T) + 1)
    o, S, _ = one("gdn", q, k, v, g, np.zeros(T), state=S0)
    dec = np.cumprod(g)
    assert np.max(np.abs(S.reshape(dv, dk) - dec[-1] * S0)) <= 1e-15 * 10
    assert np.max(np.abs(o - dec[:, None] * (q @ S0.T))) <= 1e-14


def test_gdn_orthonormal_keys_exact_recall():
    # K <= d_k orthonormal keys, beta = 1, g = 1: every binding recalls exactly.
    r = rng(13)
    dk, dv, K = 16, 8, 16
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Qm.T[:K]
    vals = r.standard_normal((K, dv))
    _, S, _ = one("gdn", keys, keys, vals, np.ones(K), np.ones(K))
    S = S.reshape(dv, dk)
    assert np.max(np.abs(keys @ S.T - vals)) <= 1e-13


def test_gdn_unrolled_transition_product():
    r = rng(14)
    T, dk, dv = 12, 6, 5
    q, k, v = r.standard_normal((T, dk)), unit(r.standard_normal((T, dk))), r.standard_normal((T, dv))
    g, b = sigmoid(r.standard_normal(T) + 2), sigmoid(r.standard_normal(T))
    S0 = r.standard_normal((dv, dk)) * 0.5
    o, S, _ = one("gdn", q, k, v, g, b, state=S0)
    o_u, S_u = forms.gdn_unrolled(q, k, v, g, b, S0)
    assert np.max(np.abs(o - o_u)) <= 1e-12 * np.max(np.abs(o_u))
    assert np.max(np.abs(S.reshape(dv, dk) - S_u)) <= 1e-12 * np.max(np.abs(S_u))


def test_figure_18_2_delta_vs_additive():
    # "Beyond attention", Figure 18.2: 4x4 state; a and b perpendicular, c
    # overlaps a; write a, b, c, then a new value under a. The delta rule
    # recalls exactly the new value for a; plain addition returns old + new
    # + (c . a) times c's value.
    r = rng(15)
    a, b = np.eye(4)[0], np.eye(4)[1]
    c = unit(np.array([1.0, 0.0, 1.0, 0.0]))
    keys = np.stack([a, b, c, a])
    vals = r.standard_normal((4, 4))
    _, S_d, _ = one("gdn", keys, keys, vals, np.ones(4), np.ones(4))
    assert np.max(np.abs(S_d.reshape(4, 4) @ a - vals[3])) <= 1e-15 * 10
    o_add, _, _ = one("gla", keys, keys, vals, np.ones((4, 4)), identity_phi=True)
    expect = vals[0] + vals[3] + (c @ a) * vals[2]
    assert np.max(np.abs(o_add[3] - expect)) <= 1e-14


# ------------------------------------------- (c') delta rule, diagonal decay

def kda_inputs(r, T, dk, dv):
    q, k, v = r.standard_normal((T, dk)), unit(r.standard_normal((T, dk))), r.standard_normal((T, dv))
    alpha = sigmoid(r.standard_normal((T, dk)) + 2.5)
    beta = sigmoid(r.standard_normal(T))
    return q, k, v, alpha, beta


def test_kda_equals_product_form():
    # "Linear attention and recurrent memory", the KDA bridge: the corrective
    # write after a per-channel decay, S Diag(alpha)(I - beta k k^T) + beta v k^T.
    r = rng(51)
    q, k, v, alpha, beta = kda_inputs(r, 50, 12, 7)
    S0 = r.standard_normal((7, 12)) * 0.3
    o, st, _ = one("kda", q, k, v, alpha, beta, state=S0)
    o_l, S_l = forms.kda_literal(q, k, v, alpha, beta, S0)
    assert np.max(np.abs(o - o_l)) <= 1e-12 * max(1.0, np.max(np.abs(o_l)))
    assert np.max(np.abs(st.reshape(7, 12) - S_l)) <= 1e-12 * max(1.0, np.max(np.abs(S_l)))


def test_kda_unrolled_transition_product():
    r = rng(52)
    q, k, v, alpha, beta = kda_inputs(r, 6, 5, 3)
    o, st, _ = one("kda", q, k, v, alpha, beta)
    o_u, S_u = forms.kda_unrolled(q, k, v, alpha, beta)
    assert np.max(np.abs(o - o_u)) <= 1e-13 and np.max(np.abs(st.reshape(3, 5) - S_u)) <= 1e-13


def test_kda_uniform_decay_is_gdn():
    # alpha_t = g_t on every channel is the scalar-gated delta rule (c).
    r = rng(53)
    T, dk, dv = 40, 8, 6
    q, k, v, _, beta = kda_inputs(r, T, dk, dv)
    g = sigmoid(r.standard_normal(T) + 3)
    o1, st1, _ = one("kda", q, k, v, np.repeat(g[:, None], dk, axis=1), beta)
    o0, st0, _ = one("gdn", q, k, v, g, beta)
    assert np.max(np.abs(o1 - o0)) <= 1e-13 * max(1.0, np.max(np.abs(o0)))
    assert np.max(np.abs(st1 - st0)) <= 1e-13 * max(1.0, np.max(np.abs(st0)))


def test_kda_beta_zero_is_channel_decay():
    # No write: each key channel of the state decays by its own running product.
    r = rng(54)
    T, dk, dv = 20, 6, 4
    q, k, v, alpha, _ = kda_inputs(r, T, dk, dv)
    S0 = r.standard_normal((dv, dk))
    o, st, _ = one("kda", q, k, v, alpha, np.zeros(T), state=S0)
    P = np.cumprod(alpha, axis=0)
    for t in (0, 7, T - 1):
        assert np.max(np.abs(o[t] - (S0 * P[t]) @ q[t])) <= 1e-13
    assert np.max(np.abs(st.reshape(dv, dk) - S0 * P[-1])) <= 1e-13


def test_kda_unit_key_full_write_recalls_exactly():
    # beta = 1 and a unit key: reading that key right after the write returns
    # the written value, whatever the decay and the state before.
    r = rng(55)
    T, dk, dv = 10, 8, 5
    _, k, v, alpha, _ = kda_inputs(r, T, dk, dv)
    S0 = r.standard_normal((dv, dk))
    o, _, _ = one("kda", k, k, v, alpha, np.ones(T), state=S0)
    assert np.max(np.abs(o - v)) <= 1e-12


# ------------------------------------------------------ all: state passing

@pytest.mark.parametrize("variant", ["norm", "norm_decay", "gla", "gdn", "kda"])
def test_split_continuation_equals_one_shot(variant):
    r = rng(16)
    T, dk, dv, T1 = 37, 8, 6, 15
    q, k, v = r.standard_normal((T, dk)), r.standard_normal((T, dk)), r.standard_normal((T, dv))
    gate = beta = None
    if variant == "norm_decay":
        gate = 0.93
    if variant == "gla":
        gate = sigmoid(r.standard_normal((T, dk)) + 2)
    if variant == "gdn":
        k = unit(k)
        gate, beta = sigmoid(r.standard_normal(T) + 3), sigmoid(r.standard_normal(T))
    if variant == "kda":
        k = unit(k)
        gate, beta = sigmoid(r.standard_normal((T, dk)) + 3), sigmoid(r.standard_normal(T))
    o, st, _ = one(variant, q, k, v, gate, beta)
    sl = lambda a, s: None if a is None else (a if np.ndim(a) == 0 else a[s])
    a, b = slice(0, T1), slice(T1, T)
    o1, st1, _ = one(variant, q[a], k[a], v[a], sl(gate, a), sl(beta, a))
    o2, st2, _ = one(variant, q[b], k[b], v[b], sl(gate, b), sl(beta, b), state=st1)
    assert np.max(np.abs(np.concatenate([o1, o2]) - o)) <= 1e-13 * max(1, np.max(np.abs(o)))
    assert np.max(np.abs(st2 - st)) <= 1e-13 * max(1, np.max(np.abs(st)))


def test_oracle_batches_are_independent():
    # A batched call equals per-sequence calls (no cross-talk between (b,h)).
    r = rng(17)
    B, H, T, d = 2, 3, 9, 4
    q, k, v = (r.standard_normal((B, H, T, d)) for _ in range(3))
    g = sigmoid(r.standard_normal((B, H, T)) + 2)
    be = sigmoid(r.standard_normal((B, H, T)))
    res = oracle.run("gdn", q, unit(k), v, g, be)
    for bb in range(B):
        for hh in range(H):
            o, S, _ = one("gdn", q[bb, hh], unit(k[bb, hh]), v[bb, hh], g[bb, hh], be[bb, hh])
            assert np.array_equal(res.o[bb, hh], o)
            assert np.array_equal(res.state[bb, hh], S)


# ------------------------------------------------------------- gradients of (a)

def _fd_loss(q, k, v, sin, W, Ws):
    r = oracle.run("norm", q, k, v, None, None, sin)
    return float(np.sum(r.o * W) + np.sum(r.state * Ws))


@pytest.mark.parametrize("with_state", [False, True])
def test_norm_backward_matches_finite_differences(with_state):
    # Every gradient of the float64 backward against central differences of
    # the C forward recurrence, entry by entry, on a tiny problem with a
    # cotangent on the outputs and on the final state (S and z).
    from oracle import backward
    g = rng(41 + with_state)
    B, H, T, dk, dv = 1, 2, 6, 3, 4
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    ss = dk * dv + dk
    sin = None
    if with_state:
        sin = g.standard_normal((B, H, ss)) * 0.3
        sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) + 1.0
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, ss))
    dq, dk_, dv_, dsin = backward.norm_backward(q, k, v, W, sin, Ws)
    eps = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk_), ("v", v, dv_)) + ((("s", sin, dsin),) if with_state else ()):
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = _fd_loss(q, k, v, sin, W, Ws)
            arr[idx] = a0 - eps
            lm = _fd_loss(q, k, v, sin, W, Ws)
            arr[idx] = a0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_norm_backward_state_only_closed_form():
    # With a cotangent on the final state alone, the gradient reaching token t
    # is the constant dS_T (and dz_T): dv_t = dS_T^T phi(k_t),
    # dk_t = (dS_T v_t + dz_T) * phi'(k_t), dq = 0, dstate_in = dstate_out.
    from oracle import backward
    g = rng(43)
    B, H, T, dk, dv = 2, 1, 5, 4, 3
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    dso = g.standard_normal((B, H, dk * dv + dk))
    dq, dk_, dv_, dsin = backward.norm_backward(q, k, v, np.zeros((B, H, T, dv)), None, dso)
    dS = dso[..., :dk * dv].reshape(B, H, dk, dv)
    dz = dso[..., dk * dv:]
    phi = np.where(k > 0, k + 1, np.exp(np.minimum(k, 0)))
    dphi = np.where(k > 0, 1.0, np.exp(np.minimum(k, 0)))
    assert np.allclose(dq, 0.0)
    assert np.allclose(dv_, np.einsum("bhkv,bhtk->bhtv", dS, phi), rtol=1e-12, atol=1e-12)
    assert np.allclose(dk_, (np.einsum("bhkv,bhtv->bhtk", dS, v) + dz[:, :, None, :]) * dphi, rtol=1e-12, atol=1e-12)
    assert np.allclose(dsin, dso)


def test_norm_backward_matches_autograd_of_the_parallel_form():
    # The same gradients from a different association order: torch autograd
    # (float64, CPU) through the explicit masked parallel form num = (L o
    # Q_phi K_phi^T) V, den = (L o Q_phi K_phi^T) 1, against the reverse
    # recurrence of oracle/backward.py (zero initial state).
    torch = pytest.importorskip("torch")
    from oracle import backward
    g = rng(47)
    B, H, T, dk, dv = 1, 2, 9, 4, 3
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    W = g.standard_normal((B, H, T, dv))
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))

    def phi(x):
        return torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))

    A = torch.tril(phi(tq) @ phi(tk).transpose(-1, -2))
    o = (A @ tv) / A.sum(-1, keepdim=True)
    (o * torch.tensor(W)).sum().backward()
    dq, dk_, dv_, _ = backward.norm_backward(q, k, v, W)
    for got, ref in ((dq, tq.grad), (dk_, tk.grad), (dv_, tv.grad)):
        assert np.allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("gamma", [0.9, 0.35])
def test_norm_decay_backward_matches_finite_differences(gamma):
    # The decayed gradients (q, k, v, the initial state and gamma itself)
    # against central differences of the C forward recurrence.
    from oracle import backward
    g = rng(59)
    B, H, T, dk, dv = 1, 2, 6, 3, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    gm = np.array([[gamma, gamma * 0.8]])
    ss = dk * dv + dk
    sin = g.standard_normal((B, H, ss)) * 0.3
    sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) + 1.0
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, ss))

    def loss():
        r = oracle.run("norm_decay", q, k, v, gm, None, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    dq, dk_, dv_, dsin, dgam = backward.norm_decay_backward(q, k, v, gm, W, sin, Ws)
    eps = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk_), ("v", v, dv_), ("s", sin, dsin), ("gamma", gm, dgam)):
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_norm_decay_backward_at_one_is_undecayed():
    # gamma = 1 gives the undecayed gradients exactly
    from oracle import backward
    g = rng(61)
    B, H, T, dk, dv = 2, 1, 7, 3, 4
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    W = g.standard_normal((B, H, T, dv))
    a = backward.norm_backward(q, k, v, W)
    b = backward.norm_decay_backward(q, k, v, np.ones((B, H)), W)
    for x, y in zip(a, b[:4]):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("C,T", [(4, 13), (8, 16), (64, 37)])
def test_norm_backward_chunked_equals_token_by_token(C, T):
    # The chunkwise form of the gradients (the tensor-core algebra) equals the
    # token-by-token reverse recurrence, ragged tail and start state included.
    from oracle import backward
    g = rng(71 + C)
    B, H, dk, dv = 1, 2, 3, 5
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    ss = dk * dv + dk
    sin = g.standard_normal((B, H, ss)) * 0.3
    sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) + 1.0
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, ss))
    a = backward.norm_backward(q, k, v, W, sin, Ws)
    b = backward.norm_backward_chunked(q, k, v, W, C, sin, Ws)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------- gradients of (c) and its per-channel form

def _delta_case(g, per_channel, B=1, H=2, T=6, dk=3, dv=2):
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    a = g.uniform(0.5, 1.0, (B, H, T, dk) if per_channel else (B, H, T))
    b = g.uniform(0.1, 0.9, (B, H, T))
    sin = g.standard_normal((B, H, dv * dk)) * 0.3
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, dv * dk))
    return q, k, v, a, b, sin, W, Ws


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_delta_backward_matches_finite_differences(variant):
    # Every gradient of the float64 backward (q, k, v, the decay, beta and the
    # initial state) against central differences of the C forward recurrence,
    # entry by entry, with cotangents on the outputs and the final state.
    from oracle import backward
    q, k, v, a, b, sin, W, Ws = _delta_case(rng(83 if variant == "gdn" else 89), variant == "kda")

    def loss():
        r = oracle.run(variant, q, k, v, a, b, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    grads = backward.delta_backward(q, k, v, a, b, W, sin, Ws)
    eps = 1e-6
    for name, arr, grad in zip(("q", "k", "v", "decay", "beta", "s"), (q, k, v, a, b, sin), grads):
        assert grad.shape == arr.shape, name
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_delta_backward_frozen_state_closed_form():
    # beta = 0 and a decay of 1 leave the state at S_0, so o_t = S_0 q_t: the
    # gradient reaching token t is D_t = dS_T + sum_{tau >= t} do_tau q_tau^T,
    # and dq_t = S_0^T do_t, dv = dk = 0, dbeta_t = (v_t - S_0 k_t) . D_t k_t,
    # dg_t = <D_t, S_0>, dstate_in = D_0.
    from oracle import backward
    g = rng(97)
    B, H, T, dk, dv = 2, 1, 5, 4, 3
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    S0 = g.standard_normal((B, H, dv, dk))
    do, dso = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, dv, dk))
    dq, dk_, dv_, dg, db, dsin = backward.delta_backward(q, k, v, np.ones((B, H, T)), np.zeros((B, H, T)), do,
                                                         S0.reshape(B, H, -1), dso.reshape(B, H, -1))
    D = dso[:, :, None] + np.cumsum(np.einsum("bhtv,bhtk->bhtvk", do, q)[:, :, ::-1], axis=2)[:, :, ::-1]   # D_t
    assert np.allclose(dq, np.einsum("bhvk,bhtv->bhtk", S0, do), rtol=1e-12, atol=1e-12)
    assert np.allclose(dv_, 0.0) and np.allclose(dk_, 0.0)
    err = v - np.einsum("bhvk,bhtk->bhtv", S0, k)
    assert np.allclose(db, np.einsum("bhtv,bhtvk,bhtk->bht", err, D, k), rtol=1e-12, atol=1e-12)
    assert np.allclose(dg, np.einsum("bhtvk,bhvk->bht", D, S0), rtol=1e-12, atol=1e-12)
    assert np.allclose(dsin.reshape(B, H, dv, dk), D[:, :, 0], rtol=1e-12, atol=1e-12)


def test_delta_backward_uniform_channels_is_scalar_gate():
    # A per-channel decay equal on every channel is the scalar gate: the same
    # gradients, the scalar gate's being the sum over channels.
    from oracle import backward
    q, k, v, a, b, sin, W, Ws = _delta_case(rng(101), False, B=2, H=1, T=7, dk=4, dv=3)
    s = backward.delta_backward(q, k, v, a, b, W, sin, Ws)
    c = backward.delta_backward(q, k, v, np.repeat(a[..., None], 4, axis=-1), b, W, sin, Ws)
    for i in (0, 1, 2, 4, 5):
        assert np.allclose(s[i], c[i], rtol=1e-12, atol=1e-12)
    assert np.allclose(s[3], c[3].sum(-1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("C,T", [(4, 13), (8, 16), (16, 37), (64, 130)])
def test_delta_backward_chunked_equals_token_by_token(C, T):
    # The chunkwise form of the scalar-gate gradients (per-chunk UT inverse,
    # the state and its gradient carried by chunks) equals the token-by-token
    # reverse recurrence, which the finite-difference pin above holds to the C
    # forward oracle: ragged tail, start state and final-state cotangent included.
    from oracle import backward
    q, k, v, a, b, sin, W, Ws = _delta_case(rng(103 + C), False, B=2, H=1, T=T, dk=6, dv=5)
    a = 1.0 / (1.0 + np.exp(-(rng(107).standard_normal(a.shape) + 1.0)))   # gates down to ~0.05
    x = backward.delta_backward(q, k, v, a, b, W, sin, Ws)
    y = backward.delta_backward_chunked(q, k, v, a, b, W, C, sin, Ws)
    for name, u, w in zip(("dq", "dk", "dv", "dg", "dbeta", "dstate_in"), x, y):
        assert u.shape == w.shape, name
        assert np.allclose(u, w, rtol=1e-11, atol=1e-12), (name, np.abs(u - w).max())


# ------------------------------------------------------------- gradients of (b)

@pytest.mark.parametrize("identity_phi", [False, True])
def test_gla_backward_matches_finite_differences(identity_phi):
    # Every gradient of the float64 backward (q, k, v, the per-channel gate,
    # the initial state) against central differences of the C forward
    # recurrence, entry by entry, with cotangents on the outputs and the
    # final state.
    from oracle import backward
    g = rng(109 + identity_phi)
    B, H, T, dk, dv = 1, 2, 6, 3, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    gm = g.uniform(0.4, 1.0, (B, H, T, dk))
    sin = g.standard_normal((B, H, dk * dv)) * 0.3
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, dk * dv))

    def loss():
        r = oracle.run("gla", q, k, v, gm, None, sin, identity_phi=identity_phi)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    grads = backward.gla_backward(q, k, v, gm, W, sin, Ws, identity_phi=identity_phi)
    eps = 1e-6
    for name, arr, grad in zip(("q", "k", "v", "gamma", "s"), (q, k, v, gm, sin), grads):
        assert grad.shape == arr.shape, name
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_gla_backward_state_only_closed_form():
    # Gate 1 and a cotangent on the final state alone: the gradient reaching
    # every token is dS_T, so dv_t = dS_T^T phi(k_t), dk_t = (dS_T v_t) o
    # phi'(k_t), dq = 0, dgamma_t = rowsums(dS_T o S_{t-1}), dstate_in = dS_T.
    from oracle import backward
    g = rng(113)
    B, H, T, dk, dv = 2, 1, 5, 4, 3
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    S0 = g.standard_normal((B, H, dk, dv))
    dS = g.standard_normal((B, H, dk, dv))
    dq, dk_, dv_, dg, dsin = backward.gla_backward(q, k, v, np.ones((B, H, T, dk)), np.zeros((B, H, T, dv)),
                                                   S0.reshape(B, H, -1), dS.reshape(B, H, -1))
    phi = np.where(k > 0, k + 1, np.exp(np.minimum(k, 0)))
    dphi = np.where(k > 0, 1.0, np.exp(np.minimum(k, 0)))
    prev = S0[:, :, None] + np.cumsum(phi[..., :, None] * v[..., None, :], axis=2) - phi[..., :, None] * v[..., None, :]
    assert np.allclose(dq, 0.0)
    assert np.allclose(dv_, np.einsum("bhkv,bhtk->bhtv", dS, phi), rtol=1e-12, atol=1e-12)
    assert np.allclose(dk_, np.einsum("bhkv,bhtv->bhtk", dS, v) * dphi, rtol=1e-12, atol=1e-12)
    assert np.allclose(dg, np.einsum("bhkv,bhtkv->bhtk", dS, prev), rtol=1e-11, atol=1e-11)
    assert np.allclose(dsin.reshape(B, H, dk, dv), dS)
