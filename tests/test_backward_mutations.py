"""The backward oracle's finite-difference pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/backward.py`` (a dropped
term, a wrong operand, a wrong feature-map derivative, a lost cotangent, a
lost decay), inside the function it targets, loads the copy, and compares its
gradients with central differences of the (unmutated) C forward oracle:
every mutant must disagree.
"""
import os
import types

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "backward.py")

MUTANTS = {
    "drops_normalizer_gradient": ("dden = -np.einsum", "dden = 0.0 * np.einsum"),
    "drops_z_term_of_dp": ("+ z[:, :, t] * dden[..., None]", ""),
    "wrong_phi_derivative": ("return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))", "return np.ones_like(x)"),
    "df_from_state_not_gradient": ('df = np.einsum("bhkv,bhv->bhk", GS, v[:, :, t]) + Gz',
                                   'df = np.einsum("bhkv,bhv->bhk", S[:, :, t], v[:, :, t]) + Gz'),
    "dv_with_query_features": ('dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", GS, f[:, :, t])',
                               'dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", GS, p[:, :, t])'),
    "drops_final_state_cotangent": ("GS = dso[..., :dk * dv].reshape(B, H, dk, dv).copy()",
                                    "GS = np.zeros((B, H, dk, dv))"),
    "z_gradient_with_key_features": ("Gz = Gz + p[:, :, t] * dden[..., None]", "Gz = Gz + f[:, :, t] * dden[..., None]"),
}
# planted in norm_decay_backward
MUTANTS_DECAY = {
    "state_gradient_not_decayed": ("G = gm[..., None, None] * G   # through", "G = G   # through"),
    "gamma_gradient_against_later_state": ('np.einsum("bhkv,bhkv->bh", G, S[:, :, t])',
                                          'np.einsum("bhkv,bhkv->bh", G, S[:, :, t + 1])'),
    "normalizer_gradient_not_decayed": ("g = gm[..., None] * g", "g = g"),
}


# planted in delta_backward (gated delta rule, scalar and per-channel decay)
MUTANTS_DELTA = {
    "drops_write_correction_of_state_gradient": ("dst = D - bt[:, :, t, None, None] * du[..., None] * kt[:, :, None, :]",
                                                 "dst = D"),
    "dk_without_state_term": ('''
                        - bt[:, :, t, None] * np.einsum("bhvk,bhv->bhk", st, du))''', ")"),
    "dk_with_undecayed_state": ('np.einsum("bhvk,bhv->bhk", st, du)', 'np.einsum("bhvk,bhv->bhk", S[:, :, t], du)'),
    "dbeta_with_value_not_error": ('db[:, :, t] = np.einsum("bhv,bhv->bh", err, du)',
                                   'db[:, :, t] = np.einsum("bhv,bhv->bh", v[:, :, t], du)'),
    "decay_gradient_against_new_state": ('np.einsum("bhvk,bhvk->bhk", dst, S[:, :, t])',
                                         'np.einsum("bhvk,bhvk->bhk", dst, S[:, :, t + 1])'),
    "state_gradient_not_decayed": ("D = dst * av[:, :, t, None, :]", "D = dst"),
    "dq_from_previous_state": ('np.einsum("bhvk,bhv->bhk", S[:, :, t + 1], do[:, :, t])',
                               'np.einsum("bhvk,bhv->bhk", S[:, :, t], do[:, :, t])'),
    "dv_without_beta": ("dvv[:, :, t] = bt[:, :, t, None] * du", "dvv[:, :, t] = du"),
}


# planted in delta_backward_chunked (scalar gate, by chunks)
MUTANTS_CHUNKED = {
    "pair_gradient_without_transposed_term": ('+ ein("...rs,...sk->...rk", F, K) + ein("...rs,...rk->...sk", F, K)',
                                              '+ ein("...rs,...sk->...rk", F, K)'),
    "state_chain_without_decay": ("return (gC[:, :, c, None, None] * X", "return (X"),
    "pseudo_value_weight_gradient_sign": ("dWm = -ein(", "dWm = ein("),
    "dbeta_without_pair_term": (" + (dA * E * KK).sum(-1)", ""),
    "gate_drops_carried_state_term": ('db[..., -1] += gC * ein("...ik,...ik->...", dSC, S0) + cs.sum(-1)',
                                      "db[..., -1] += cs.sum(-1)"),
    "inclusive_mask_in_solve": ("A = strict * be", "A = lower * be"),
    "gate_prefix_sum_not_reversed": ("dlg = np.flip(np.cumsum(np.flip(db, -1), -1), -1)", "dlg = np.cumsum(db, -1)"),
    "gradient_chain_without_intra_chunk_output": ('Qh = gam[..., None] * Q - ein("...rs,...sk->...rk", P, W)',
                                                  "Qh = gam[..., None] * Q"),
}


# planted in gla_backward (per-channel gated attention)
MUTANTS_GLA = {
    "gate_gradient_against_new_state": ('dg[:, :, t] = np.einsum("bhkv,bhkv->bhk", D, S[:, :, t])',
                                        'dg[:, :, t] = np.einsum("bhkv,bhkv->bhk", D, S[:, :, t + 1])'),
    "state_gradient_not_decayed": ("D = gm[:, :, t, :, None] * D", "D = D"),
    "dq_from_previous_state": ('dq[:, :, t] = np.einsum("bhkv,bhv->bhk", S[:, :, t + 1], do[:, :, t])',
                               'dq[:, :, t] = np.einsum("bhkv,bhv->bhk", S[:, :, t], do[:, :, t])'),
    "dv_with_query_features": ('dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", D, f[:, :, t])',
                               'dvv[:, :, t] = np.einsum("bhkv,bhk->bhv", D, p[:, :, t])'),
    "dk_without_feature_map_derivative": ("v[:, :, t]) * dfk[:, :, t]", "v[:, :, t])"),
    "output_cotangent_with_key_features": ("D = D + p[:, :, t, :, None] * do[:, :, t, None, :]",
                                           "D = D + f[:, :, t, :, None] * do[:, :, t, None, :]"),
    "drops_final_state_cotangent": ("D = np.zeros((B, H, dk, dv)) if dstate_out is None else np.asarray(dstate_out, np.float64).reshape(B, H, dk, dv).copy()",
                                    "D = np.zeros((B, H, dk, dv))"),
}


def _split(text):
    """(head, norm_backward, norm_decay_backward) sources."""
    a = text.index("def norm_backward(")
    b = text.index("def norm_decay_backward(")
    return text[:a], text[a:b], text[b:]


def _load(text):
    mod = types.ModuleType("backward_mutant")
    exec(compile(text, "backward_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.fixture(scope="module")
def case():
    g = np.random.default_rng(53)
    B, H, T, dk, dv = 1, 1, 5, 3, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    ss = dk * dv + dk
    sin = g.standard_normal((B, H, ss)) * 0.3
    sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) + 1.0
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, ss))

    def loss():
        r = oracle.run("norm", q, k, v, None, None, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    eps = 1e-6
    fd = []
    for arr in (q, k, v, sin):
        grad = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            grad[idx] = (lp - lm) / (2 * eps)
        fd.append(grad)
    return (q, k, v, W, sin, Ws), fd


@pytest.fixture(scope="module")
def case_decay():
    g = np.random.default_rng(67)
    B, H, T, dk, dv = 1, 1, 5, 2, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    gm = np.array([[0.7]])
    ss = dk * dv + dk
    sin = g.standard_normal((B, H, ss)) * 0.3
    sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) + 1.0
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, ss))

    def loss():
        r = oracle.run("norm_decay", q, k, v, gm, None, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    eps = 1e-6
    fd = []
    for arr in (q, k, v, sin, gm):
        grad = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            grad[idx] = (lp - lm) / (2 * eps)
        fd.append(grad)
    return (q, k, v, gm, W, sin, Ws), fd


def _agrees(mod, case):
    (q, k, v, W, sin, Ws), fd = case
    got = mod.norm_backward(q, k, v, W, sin, Ws)
    return all(np.allclose(gr, f, rtol=1e-6, atol=1e-6) for gr, f in zip(got, fd))


def _agrees_decay(mod, case):
    (q, k, v, gm, W, sin, Ws), fd = case
    got = mod.norm_decay_backward(q, k, v, gm, W, sin, Ws)
    return all(np.allclose(gr, f, rtol=1e-6, atol=1e-6) for gr, f in zip(got, fd))


def test_unmutated_backward_agrees(case, case_decay):
    with open(SRC) as fh:
        mod = _load(fh.read())
    assert _agrees(mod, case)
    assert _agrees_decay(mod, case_decay)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, case):
    old, new = MUTANTS[name]
    with open(SRC) as fh:
        head, plain, decay = _split(fh.read())
    if head.count(old) == 1:   # a helper both functions share
        head = head.replace(old, new)
    else:
        assert plain.count(old) == 1, name
        plain = plain.replace(old, new)
    assert not _agrees(_load(head + plain + decay), case), name


@pytest.mark.parametrize("name", sorted(MUTANTS_DECAY))
def test_decay_mutant_is_caught(name, case_decay):
    old, new = MUTANTS_DECAY[name]
    with open(SRC) as fh:
        head, plain, decay = _split(fh.read())
    assert decay.count(old) == 1, name
    assert not _agrees_decay(_load(head + plain + decay.replace(old, new)), case_decay), name


def _delta_fd_case(variant, seed):
    g = np.random.default_rng(seed)
    B, H, T, dk, dv = 1, 1, 5, 3, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    a = g.uniform(0.5, 1.0, (B, H, T, dk) if variant == "kda" else (B, H, T))
    b = g.uniform(0.1, 0.9, (B, H, T))
    sin = g.standard_normal((B, H, dv * dk)) * 0.3
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, dv * dk))

    def loss():
        r = oracle.run(variant, q, k, v, a, b, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    eps = 1e-6
    fd = []
    for arr in (q, k, v, a, b, sin):
        grad = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            grad[idx] = (lp - lm) / (2 * eps)
        fd.append(grad)
    return (q, k, v, a, b, W, sin, Ws), fd


@pytest.fixture(scope="module")
def delta_cases():
    return {"gdn": _delta_fd_case("gdn", 103), "kda": _delta_fd_case("kda", 107)}


def _agrees_delta(mod, case):
    (q, k, v, a, b, W, sin, Ws), fd = case
    got = mod.delta_backward(q, k, v, a, b, W, sin, Ws)
    return all(np.allclose(gr, f, rtol=1e-6, atol=1e-6) for gr, f in zip(got, fd))


def test_unmutated_delta_backward_agrees(delta_cases):
    with open(SRC) as fh:
        mod = _load(fh.read())
    for case in delta_cases.values():
        assert _agrees_delta(mod, case)


@pytest.mark.parametrize("name", sorted(MUTANTS_DELTA))
def test_delta_mutant_is_caught(name, delta_cases):
    old, new = MUTANTS_DELTA[name]
    with open(SRC) as fh:
        text = fh.read()
    i = text.index("def delta_backward(")
    head, body = text[:i], text[i:]
    assert body.count(old) == 1, name
    mod = _load(head + body.replace(old, new))
    # caught when it disagrees with the finite differences on either decay
    assert not all(_agrees_delta(mod, c) for c in delta_cases.values()), name


def _agrees_chunked(mod, case, C):
    (q, k, v, a, b, W, sin, Ws), fd = case
    got = mod.delta_backward_chunked(q, k, v, a, b, W, C, sin, Ws)
    return all(np.allclose(gr, f, rtol=1e-6, atol=1e-6) for gr, f in zip(got, fd))


def test_unmutated_delta_backward_chunked_agrees(delta_cases):
    with open(SRC) as fh:
        mod = _load(fh.read())
    for C in (2, 4):
        assert _agrees_chunked(mod, delta_cases["gdn"], C)


@pytest.mark.parametrize("name", sorted(MUTANTS_CHUNKED))
def test_delta_chunked_mutant_is_caught(name, delta_cases):
    old, new = MUTANTS_CHUNKED[name]
    with open(SRC) as fh:
        text = fh.read()
    i = text.index("def delta_backward_chunked(")
    j = text.index("def gla_backward(")
    head, body, tail = text[:i], text[i:j], text[j:]
    assert body.count(old) == 1, name
    mod = _load(head + body.replace(old, new) + tail)
    # caught when either chunk size (both leave a ragged last chunk) disagrees
    assert not all(_agrees_chunked(mod, delta_cases["gdn"], C) for C in (2, 4)), name


@pytest.fixture(scope="module")
def gla_case():
    g = np.random.default_rng(127)
    B, H, T, dk, dv = 1, 1, 5, 3, 2
    q, k, v = g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dk)), g.standard_normal((B, H, T, dv))
    gm = g.uniform(0.4, 1.0, (B, H, T, dk))
    sin = g.standard_normal((B, H, dk * dv)) * 0.3
    W, Ws = g.standard_normal((B, H, T, dv)), g.standard_normal((B, H, dk * dv))

    def loss():
        r = oracle.run("gla", q, k, v, gm, None, sin)
        return float(np.sum(r.o * W) + np.sum(r.state * Ws))

    eps = 1e-6
    fd = []
    for arr in (q, k, v, gm, sin):
        grad = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            lp = loss()
            arr[idx] = a0 - eps
            lm = loss()
            arr[idx] = a0
            grad[idx] = (lp - lm) / (2 * eps)
        fd.append(grad)
    return (q, k, v, gm, W, sin, Ws), fd


def _agrees_gla(mod, case):
    (q, k, v, gm, W, sin, Ws), fd = case
    got = mod.gla_backward(q, k, v, gm, W, sin, Ws)
    return all(np.allclose(gr, f, rtol=1e-6, atol=1e-6) for gr, f in zip(got, fd))


def test_unmutated_gla_backward_agrees(gla_case):
    with open(SRC) as fh:
        assert _agrees_gla(_load(fh.read()), gla_case)


@pytest.mark.parametrize("name", sorted(MUTANTS_GLA))
def test_gla_mutant_is_caught(name, gla_case):
    old, new = MUTANTS_GLA[name]
    with open(SRC) as fh:
        text = fh.read()
    i = text.index("def gla_backward(")
    head, body = text[:i], text[i:]
    assert body.count(old) == 1, name
    assert not _agrees_gla(_load(head + body.replace(old, new)), gla_case), name
