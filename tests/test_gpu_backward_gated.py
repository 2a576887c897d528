"""Gradients of the gated prefills (la_backward_gated: the gated delta rule
with a scalar gate or a per-channel decay, and the per-channel gated
variant) against the float64 oracle's (oracle/backward.py, ``delta_backward``
and ``gla_backward``, pinned by finite differences of the forward oracle), on
the same seeded inputs."""
import numpy as np
import pytest

import workloads as W
from _helpers import TOL, oracle_inputs, slice_rel_err, to_torch

pytestmark = pytest.mark.gpu

la = pytest.importorskip("gated_delta_rule_causal_gb300")


def _workload(variant, B, H, T, d, io, dv=None):
    base = {"gdn": W.GDN_B2H16_T8192_D128, "gla": W.GLA_B4H16_T4096_D128,
            "norm_decay": W.NORM_DECAY_B4H8_T2048_D64,
            "kda": W.KDA_DECODE_N256H16_D128.with_(B=4, H=16, T=2048, decode_steps=0, state_std=0.0)}[variant]
    return W.small(base, B=B, H=H, T=T, dk=d, dv=dv or d).with_(io=io)


def _case(variant, B, H, T, d, io, seed, with_state=True, with_dstate=True, flags=0, dv=None):
    import torch
    from oracle import backward
    dv = dv or d
    w = _workload(variant, B, H, T, d, io, dv)
    inp = W.draw(w, seed)
    q, k, v, g, b = oracle_inputs(inp)
    rng = np.random.default_rng(seed + 1000)
    ss = d * dv + (d if variant == "norm_decay" else 0)
    do_s = W.round_io(rng.standard_normal((B, H, T, dv)), io)
    do64 = W.as_f64(do_s)
    sin = (rng.standard_normal((B, H, ss)) * 0.1).astype(np.float32) if with_state else None
    if sin is not None and variant == "norm_decay":   # a positive normalizer state
        sin[..., d * dv:] = np.abs(sin[..., d * dv:]) * 50 + 1.0
    dso = (rng.standard_normal((B, H, ss)) * 0.05).astype(np.float32) if with_dstate else None
    h = la.Handle(B, H, d, dv, io=io, flags=flags)
    dev = h.device
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    got = h.backward_gated(to_torch(inp.q, dev), to_torch(inp.k, dev), to_torch(inp.v, dev),
                           to_torch(inp.gate, dev), to_torch(inp.beta, dev), to_torch(do_s, dev), t(sin), t(dso),
                           variant=variant)
    if variant in ("gla", "norm_decay"):
        assert got[4] is None
        got = got[:4] + got[5:]
    torch.cuda.synchronize()
    # the scalar-gate rule in bf16 with square heads: four chunkwise launches;
    # otherwise the row kernel and its conversion (norm_decay: after the forward's)
    if variant == "gdn" and io == "bf16" and dv == d:
        assert h.last_launches() == 4
    elif variant == "norm_decay":
        assert h.last_launches() >= 3
    else:
        assert h.last_launches() == 2
    assert h.status() == la.LA_OK
    h.close()
    if variant == "gla":
        ref = backward.gla_backward(q, k, v, g, do64, sin, dso, identity_phi=bool(flags & la.LA_FLAG_IDENTITY_PHI))
    elif variant == "norm_decay":
        rq, rk, rv, rs, rg = backward.norm_decay_backward(q, k, v, g, do64, sin, dso)
        ref = (rq, rk, rv, rg, rs)
    else:
        ref = backward.delta_backward(q, k, v, g, b, do64, sin, dso)
    return [x.float().cpu().numpy() for x in got], ref


NAMES = ("dq", "dk", "dv", "dgate", "dbeta", "dstate_in")
NAMES_GLA = ("dq", "dk", "dv", "dgate", "dstate_in")


def names(variant):
    return NAMES_GLA if variant in ("gla", "norm_decay") else NAMES


@pytest.mark.parametrize("variant", ["gdn", "kda", "gla", "norm_decay"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("io", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 37, 200])
def test_backward_gated_parity(variant, d, io, T):
    got, ref = _case(variant, 1, 2, T, d, io, seed=T + d + {"gdn": 0, "kda": 7, "gla": 13, "norm_decay": 19}[variant])
    for name, x, r in zip(names(variant), got, ref):
        assert x.shape == r.shape, name
        assert np.all(np.isfinite(x)), name
        assert slice_rel_err(x, r) <= TOL[io], (name, slice_rel_err(x, r))


@pytest.mark.parametrize("with_state,with_dstate", [(False, False), (True, False), (False, True)])
def test_backward_gated_optional_states(with_state, with_dstate):
    got, ref = _case("gdn", 2, 3, 65, 64, "bf16", seed=5, with_state=with_state, with_dstate=with_dstate)
    for name, x, r in zip(NAMES, got, ref):
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))


@pytest.mark.parametrize("variant", ["gdn", "kda", "gla", "norm_decay"])
def test_backward_gated_long_sequence(variant):
    # 2048 tokens: 128 segments walked back through their checkpoints
    got, ref = _case(variant, 1, 2, 2048, 64, "bf16", seed=17)
    for name, x, r in zip(names(variant), got, ref):
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_gla_identity_feature_map(d):
    # LA_FLAG_IDENTITY_PHI: the per-channel gated variant without phi
    got, ref = _case("gla", 1, 2, 100, d, "bf16", seed=29, flags=la.LA_FLAG_IDENTITY_PHI)
    for name, x, r in zip(NAMES_GLA, got, ref):
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))


def test_backward_gated_rejects_what_it_cannot_run():
    import torch
    h = la.Handle(1, 1, 32, 32)
    z = torch.zeros((1, 1, 4, 32), dtype=torch.bfloat16, device=h.device)
    g = torch.ones((1, 1, 4), device=h.device)
    with pytest.raises(la.LAError) as e:
        h.backward_gated(z, z, z, g, g, z)
    assert e.value.code == la.LA_ERR_UNSUPPORTED
    h.close()


def test_backward_gdn_full_size_sampled_heads():
    # The gated delta rule's gradients at the benchmark's full size (B2 H16
    # T8192 d128, bf16: the chunkwise path, every sequence-head on the GPU),
    # with a final-state cotangent; the first and the last sequence-head
    # against the float64 token-by-token oracle (about 1 GB of states each).
    import torch
    from oracle import backward
    w = W.GDN_B2H16_T8192_D128
    inp = W.draw(w, 0)
    q, k, v, g, b = oracle_inputs(inp)
    rng = np.random.default_rng(1)
    do_s = W.round_io(rng.standard_normal((w.B, w.H, w.T, w.dv)), w.io)
    dso = (rng.standard_normal((w.B, w.H, w.dv * w.dk)) * 0.05).astype(np.float32)
    h = la.Handle(w.B, w.H, w.dk, w.dv, io=w.io)
    dev = h.device
    got = h.backward_gated(to_torch(inp.q, dev), to_torch(inp.k, dev), to_torch(inp.v, dev), to_torch(inp.gate, dev),
                           to_torch(inp.beta, dev), to_torch(do_s, dev), None, torch.from_numpy(dso).to(dev),
                           variant="gdn")
    torch.cuda.synchronize()
    assert h.last_launches() == 4 and h.status() == la.LA_OK
    h.close()
    got = [x.float().cpu().numpy() for x in got]
    do64 = W.as_f64(do_s)
    for bi, hi in ((0, 0), (w.B - 1, w.H - 1)):
        sl = lambda a: a[bi:bi + 1, hi:hi + 1]
        ref = backward.delta_backward(sl(q), sl(k), sl(v), sl(g), sl(b), sl(do64), None, sl(dso))
        for name, x, r in zip(NAMES, got, ref):
            e = slice_rel_err(sl(x), r)
            assert np.all(np.isfinite(sl(x))), name
            assert e <= TOL["bf16"], (bi, hi, name, e)


def test_backward_gdn_more_chain_ctas_than_sms():
    # 80 sequence-heads: 2 directions x 80 x 2 = 320 chunk-chain CTAs, more than
    # the GPU has SMs, so the chains run in several waves (no chain waits on
    # another CTA), and 240 per-chunk CTAs of each per-chunk kernel.
    got, ref = _case("gdn", 4, 20, 130, 64, "bf16", seed=41)
    for name, x, r in zip(NAMES, got, ref):
        assert np.all(np.isfinite(x)), name
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))


@pytest.mark.parametrize("gate_mu,beta_mu", [(-1.0, 2.0), (-3.0, 0.0)])
def test_backward_gdn_strong_gates(gate_mu, beta_mu):
    # Strong decays (g = sigmoid(N(mu, 1)): about 0.27 or 0.05 per token) make
    # the chunk's factors e^{b_r - b_s}, gam and lam tiny, down to fp32
    # underflow across a chunk; beta near 1 makes the UT solve's entries large.
    import torch
    from oracle import backward
    w = W.small(W.GDN_B2H16_T8192_D128, B=1, H=2, T=200, dk=128, dv=128).with_(io="bf16", gate_mu=gate_mu,
                                                                                  beta_mu=beta_mu)
    inp = W.draw(w, 53)
    q, k, v, g, b = oracle_inputs(inp)
    rng = np.random.default_rng(54)
    do_s = W.round_io(rng.standard_normal((w.B, w.H, w.T, w.dv)), "bf16")
    dso = (rng.standard_normal((w.B, w.H, w.dv * w.dk)) * 0.05).astype(np.float32)
    h = la.Handle(w.B, w.H, w.dk, w.dv)
    dev = h.device
    got = h.backward_gated(to_torch(inp.q, dev), to_torch(inp.k, dev), to_torch(inp.v, dev), to_torch(inp.gate, dev),
                           to_torch(inp.beta, dev), to_torch(do_s, dev), None, torch.from_numpy(dso).to(dev),
                           variant="gdn")
    torch.cuda.synchronize()
    assert h.last_launches() == 4
    h.close()
    ref = backward.delta_backward(q, k, v, g, b, W.as_f64(do_s), None, dso)
    for name, x, r in zip(NAMES, [x.float().cpu().numpy() for x in got], ref):
        assert np.all(np.isfinite(x)), name
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))


@pytest.mark.parametrize("variant", ["gdn", "kda", "gla"])
@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
def test_backward_gated_rectangular_heads(variant, dk, dv):
    # d_k != d_v: the token-serial kernel (the chunkwise form takes square heads)
    got, ref = _case(variant, 1, 2, 70, dk, "bf16", seed=61 + dk, dv=dv)
    for name, x, r in zip(names(variant), got, ref):
        assert x.shape == r.shape, name
        assert slice_rel_err(x, r) <= TOL["bf16"], (name, slice_rel_err(x, r))
