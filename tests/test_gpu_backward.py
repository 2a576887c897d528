"""Gradients of the normalized prefill (la_backward) against the float64
oracle's (oracle/backward.py, itself pinned by finite differences of the
forward oracle), on the same seeded inputs. bf16 io with d_k = d_v = 64 takes
the chunkwise tensor-core backward (five launches); other heads of 64 or 128
the forward and then the row-split token-serial kernel; smaller heads the
one-CTA-per-head kernel (one launch)."""
import numpy as np
import pytest

import workloads as W
from _helpers import TOL, oracle_inputs, slice_rel_err, to_torch

pytestmark = pytest.mark.gpu

la = pytest.importorskip("gated_delta_rule_causal_gb300")


def _case(B, H, T, dk, dv, io, seed, with_state, with_dstate):
    import torch
    from oracle import backward
    w = W.small(W.NORM_B4H8_T2048_D64, B=B, H=H, T=T, dk=dk, dv=dv).with_(io=io)
    inp = W.draw(w, seed)
    q, k, v, _, _ = oracle_inputs(inp)
    rng = np.random.default_rng(seed + 1000)
    ss = dk * dv + dk
    # the gradient of the outputs, rounded to the io dtype as the GPU reads it
    do_s = W.round_io(rng.standard_normal((B, H, T, dv)), io)
    do64 = W.as_f64(do_s)
    sin = dso = None
    if with_state:
        sin = (rng.standard_normal((B, H, ss)) * 0.1).astype(np.float32)
        sin[..., dk * dv:] = np.abs(sin[..., dk * dv:]) * 50 + 1.0
    if with_dstate:
        dso = (rng.standard_normal((B, H, ss)) * 0.01).astype(np.float32)
    h = la.Handle(B, H, dk, dv, io=io)
    dev = h.device
    tq, tk, tv = to_torch(inp.q, dev), to_torch(inp.k, dev), to_torch(inp.v, dev)
    gsin = None if sin is None else torch.from_numpy(sin).to(dev)
    gdso = None if dso is None else torch.from_numpy(dso).to(dev)
    dq, dk_, dv_, dsin = h.backward(tq, tk, tv, to_torch(do_s, dev), gsin, gdso)
    torch.cuda.synchronize()
    chunked = io == "bf16" and dk == 64 and dv == 64
    rows = not chunked and dk in (64, 128) and dv in (64, 128)
    n = h.last_launches()
    # chunkwise: one five-launch chain per group of sequence-heads whose
    # per-chunk states fit the handle's workspace; heads of 64 or 128 outside
    # it: the forward's launches, then the row kernel and its conversion;
    # smaller heads: one CUDA-core kernel
    if chunked:
        assert n >= 5 and n % 5 == 0, n
    elif rows:
        assert n >= 3, n
    else:
        assert n == 1, n
    assert h.status() == la.LA_OK
    h.close()
    rq, rk, rv, rs = backward.norm_backward(q, k, v, do64, sin, dso)
    got = [x.float().cpu().numpy() for x in (dq, dk_, dv_, dsin)]
    return got, (rq, rk, rv, rs)


@pytest.mark.parametrize("dk,dv", [(64, 64), (32, 32), (16, 64), (64, 16), (128, 128), (64, 128)])
@pytest.mark.parametrize("io", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 37, 200])
def test_backward_parity(dk, dv, io, T):
    got, ref = _case(1, 2, T, dk, dv, io, seed=T + dk, with_state=True, with_dstate=True)
    for name, g, r in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert np.all(np.isfinite(g)), name
        assert slice_rel_err(g, r) <= TOL[io], (name, slice_rel_err(g, r))


@pytest.mark.parametrize("with_state,with_dstate", [(False, False), (True, False), (False, True)])
def test_backward_optional_states(with_state, with_dstate):
    got, ref = _case(2, 3, 65, 64, 64, "bf16", seed=5, with_state=with_state, with_dstate=with_dstate)
    for name, g, r in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert slice_rel_err(g, r) <= TOL["bf16"], (name, slice_rel_err(g, r))


@pytest.mark.parametrize("io", ["bf16", "fp32"])
def test_backward_long_sequence(io):
    # 2048 tokens: 32 chunks carried by the chunkwise form (bf16), or 128
    # checkpointed segments of the row kernel (fp32); each meets its io
    # dtype's bound
    got, ref = _case(1, 2, 2048, 64, 64, io, seed=7, with_state=False, with_dstate=True)
    for name, g, r in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert slice_rel_err(g, r) <= TOL[io], (name, slice_rel_err(g, r))


def test_backward_workload_shape():
    # the normalized workload's shapes, B4 H8 T2048 d64, every head (their
    # per-chunk states exceed the handle's workspace: two head groups)
    got, ref = _case(4, 8, 2048, 64, 64, "bf16", seed=11, with_state=True, with_dstate=True)
    for name, g, r in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert np.all(np.isfinite(g)), name
        assert slice_rel_err(g, r) <= TOL["bf16"], (name, slice_rel_err(g, r))


def test_backward_rejects_what_it_does_not_cover():
    import torch
    # a head of 16 keys and 128 values: neither both in {16, 32, 64} nor both in {64, 128}
    h = la.Handle(1, 1, 16, 128)
    xk = torch.zeros((1, 1, 4, 16), dtype=torch.bfloat16, device=h.device)
    xv = torch.zeros((1, 1, 4, 128), dtype=torch.bfloat16, device=h.device)
    with pytest.raises(la.LAError) as e:
        h.backward(xk, xk, xv, xv)
    assert e.value.code == la.LA_ERR_UNSUPPORTED
    h.close()
    h = la.Handle(1, 1, 64, 64)
    x = torch.zeros((1, 1, 4, 64), dtype=torch.bfloat16, device=h.device)
    with pytest.raises(la.LAError):
        h.backward(x, x, x, x, variant="gla")
    h.close()
