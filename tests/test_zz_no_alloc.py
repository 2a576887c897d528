"""la_forward_noalloc: the prefill for callers that cannot let a library
allocate device memory (a host framework that owns the GPU's memory, or a
loop that must not allocate after start-up). It must give what la_forward
gives, call after call, while its scratch lives in a static device array.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest

import oracle
import workloads as W
from _helpers import TOL, from_torch, oracle_inputs, slice_rel_err, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import gated_delta_rule_causal_gb300 as la  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    la.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_both(w, seed, gate_for_norm=False):
    x = W.draw(w, seed)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (to_torch(a, dev) for a in (x.q, x.k, x.v))
    g, b = to_torch(x.gate, dev), to_torch(x.beta, dev)
    if gate_for_norm:
        # a stray gate pointer with the undecayed variant must be ignored, as la_forward ignores it
        g = torch.full((w.B, w.H), 0.5, device=dev)
    var = la.VARIANTS[w.variant]
    ss = la.state_size(w.variant, w.dk, w.dv)
    sin = torch.randn((w.B, w.H, ss), device=dev) * 0.1
    if w.variant == "norm":
        sin[..., w.dk * w.dv:] = sin[..., w.dk * w.dv:].abs() * 50 + 1.0

    h = la.Handle(w.B, w.H, w.dk, w.dv)
    den_ref = torch.empty((w.B, w.H, w.T), device=dev) if w.variant == "norm" else None
    o_ref, s_ref, _ = h.forward(q, k, v, g, b, sin, variant=w.variant, chunk=64, den_out=den_ref)

    o = torch.empty_like(o_ref)
    s = torch.empty_like(s_ref)
    den = torch.empty_like(den_ref) if den_ref is not None else None
    cfg = la.la_config(w.B, w.H, w.dk, w.dv, la.LA_BF16, 0, dev.index)
    P = lambda t: None if t is None else t.data_ptr()
    rc = la.la_forward_noalloc(cfg, P(q), P(k), P(v), P(g), P(b), P(sin), P(o), P(s), P(den), var, w.T,
                               la._stream_ptr(None))
    assert rc == la.LA_OK
    assert la.la_noalloc_status(dev.index, la._stream_ptr(None)) == la.LA_OK
    torch.cuda.synchronize()
    h.close()
    return (from_torch(o), s.cpu().numpy(), None if den is None else den.cpu().numpy(),
            from_torch(o_ref), s_ref.cpu().numpy(), None if den_ref is None else den_ref.cpu().numpy())


def _rel(x, r):
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-30))


@pytest.mark.parametrize("variant,d", [("norm", 128), ("norm", 64), ("gla", 128), ("gdn", 128)])
def test_noalloc_matches_la_forward_twice(variant, d):
    # B*H = 2 with 16 chunks: norm (d = 128) and gla split into segments, so
    # their summaries go through the static scratch; norm at d = 64 runs the
    # single cluster launch; two calls in a row with different data must both
    # match la_forward.
    base = {"norm": W.NORM_B4H8_T2048_D64, "gla": W.GLA_B4H16_T4096_D128, "gdn": W.GDN_B2H16_T8192_D128}[variant]
    w = W.small(base, B=1, H=2, T=1000, dk=d, dv=d)
    for seed in (1, 2):
        o, s, den, o_ref, s_ref, den_ref = _run_both(w, seed)
        assert _rel(o, o_ref) <= TOL["bf16"]
        assert _rel(s, s_ref) <= TOL["bf16"]
        if den is not None:
            assert float(np.max(np.abs(den - den_ref) / den_ref)) <= TOL["bf16"]


def test_noalloc_gdn_shallow_ring_is_bit_identical():
    # 32 sequence-heads of d = 128 leave the 16 MiB static scratch room for a
    # ring of only a few chunks per head, so the prep CTAs wait for ring
    # positions the chain CTAs free; la_forward's ring is 8 chunks deep. The
    # arithmetic of every chunk is the same either way.
    w = W.small(W.GDN_B2H16_T8192_D128, B=2, H=16, T=1000, dk=128, dv=128)
    o, s, _, o_ref, s_ref, _ = _run_both(w, 3)
    assert np.array_equal(o, o_ref)
    assert np.array_equal(s, s_ref)


def test_noalloc_rejects_what_it_cannot_run():
    dev = torch.cuda.current_device()
    x = torch.zeros(16, device="cuda")
    P = x.data_ptr()
    st = la._stream_ptr(None)
    fp32 = la.la_config(1, 1, 64, 64, la.LA_FP32, 0, dev)
    assert la.la_forward_noalloc(fp32, P, P, P, None, None, None, P, None, None, la.LA_NORM_ELU1, 8, st) == la.LA_ERR_UNSUPPORTED
    bf = la.la_config(1, 1, 64, 64, la.LA_BF16, 0, dev)
    assert la.la_forward_noalloc(bf, P, P, P, None, None, None, P, None, None, la.LA_GDN, 8, st) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_noalloc(bf, P + 4, P, P, None, None, None, P, None, None, la.LA_NORM_ELU1, 8, st) == la.LA_ERR_MISALIGNED


def test_noalloc_ignores_a_gate_for_the_undecayed_normalized_variant():
    w = W.small(W.NORM_B4H8_T2048_D64, B=1, H=2, T=1000, dk=128, dv=128)
    o, s, den, o_ref, s_ref, den_ref = _run_both(w, 4, gate_for_norm=True)
    assert _rel(o, o_ref) <= TOL["bf16"]
    assert _rel(s, s_ref) <= TOL["bf16"]


@pytest.mark.parametrize("variant", ["norm", "gla", "gdn"])
def test_noalloc_matches_the_oracle(variant):
    # One call per variant against the float64 oracle directly, on the same
    # seeded inputs (T with a ragged tail; the norm and gla shapes split
    # into segments whose summaries live in the static scratch).
    base = {"norm": W.NORM_B4H8_T2048_D64, "gla": W.GLA_B4H16_T4096_D128, "gdn": W.GDN_B2H16_T8192_D128}[variant]
    w = W.small(base, B=1, H=2, T=777, dk=128, dv=128)
    x = W.draw(w, 5)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (to_torch(a, dev) for a in (x.q, x.k, x.v))
    g, b = to_torch(x.gate, dev), to_torch(x.beta, dev)
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=torch.bfloat16, device=dev)
    s = torch.empty((w.B, w.H, la.state_size(w.variant, w.dk, w.dv)), device=dev)
    den = torch.empty((w.B, w.H, w.T), device=dev) if variant == "norm" else None
    cfg = la.la_config(w.B, w.H, w.dk, w.dv, la.LA_BF16, 0, dev.index)
    P = lambda t: None if t is None else t.data_ptr()
    st = la._stream_ptr(None)
    assert la.la_forward_noalloc(cfg, P(q), P(k), P(v), P(g), P(b), None, P(o), P(s), P(den),
                                 la.VARIANTS[variant], w.T, st) == la.LA_OK
    assert la.la_noalloc_status(dev.index, st) == la.LA_OK
    ref = oracle.run(w.variant, *oracle_inputs(x))
    assert slice_rel_err(from_torch(o), ref.o) <= TOL["bf16"]
    assert slice_rel_err(s.cpu().numpy(), ref.state) <= TOL["bf16"]
    if den is not None:
        assert float(np.max(np.abs(den.cpu().numpy() - ref.den) / ref.den)) <= TOL["bf16"]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("variant,T", [("gdn", 128), ("norm", 512)])
def test_noalloc_status_reports_an_expired_wait(variant, T):
    # The test hook makes the chunked kernel wait once on a barrier nothing
    # signals; the wait gives up after 1 ms and records it in the status word
    # of the static scratch. la_noalloc_status reports it once, then the word
    # is clear, and the next call computes normally.
    base = {"norm": W.NORM_B4H8_T2048_D64, "gdn": W.GDN_B2H16_T8192_D128}[variant]
    w = W.small(base, B=1, H=2, T=T, dk=64, dv=64)
    x = W.draw(w, 0)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (to_torch(a, dev) for a in (x.q, x.k, x.v))
    g, b = to_torch(x.gate, dev), to_torch(x.beta, dev)
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=torch.bfloat16, device=dev)
    s = torch.empty((w.B, w.H, la.state_size(w.variant, w.dk, w.dv)), device=dev)
    P = lambda t: None if t is None else t.data_ptr()
    st = la._stream_ptr(None)
    hook = la.la_config(w.B, w.H, w.dk, w.dv, la.LA_BF16, la.LA_FLAG_TEST_TIMEOUT, dev.index)
    assert la.la_forward_noalloc(hook, P(q), P(k), P(v), P(g), P(b), None, P(o), P(s), None,
                                 la.VARIANTS[variant], w.T, st) == la.LA_OK
    assert la.la_noalloc_status(dev.index, st) == la.LA_ERR_TIMEOUT
    assert la.la_noalloc_status(dev.index, st) == la.LA_OK      # read once, then cleared
    plain = la.la_config(w.B, w.H, w.dk, w.dv, la.LA_BF16, 0, dev.index)
    assert la.la_forward_noalloc(plain, P(q), P(k), P(v), P(g), P(b), None, P(o), P(s), None,
                                 la.VARIANTS[variant], w.T, st) == la.LA_OK
    assert la.la_noalloc_status(dev.index, st) == la.LA_OK
    ref = oracle.run(w.variant, *oracle_inputs(x))
    assert slice_rel_err(from_torch(o), ref.o) <= TOL["bf16"]
    assert la.la_noalloc_status(dev.index + 1000, st) == la.LA_ERR_INVALID_ARG
