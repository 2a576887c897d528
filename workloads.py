"""Seeded synthetic inputs for the causal linear-attention operator.

This module draws and rounds inputs. It holds none of the operator's arithmetic.
The oracle (``oracle/``) and the CUDA path both consume what it returns, so it
imports neither of them.

Recipe (shared by tests, ``bench.py`` and ``__graft_entry__.smoke``):

* ``numpy.random.Generator(PCG64(SeedSequence(seed)))``, default seed 0.
* Arrays are drawn in float64 in a fixed order: q, k, v, gate, beta. Keys of
  the gated delta rule are L2-normalized per token in float64. This is an
  input precondition ("keys have length 1", Transformers & Math module 18,
  section 18.2). The operator itself never normalizes them.
* Each array is then rounded once, to nearest-even, to its storage type:
  q/k/v/out to the I/O dtype (bf16 or fp32), gates and beta to fp32, and the
  initial state to fp32. bf16 rounding goes float64 -> float32 -> bf16, both
  steps to nearest-even.
* Decode workloads draw the initial state from ``SeedSequence([seed])`` and
  step ``s`` from ``SeedSequence([seed, 1 + s])``, so any single step can be
  regenerated on its own.

bf16 values are carried as ``uint16`` bit patterns, because numpy has no bf16
type. ``as_f64`` turns any stored array back into the exact float64 values
that both sides consume.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

VARIANTS = ("norm", "gla", "gdn")


# --------------------------------------------------------------------------
# rounding helpers
# --------------------------------------------------------------------------

def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 (via float32, both round-to-nearest-even)."""
    f32 = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 values of a stored array (uint16 means bf16 bits)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


def round_io(x: np.ndarray, io: str) -> np.ndarray:
    if io == "bf16":
        return f64_to_bf16_bits(x)
    if io == "fp32":
        return x.astype(np.float32)
    raise ValueError(f"unknown io dtype {io!r}")


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtypes and value distributions."""
    name: str
    variant: str          # norm | gla | gdn | norm_decay | kda
    B: int
    H: int
    T: int                # tokens per sequence (1 for one decode step)
    dk: int
    dv: int
    io: str               # bf16 | fp32
    qkv_scale: float = 1.0        # q,k,v ~ N(0,1) * qkv_scale
    unit_keys: bool = False       # L2-normalize k per token (gated delta rule)
    gate_mu: float = 0.0          # gate = sigmoid(N(gate_mu, 1))
    beta_mu: float = 0.0          # beta = sigmoid(N(beta_mu, 1))
    state_std: float = 0.0        # initial state ~ N(0, state_std); 0 means S_0 = 0
    decode_steps: int = 0         # >0: a decode workload with this many steps
    chunk: int = 64
    note: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five workloads of the operator's specification, by what they are.
NORM_T64_D16 = Workload(
    "norm_b1h1_t64_d16_fp32", "norm", 1, 1, 64, 16, 16, "fp32",
    note="normalized elu+1, q,k,v iid N(0,1), S_0=z_0=0; correctness case")
NORM_B4H8_T2048_D64 = Workload(
    "norm_b4h8_t2048_d64_bf16", "norm", 4, 8, 2048, 64, 64, "bf16", qkv_scale=0.5,
    note="normalized elu+1, bf16 q,k,v iid N(0,1)*0.5, fp32 state and normalizer")
GLA_B4H16_T4096_D128 = Workload(
    "gla_b4h16_t4096_d128_bf16", "gla", 4, 16, 4096, 128, 128, "bf16",
    qkv_scale=1.0 / math.sqrt(128.0), gate_mu=3.0,
    note="per-channel gate gamma=sigmoid(N(3,1)) fp32, bf16 q,k,v N(0,1)/sqrt(128)")
NORM_DECAY_B4H8_T2048_D64 = Workload(
    "norm_decay_b4h8_t2048_d64_bf16", "norm_decay", 4, 8, 2048, 64, 64, "bf16", qkv_scale=0.5, gate_mu=4.0,
    note="normalized elu+1 with a fixed decay per head gamma=sigmoid(N(4,1)), bf16 q,k,v N(0,1)*0.5")
KDA_DECODE_N256H16_D128 = Workload(
    "kda_decode_n256h16_d128_s256", "kda", 256, 16, 1, 128, 128, "bf16",
    unit_keys=True, gate_mu=4.0, beta_mu=0.0, state_std=0.02, decode_steps=256,
    note="delta rule with a per-channel decay, decode: alpha=sigmoid(N(4,1)) per channel, 256 steps")
GDN_B2H16_T8192_D128 = Workload(
    "gdn_b2h16_t8192_d128_bf16", "gdn", 2, 16, 8192, 128, 128, "bf16",
    unit_keys=True, gate_mu=4.0, beta_mu=0.0,
    note="gated delta rule, bf16 q,v N(0,1), unit k, beta=sigmoid(N(0,1)), g=sigmoid(N(4,1))")
KDA_B2H16_T8192_D128 = Workload(
    "kda_b2h16_t8192_d128_bf16", "kda", 2, 16, 8192, 128, 128, "bf16",
    unit_keys=True, gate_mu=4.0, beta_mu=0.0,
    note="delta rule with a per-channel decay, prefill: the gated delta shapes, alpha=sigmoid(N(4,1)) per channel")
GDN_DECODE_N256H16_D128 = Workload(
    "gdn_decode_n256h16_d128_s1024", "gdn", 256, 16, 1, 128, 128, "bf16",
    unit_keys=True, gate_mu=4.0, beta_mu=0.0, state_std=0.02, decode_steps=1024,
    note="gated delta decode: fp32 state N(0,0.02), 1024 single-token steps")

ALL = (NORM_T64_D16, NORM_B4H8_T2048_D64, GLA_B4H16_T4096_D128,
       GDN_B2H16_T8192_D128, GDN_DECODE_N256H16_D128)
# Beyond the five: the normalized variant with a fixed decay per head, on
# the shapes of the normalized headline workload; the delta rule with a
# per-channel decay, prefill on the gated delta shapes and decode.
EXTRA = (NORM_DECAY_B4H8_T2048_D64, KDA_B2H16_T8192_D128, KDA_DECODE_N256H16_D128)
BY_NAME = {w.name: w for w in ALL + EXTRA}


# --------------------------------------------------------------------------
# drawing
# --------------------------------------------------------------------------

@dataclass
class Inputs:
    """Stored (rounded) inputs of one call. Arrays are C-contiguous."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    gate: np.ndarray | None   # norm: None; gla, kda: [B,H,T,dk]; gdn: [B,H,T]; norm_decay: [B,H]
    beta: np.ndarray | None   # gdn: [B,H,T]; else None
    state: np.ndarray | None  # fp32 initial state or None (zeros)


def _draw_qkvgb(rng: np.random.Generator, w: Workload, lead: tuple) -> tuple:
    q = rng.standard_normal(lead + (w.dk,)) * w.qkv_scale
    k = rng.standard_normal(lead + (w.dk,)) * w.qkv_scale
    v = rng.standard_normal(lead + (w.dv,)) * w.qkv_scale
    if w.unit_keys:
        k = _unit_rows(k)
    gate = beta = None
    if w.variant == "gla":
        gate = _sigmoid(rng.standard_normal(lead + (w.dk,)) + w.gate_mu)
    elif w.variant == "gdn":
        gate = _sigmoid(rng.standard_normal(lead) + w.gate_mu)
        beta = _sigmoid(rng.standard_normal(lead) + w.beta_mu)
    elif w.variant == "norm_decay":   # one fixed decay per sequence-head
        gate = _sigmoid(rng.standard_normal(lead[:2]) + w.gate_mu)
    elif w.variant == "kda":          # per-channel decay of the delta rule
        gate = _sigmoid(rng.standard_normal(lead + (w.dk,)) + w.gate_mu)
        beta = _sigmoid(rng.standard_normal(lead) + w.beta_mu)
    return q, k, v, gate, beta


def state_shape(w: Workload) -> tuple:
    """Flat fp32 state of one call: S (+ z for norm, norm_decay) per (b,h)."""
    if w.variant in ("norm", "norm_decay"):
        return (w.B * w.H * (w.dk * w.dv + w.dk),)
    return (w.B * w.H * w.dk * w.dv,)


def _draw_state(rng: np.random.Generator, w: Workload) -> np.ndarray | None:
    if w.state_std <= 0.0:
        return None
    s = rng.standard_normal(state_shape(w)) * w.state_std
    return s.astype(np.float32)


def draw(w: Workload, seed: int = 0) -> Inputs:
    """Inputs of a prefill call, [B,H,T,*] layout."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    q, k, v, gate, beta = _draw_qkvgb(rng, w, (w.B, w.H, w.T))
    state = _draw_state(rng, w)
    return Inputs(
        q=round_io(q, w.io), k=round_io(k, w.io), v=round_io(v, w.io),
        gate=None if gate is None else gate.astype(np.float32),
        beta=None if beta is None else beta.astype(np.float32),
        state=state)


def draw_decode_state(w: Workload, seed: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed])))
    s = rng.standard_normal(state_shape(w)) * w.state_std
    return s.astype(np.float32)


def draw_decode_step(w: Workload, step: int, seed: int = 0) -> Inputs:
    """Inputs of decode step ``step``: q,k,v [B,H,d], gate/beta [B,H]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1 + step])))
    q, k, v, gate, beta = _draw_qkvgb(rng, w, (w.B, w.H))
    return Inputs(
        q=round_io(q, w.io), k=round_io(k, w.io), v=round_io(v, w.io),
        gate=None if gate is None else gate.astype(np.float32),
        beta=None if beta is None else beta.astype(np.float32),
        state=None)


def small(w: Workload, **kw) -> Workload:
    """A reduced copy of a workload (same distributions), for fast parity."""
    return w.with_(name=w.name + "_small", **kw)


# --------------------------------------------------------------------------
# associative-recall probe
# --------------------------------------------------------------------------

@dataclass
class Probe:
    """A recall probe as one call's inputs: K writes (a second K writes of new
    values under the same keys when `rewrite`), then K reads, one per key.
    The output at read token `read0 + j` is the recall for key j; `target[j]`
    is the value most recently written under it."""
    inputs: Inputs
    target: np.ndarray    # [K, dv] float64 (exact: one-hot values)
    read0: int
    K: int
    variant: str
    identity_phi: bool


def recall_probe(variant: str, K: int, dk: int, dv: int, keys: str = "random", rewrite: bool = False,
                 io: str = "fp32", seed: int = 0) -> Probe:
    """Store K key-value bindings and read each back through one call.

    * Keys: "random" unit vectors (N(0,1) rows normalized in float64) or
      "orthonormal" ones (K <= dk; columns of a QR factor of a Gaussian).
    * Values: one-hot, v_j = e_j (orthonormal; dv >= K); rewritten values
      are e_{(j+1) mod K}.
    * variant "gla": additive memory (S += k v^T), i.e. the per-channel gated
      form with gate 1 and no feature map; reads carry v = 0, so they write
      nothing. variant "gdn": the delta rule with beta = 1 and g = 1 on
      writes, beta = 0 on reads.
    * q is the key being read on read tokens and 0 elsewhere.
    B = H = 1. Values and keys are rounded to `io` like any other input.
    """
    if variant not in ("gla", "gdn"):
        raise ValueError("the probe runs the additive (gla) or delta (gdn) rule")
    if dv < K:
        raise ValueError("one-hot values need dv >= K")
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    if keys == "random":
        kk = _unit_rows(rng.standard_normal((K, dk)))
    elif keys == "orthonormal":
        if K > dk:
            raise ValueError("at most dk orthonormal keys")
        qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        kk = qm[:, :K].T.copy()
    else:
        raise ValueError(f"unknown key kind {keys!r}")
    eye = np.eye(dv)
    old = eye[:K]
    new = eye[[(j + 1) % K for j in range(K)]]
    nw = 2 * K if rewrite else K
    T = nw + K
    q = np.zeros((T, dk))
    k = np.zeros((T, dk))
    v = np.zeros((T, dv))
    k[:K], v[:K] = kk, old
    if rewrite:
        k[K:2 * K], v[K:2 * K] = kk, new
    q[nw:], k[nw:] = kk, kk
    lead = (1, 1)
    gate = beta = None
    if variant == "gla":
        gate = np.ones(lead + (T, dk), np.float32)
    else:
        gate = np.ones(lead + (T,), np.float32)
        beta = np.zeros(lead + (T,), np.float32)
        beta[..., :nw] = 1.0
    inp = Inputs(q=round_io(q.reshape(lead + (T, dk)), io), k=round_io(k.reshape(lead + (T, dk)), io),
                 v=round_io(v.reshape(lead + (T, dv)), io), gate=gate, beta=beta, state=None)
    return Probe(inputs=inp, target=new if rewrite else old, read0=nw, K=K, variant=variant,
                 identity_phi=(variant == "gla"))
