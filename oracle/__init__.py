"""Float64 CPU oracle for the causal linear-attention operator.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
and its Python binding never import it, and it imports nothing from them.

``run`` calls the plain C recurrences in ``la_oracle.c`` (token by token,
double precision). ``forms`` holds the independent algebraic forms that the
pages state are equal to the recurrence (masked-parallel, literal, unrolled).
The tests use them to pin the C recurrences.

Arrays use the operator's layouts: q,k [B,H,T,dk]; v [B,H,T,dv]; gla gate
[B,H,T,dk]; gdn gate/beta [B,H,T]; norm_decay gate [B,H] (one decay per
sequence-head); kda gate [B,H,T,dk] (per-channel decay) and beta [B,H,T];
state per (b,h): norm and norm_decay S[dk,dv] then z[dk]; gla S[dk,dv];
gdn and kda S[dv,dk].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile la_oracle.c with gcc (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # LA_ORACLE_LIB points the pin tests at a deliberately mutated
            # build of la_oracle.c (tests/test_oracle_mutations.py).
            lib = ctypes.CDLL(os.environ.get("LA_ORACLE_LIB") or build())
            P = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.la_oracle_norm.argtypes = [i, i, i, i, P, P, P, P, P, P, P, i]
            lib.la_oracle_norm_decay.argtypes = [i, i, i, i, P, P, P, P, P, P, P, P, i]
            lib.la_oracle_gla.argtypes = [i, i, i, i, P, P, P, P, P, P, P, i, i]
            lib.la_oracle_gdn.argtypes = [i, i, i, i, P, P, P, P, P, P, P, P, i]
            lib.la_oracle_kda.argtypes = [i, i, i, i, P, P, P, P, P, P, P, P, i]
            for f in (lib.la_oracle_norm, lib.la_oracle_norm_decay, lib.la_oracle_gla, lib.la_oracle_gdn,
                      lib.la_oracle_kda):
                f.restype = ctypes.c_int
            lib.la_oracle_threads_available.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads_available() -> int:
    return int(_load().la_oracle_threads_available())


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


@dataclass
class Result:
    o: np.ndarray            # [B,H,T,dv]
    state: np.ndarray        # [B,H,*] flat per-(b,h) state (see module doc)
    den: np.ndarray | None   # norm, norm_decay: [B,H,T] denominators phi(q)^T z


def state_size(variant: str, dk: int, dv: int) -> int:
    return dk * dv + (dk if variant in ("norm", "norm_decay") else 0)


def run(variant: str, q, k, v, gate=None, beta=None, state_in=None,
        identity_phi: bool = False, nthreads: int = 0) -> Result:
    """Run the float64 recurrence. q,k,v: [B,H,T,d] float arrays."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    BH = B * H
    ss = state_size(variant, dk, dv)
    sin = None if state_in is None else _f64(np.reshape(state_in, (BH, ss)))
    o = np.empty((B, H, T, dv), dtype=np.float64)
    sout = np.empty((B, H, ss), dtype=np.float64)
    den = None
    if variant == "norm":
        den = np.empty((B, H, T), dtype=np.float64)
        rc = lib.la_oracle_norm(BH, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(sin),
                                _ptr(o), _ptr(sout), _ptr(den), nthreads)
        if rc == 2:
            raise FloatingPointError("normalizer denominator not positive")
    elif variant == "norm_decay":
        gm = _f64(gate)
        assert gm.shape == (B, H)
        den = np.empty((B, H, T), dtype=np.float64)
        rc = lib.la_oracle_norm_decay(BH, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(gm), _ptr(sin),
                                      _ptr(o), _ptr(sout), _ptr(den), nthreads)
        if rc == 2:
            raise FloatingPointError("normalizer denominator not positive")
    elif variant == "gla":
        gm = _f64(gate)
        assert gm.shape == (B, H, T, dk)
        rc = lib.la_oracle_gla(BH, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(gm), _ptr(sin),
                               _ptr(o), _ptr(sout), int(identity_phi), nthreads)
    elif variant == "gdn":
        g, b = _f64(gate), _f64(beta)
        assert g.shape == (B, H, T) and b.shape == (B, H, T)
        rc = lib.la_oracle_gdn(BH, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                               _ptr(sin), _ptr(o), _ptr(sout), nthreads)
    elif variant == "kda":
        a, b = _f64(gate), _f64(beta)
        assert a.shape == (B, H, T, dk) and b.shape == (B, H, T)
        rc = lib.la_oracle_kda(BH, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                               _ptr(sin), _ptr(o), _ptr(sout), nthreads)
    else:
        raise ValueError(variant)
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return Result(o=o, state=sout, den=den)


def split_norm_state(state: np.ndarray, dk: int, dv: int):
    """(S [...,dk,dv], z [...,dk]) views of a flat norm state."""
    lead = state.shape[:-1]
    S = state[..., : dk * dv].reshape(lead + (dk, dv))
    z = state[..., dk * dv:]
    return S, z
