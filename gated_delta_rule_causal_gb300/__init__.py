"""GB300 (sm_103a) causal linear attention with a fixed matrix state.

Thin ctypes binding over the C ABI in ``include/la.h``. Every step of the
operator runs in the CUDA library built from ``csrc/``. This module only
marshals arguments: torch supplies device memory and streams. There is no
fallback. If the library has not been built, or no GB300 is present, the
calls raise.

Low level (same names as the C ABI): ``la_create``, ``la_forward``, ``la_forward_host``,
``la_decode_step``, ``la_status``, ``la_destroy``, ``la_last_error``,
``la_last_launches``, ``la_version``, ``la_forward_noalloc``, ``la_noalloc_status``. Convenience: ``Handle`` takes torch
tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB as LIB_PATH, build  # noqa: F401  (build() compiles in-tree)

LA_NORM_ELU1, LA_GLA, LA_GDN, LA_NORM_DECAY, LA_KDA = 0, 1, 2, 3, 4
LA_BF16, LA_FP32 = 0, 1
LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_MISALIGNED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(6)
LA_FLAG_IDENTITY_PHI = 0x1
LA_FLAG_SEQUENTIAL_CHUNKS = 0x2
LA_FLAG_TEST_TIMEOUT = 0x100

VARIANTS = {"norm": LA_NORM_ELU1, "gla": LA_GLA, "gdn": LA_GDN, "norm_decay": LA_NORM_DECAY, "kda": LA_KDA}
ERRORS = {1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_MISALIGNED",
          4: "LA_ERR_CUDA", 5: "LA_ERR_TIMEOUT"}


class la_config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("io", ctypes.c_int), ("flags", ctypes.c_uint), ("device", ctypes.c_int)]


class LAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is missing: build it with "
                    "gated_delta_rule_causal_gb300.build() (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            vp, fp, i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            L.la_create.argtypes = [ctypes.POINTER(la_config), ctypes.POINTER(ctypes.c_void_p)]
            L.la_create.restype = i
            L.la_forward.argtypes = [vp, vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, i, vp]
            L.la_forward.restype = i
            L.la_forward_host.argtypes = [vp, vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, i, vp]
            L.la_forward_host.restype = i
            L.la_decode_step.argtypes = [vp, vp, vp, vp, fp, fp, fp, vp, fp, fp, i, vp]
            L.la_backward.restype = i
            L.la_backward.argtypes = [vp, vp, vp, vp, fp, vp, fp, vp, vp, vp, fp, i, i, vp]
            L.la_backward_gated.restype = i
            L.la_backward_gated.argtypes = [vp, vp, vp, vp, fp, fp, fp, vp, fp, vp, vp, vp, fp, fp, fp, i, i, vp]
            L.la_decode_step.restype = i
            L.la_status.argtypes = [vp, vp]
            L.la_status.restype = i
            L.la_destroy.argtypes = [vp]
            L.la_destroy.restype = None
            L.la_last_error.argtypes = [vp]
            L.la_last_error.restype = ctypes.c_char_p
            L.la_last_launches.argtypes = [vp]
            L.la_last_launches.restype = i
            L.la_version.argtypes = []
            L.la_version.restype = i
            L.la_forward_noalloc.argtypes = [ctypes.POINTER(la_config), vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, vp]
            L.la_forward_noalloc.restype = i
            L.la_noalloc_status.argtypes = [i, vp]
            L.la_noalloc_status.restype = i
            _lib = L
    return _lib


# ------------------------------------------------------------------ raw ABI

def la_version() -> int:
    return lib().la_version()


def la_create(B, H, d_k, d_v, io=LA_BF16, flags=0, device=0) -> tuple[int, ctypes.c_void_p]:
    h = ctypes.c_void_p()
    cfg = la_config(B, H, d_k, d_v, io, flags, device)
    rc = lib().la_create(ctypes.byref(cfg), ctypes.byref(h))
    return rc, h


def la_forward(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T, chunk, stream) -> int:
    return lib().la_forward(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T, chunk, stream)


def la_forward_host(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T, chunk, stream) -> int:
    """la_forward with every tensor in (page-locked) host memory (see la.h)."""
    return lib().la_forward_host(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, T, chunk, stream)


def la_decode_step(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, stream) -> int:
    return lib().la_decode_step(h, q, k, v, gate, beta, state_in, out, state_out, den_out, variant, stream)


def la_forward_noalloc(cfg: la_config, q, k, v, gate, beta, state_in, out, state_out, den_out,
                       variant, T, stream) -> int:
    """Prefill without any device allocation by the library (see la.h)."""
    return lib().la_forward_noalloc(ctypes.byref(cfg), q, k, v, gate, beta, state_in, out, state_out,
                                    den_out, variant, T, stream)


def la_noalloc_status(device: int, stream) -> int:
    """Read and clear the status word of la_forward_noalloc calls on `device` (see la.h)."""
    return lib().la_noalloc_status(device, stream)


def la_status(h, stream) -> int:
    return lib().la_status(h, stream)


def la_destroy(h) -> None:
    lib().la_destroy(h)


def la_last_error(h) -> str:
    s = lib().la_last_error(h)
    return s.decode() if s else ""


def la_last_launches(h) -> int:
    return lib().la_last_launches(h)


# ------------------------------------------------------------------ torch marshalling

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def state_size(variant: str, d_k: int, d_v: int) -> int:
    """fp32 elements of one sequence-head's state (norm and norm_decay append z)."""
    return d_k * d_v + (d_k if variant in ("norm", "norm_decay") else 0)


class Handle:
    """One configured operator instance (B, H, d_k, d_v, io dtype, device)."""

    def __init__(self, B, H, d_k, d_v, io="bf16", flags=0, device=None):
        import torch
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.B, self.H, self.d_k, self.d_v = B, H, d_k, d_v
        self.io = io
        self.dtype = torch.bfloat16 if io == "bf16" else torch.float32
        self.device = dev
        rc, h = la_create(B, H, d_k, d_v, LA_BF16 if io == "bf16" else LA_FP32, flags, dev.index)
        if rc != LA_OK:
            raise LAError(rc, "la_create failed")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            la_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != LA_OK:
            raise LAError(rc, la_last_error(self._h))

    def _expect(self, name, t, shape, dtype):
        import torch
        if t is None:
            return
        if not isinstance(t, torch.Tensor) or t.device != self.device or t.dtype != dtype:
            raise ValueError(f"{name}: expected a {dtype} tensor on {self.device}")
        if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous shape {tuple(shape)}, got {tuple(t.shape)}")

    def forward(self, q, k, v, gate=None, beta=None, state_in=None, *, variant="gdn", chunk=0,
                out=None, state_out=None, den_out=None, return_state=True, stream=None):
        """Prefill: q,k [B,H,T,d_k], v [B,H,T,d_v]. Returns (out, state_out, den_out)."""
        import torch
        var = VARIANTS[variant]
        B, H, T = q.shape[0], q.shape[1], q.shape[2]
        if (B, H) != (self.B, self.H):
            raise ValueError("q batch/heads differ from the handle's")
        self._expect("q", q, (B, H, T, self.d_k), self.dtype)
        self._expect("k", k, (B, H, T, self.d_k), self.dtype)
        self._expect("v", v, (B, H, T, self.d_v), self.dtype)
        if var == LA_GLA:
            self._expect("gate", gate, (B, H, T, self.d_k), torch.float32)
        elif var == LA_KDA:
            self._expect("gate", gate, (B, H, T, self.d_k), torch.float32)
            self._expect("beta", beta, (B, H, T), torch.float32)
        elif var == LA_NORM_DECAY:
            self._expect("gate", gate, (B, H), torch.float32)
        elif var == LA_GDN:
            self._expect("gate", gate, (B, H, T), torch.float32)
            self._expect("beta", beta, (B, H, T), torch.float32)
        ss = state_size(variant, self.d_k, self.d_v)
        self._expect("state_in", state_in, (B, H, ss), torch.float32)
        if out is None:
            out = torch.empty((B, H, T, self.d_v), dtype=self.dtype, device=self.device)
        if state_out is None and return_state:
            state_out = torch.empty((B, H, ss), dtype=torch.float32, device=self.device)
        rc = la_forward(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(state_in),
                        _ptr(out), _ptr(state_out), _ptr(den_out), var, T, chunk, _stream_ptr(stream))
        self._check(rc)
        return out, state_out, den_out

    def forward_host(self, q, k, v, gate=None, beta=None, state_in=None, *, variant="gdn", chunk=0,
                     out=None, state_out=None, den_out=None, return_state=True, stream=None):
        """Prefill from pinned host tensors (CPU, ``pin_memory()``); the outputs
        are pinned host tensors too. The copies overlap the kernels inside the
        library. Returns (out, state_out, den_out), complete once ``stream``
        (default: the current stream) reaches the end of the call."""
        import torch
        var = VARIANTS[variant]
        B, H, T = q.shape[0], q.shape[1], q.shape[2]
        if (B, H) != (self.B, self.H):
            raise ValueError("q batch/heads differ from the handle's")
        cpu = torch.device("cpu")

        def chk(name, t, shape, dtype):
            if t is None:
                return
            if not isinstance(t, torch.Tensor) or t.device != cpu or t.dtype != dtype:
                raise ValueError(f"{name}: expected a {dtype} host tensor")
            if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
                raise ValueError(f"{name}: expected contiguous shape {tuple(shape)}, got {tuple(t.shape)}")

        chk("q", q, (B, H, T, self.d_k), self.dtype)
        chk("k", k, (B, H, T, self.d_k), self.dtype)
        chk("v", v, (B, H, T, self.d_v), self.dtype)
        if var == LA_GLA:
            chk("gate", gate, (B, H, T, self.d_k), torch.float32)
        elif var == LA_KDA:
            chk("gate", gate, (B, H, T, self.d_k), torch.float32)
            chk("beta", beta, (B, H, T), torch.float32)
        elif var == LA_NORM_DECAY:
            chk("gate", gate, (B, H), torch.float32)
        elif var == LA_GDN:
            chk("gate", gate, (B, H, T), torch.float32)
            chk("beta", beta, (B, H, T), torch.float32)
        ss = state_size(variant, self.d_k, self.d_v)
        chk("state_in", state_in, (B, H, ss), torch.float32)
        if out is None:
            out = torch.empty((B, H, T, self.d_v), dtype=self.dtype).pin_memory()
        if state_out is None and return_state:
            state_out = torch.empty((B, H, ss), dtype=torch.float32).pin_memory()
        chk("out", out, (B, H, T, self.d_v), self.dtype)
        chk("state_out", state_out, (B, H, ss), torch.float32)
        rc = la_forward_host(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(state_in),
                             _ptr(out), _ptr(state_out), _ptr(den_out), var, T, chunk, _stream_ptr(stream))
        self._check(rc)
        return out, state_out, den_out

    def decode_step(self, q, k, v, gate=None, beta=None, state_in=None, *, variant="gdn",
                    out=None, state_out=None, den_out=None, stream=None):
        """One token: q,k [B,H,d_k], v [B,H,d_v]; state_out may be state_in (in place)."""
        import torch
        var = VARIANTS[variant]
        B, H = self.B, self.H
        self._expect("q", q, (B, H, self.d_k), self.dtype)
        self._expect("k", k, (B, H, self.d_k), self.dtype)
        self._expect("v", v, (B, H, self.d_v), self.dtype)
        ss = state_size(variant, self.d_k, self.d_v)
        if out is None:
            out = torch.empty((B, H, self.d_v), dtype=self.dtype, device=self.device)
        if state_out is None:
            state_out = torch.empty((B, H, ss), dtype=torch.float32, device=self.device)
        rc = la_decode_step(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(state_in),
                            _ptr(out), _ptr(state_out), _ptr(den_out), var, _stream_ptr(stream))
        self._check(rc)
        return out, state_out, den_out

    def backward(self, q, k, v, dout, state_in=None, dstate_out=None, *, variant="norm",
                 dq=None, dk=None, dv=None, dstate_in=None, return_dstate=True, stream=None):
        """Gradients of a normalized prefill: q,k [B,H,T,d_k], v and dout
        [B,H,T,d_v]; dstate_out optional. Returns (dq, dk, dv, dstate_in)."""
        import torch
        var = VARIANTS[variant]
        B, H, T = q.shape[0], q.shape[1], q.shape[2]
        if (B, H) != (self.B, self.H):
            raise ValueError("q batch/heads differ from the handle's")
        for name, t, d in (("q", q, self.d_k), ("k", k, self.d_k), ("v", v, self.d_v), ("dout", dout, self.d_v)):
            self._expect(name, t, (B, H, T, d), self.dtype)
        ss = state_size(variant, self.d_k, self.d_v)
        self._expect("state_in", state_in, (B, H, ss), torch.float32)
        self._expect("dstate_out", dstate_out, (B, H, ss), torch.float32)
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        if dstate_in is None and return_dstate:
            dstate_in = torch.empty((B, H, ss), dtype=torch.float32, device=self.device)
        rc = lib().la_backward(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(state_in), _ptr(dout), _ptr(dstate_out),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dstate_in), var, T, _stream_ptr(stream))
        self._check(rc)
        return dq, dk, dv, dstate_in

    def backward_gated(self, q, k, v, gate, beta, dout, state_in=None, dstate_out=None, *, variant="gdn",
                       return_dstate=True, stream=None):
        """Gradients of a gated delta rule prefill (variant "gdn": gate
        [B,H,T]; "kda": gate [B,H,T,d_k]; beta [B,H,T]), of a per-channel
        gated one ("gla": gate [B,H,T,d_k]) or of a normalized one with a fixed
        decay ("norm_decay": gate [B,H]); the last two take no beta. Returns
        (dq, dk, dv, dgate, dbeta, dstate_in); dbeta is None without beta."""
        import torch
        var = VARIANTS[variant]
        B, H, T = q.shape[0], q.shape[1], q.shape[2]
        if (B, H) != (self.B, self.H):
            raise ValueError("q batch/heads differ from the handle's")
        for name, t, d in (("q", q, self.d_k), ("k", k, self.d_k), ("v", v, self.d_v), ("dout", dout, self.d_v)):
            self._expect(name, t, (B, H, T, d), self.dtype)
        gshape = ((B, H, T, self.d_k) if variant in ("kda", "gla") else (B, H) if variant == "norm_decay"
                  else (B, H, T))
        self._expect("gate", gate, gshape, torch.float32)
        if variant in ("gla", "norm_decay"):
            beta = None
        self._expect("beta", beta, (B, H, T), torch.float32)
        ss = state_size(variant, self.d_k, self.d_v)
        self._expect("state_in", state_in, (B, H, ss), torch.float32)
        self._expect("dstate_out", dstate_out, (B, H, ss), torch.float32)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dgate = torch.empty_like(gate)
        dbeta = None if beta is None else torch.empty_like(beta)
        dstate_in = torch.empty((B, H, ss), dtype=torch.float32, device=self.device) if return_dstate else None
        rc = lib().la_backward_gated(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta), _ptr(state_in),
                                     _ptr(dout), _ptr(dstate_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgate),
                                     _ptr(dbeta), _ptr(dstate_in), var, T, _stream_ptr(stream))
        self._check(rc)
        return dq, dk, dv, dgate, dbeta, dstate_in

    def last_launches(self) -> int:
        """Kernels the last forward / decode_step call enqueued."""
        return la_last_launches(self._h)

    def status(self, stream=None) -> int:
        """Synchronize the stream and return (and clear) the device status."""
        return la_status(self._h, _stream_ptr(stream))
