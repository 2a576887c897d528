"""Shared helpers of the parity tests: marshal seeded inputs to the GPU path
and to the oracle, and compare the two as the operator's contract states."""
from __future__ import annotations

import numpy as np

import workloads as W

TOL = {"bf16": 2e-2, "fp32": 1e-4}   # max relative error per (b,h) slice


def to_torch(a, device):
    """Stored array -> torch tensor with the same bits (uint16 means bf16)."""
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_torch(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return W.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.double().cpu().numpy()


def slice_rel_err(x: np.ndarray, ref: np.ndarray, lead: int = 2) -> float:
    """max over leading (b,h) slices of max|x - ref| / max|ref|."""
    x = np.asarray(x, np.float64).reshape(int(np.prod(ref.shape[:lead])), -1)
    r = np.asarray(ref, np.float64).reshape(x.shape)
    num = np.max(np.abs(x - r), axis=1)
    den = np.maximum(np.max(np.abs(r), axis=1), 1e-30)
    return float(np.max(num / den))


def oracle_inputs(inp: W.Inputs):
    return (W.as_f64(inp.q), W.as_f64(inp.k), W.as_f64(inp.v),
            None if inp.gate is None else inp.gate.astype(np.float64),
            None if inp.beta is None else inp.beta.astype(np.float64))


def run_gpu_prefill(h, w: W.Workload, inp: W.Inputs, chunk=0, state_in=None, with_den=False):
    """Run la_forward on inputs `inp` (state_in: numpy fp32 or None)."""
    import torch
    dev = h.device
    q, k, v = to_torch(inp.q, dev), to_torch(inp.k, dev), to_torch(inp.v, dev)
    gate, beta = to_torch(inp.gate, dev), to_torch(inp.beta, dev)
    sin = None
    if state_in is not None:
        sin = torch.from_numpy(np.ascontiguousarray(state_in, np.float32)).to(dev).reshape(w.B, w.H, -1)
    den = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev) if with_den else None
    out, sout, den = h.forward(q, k, v, gate, beta, sin, variant=w.variant, chunk=chunk, den_out=den)
    torch.cuda.synchronize()
    return from_torch(out), sout.cpu().numpy().astype(np.float64), (None if den is None else den.cpu().numpy())
