"""Associative recall through the operator: a fixed-size state as a memory.

K key-value bindings are written, then each key is read back in the same call
(workloads.recall_probe). The pages measure this with the additive rule and
contrast it with the delta rule:

* "Linear attention and Hyena" §11.6: with K random unit keys and orthonormal
  values the mean retrieval error (1/K) sum_j |v^_j - v_j| grows like
  sqrt(K/d_k), printed as 1.99 (K=64, d_k=16), 0.98 (K=64, d_k=64) and 2.81
  (K=128, d_k=16); with K <= d_k orthonormal keys recall is exact.
* "Beyond attention" §18.2 and Figure 18.2: writing a new value under a key
  already used, the additive rule returns old and new piled together, the
  delta rule exactly the new one.

CPU tests pin the oracle to these statements and to the closed form of the
additive crosstalk; GPU tests run the same probes through la_forward.
"""
import numpy as np
import pytest

import oracle
import workloads as W

PRINTED = [(16, 64, 1.99), (64, 64, 0.98), (16, 128, 2.81)]


def oracle_recall(p: W.Probe) -> np.ndarray:
    x = p.inputs
    r = oracle.run(p.variant, W.as_f64(x.q), W.as_f64(x.k), W.as_f64(x.v), x.gate, x.beta,
                   identity_phi=p.identity_phi)
    return r.o[0, 0, p.read0:p.read0 + p.K]


def mean_error(recall: np.ndarray, target: np.ndarray) -> float:
    return float(np.mean(np.linalg.norm(recall - target, axis=1)))


# ------------------------------------------------------------------ oracle pins

@pytest.mark.parametrize("dk,K,printed", PRINTED)
def test_additive_recall_error_grows_like_sqrt_k_over_dk(dk, K, printed):
    p = W.recall_probe("gla", K, dk, K, keys="random", io="fp32", seed=dk * 1000 + K)
    rec = oracle_recall(p)
    # Closed form of the crosstalk with one-hot values: the recall of key j is
    # v_j + sum_{i != j} (k_i . k_j) v_i, so its error is the norm of the
    # off-diagonal column j of the key Gram matrix.
    kk = W.as_f64(p.inputs.k)[0, 0, :K]
    gram = kk @ kk.T
    off = gram - np.diag(np.diag(gram))
    err_closed = np.linalg.norm(off, axis=0)
    assert np.max(np.abs(np.linalg.norm(rec - p.target, axis=1) - err_closed)) <= 1e-12
    # E[(k_i . k_j)^2] = 1/d_k for independent random unit keys, so the error
    # is about sqrt((K-1)/d_k); the pages' printed values agree with it.
    e = mean_error(rec, p.target)
    assert abs(e - np.sqrt((K - 1) / dk)) <= 0.1 * np.sqrt((K - 1) / dk)
    assert abs(e - printed) <= 0.1 * printed


@pytest.mark.parametrize("variant", ["gla", "gdn"])
@pytest.mark.parametrize("dk", [16, 64])
def test_below_capacity_recall_is_exact(variant, dk):
    p = W.recall_probe(variant, dk, dk, dk, keys="orthonormal", io="fp32", seed=dk)
    assert mean_error(oracle_recall(p), p.target) <= 1e-6   # keys rounded to fp32


def test_rewrite_delta_recalls_new_additive_recalls_both():
    pd = W.recall_probe("gdn", 16, 16, 16, keys="orthonormal", rewrite=True, io="fp32", seed=3)
    pa = W.recall_probe("gla", 16, 16, 16, keys="orthonormal", rewrite=True, io="fp32", seed=3)
    old = np.eye(16)
    assert mean_error(oracle_recall(pd), pd.target) <= 1e-6
    assert mean_error(oracle_recall(pa), pa.target + old) <= 1e-6


def test_delta_overwrite_disturbs_overlapping_keys_only():
    # Figure 18.2: keys a, b perpendicular, c overlapping a; after a new value
    # under a the delta rule recalls it exactly for a, keeps b, and disturbs c.
    a, b = np.array([1.0, 0, 0, 0]), np.array([0, 1.0, 0, 0])
    c = np.array([0.6, 0, 0.8, 0])
    va, vb, vc, va2 = np.eye(4)
    k = np.array([a, b, c, a, a, b, c])
    v = np.array([va, vb, vc, va2, 0 * va, 0 * va, 0 * va])
    beta = np.array([1, 1, 1, 1, 0, 0, 0], np.float64)
    q = np.array([0 * a, 0 * a, 0 * a, 0 * a, a, b, c])
    r = oracle.run("gdn", q[None, None], k[None, None], v[None, None], np.ones((1, 1, 7)), beta[None, None])
    o = r.o[0, 0]
    assert np.max(np.abs(o[4] - va2)) <= 1e-12          # a: exactly the new value
    assert np.max(np.abs(o[5] - vb)) <= 1e-12           # b: untouched (perpendicular)
    assert np.linalg.norm(o[6] - vc) > 0.1              # c: disturbed by the rewrite of a


# ------------------------------------------------------------------ GPU, through la_forward

@pytest.mark.gpu
@pytest.mark.parametrize("dk,K,io,chunk", [(16, 64, "fp32", 1), (64, 64, "bf16", 64), (64, 64, "bf16", 1)])
def test_gpu_additive_probe(dk, K, io, chunk):
    torch = pytest.importorskip("torch")
    import gated_delta_rule_causal_gb300 as la
    from _helpers import run_gpu_prefill, slice_rel_err

    la.build()
    p = W.recall_probe("gla", K, dk, K, keys="random", io=io, seed=dk * 1000 + K)
    w = W.Workload("recall_probe", "gla", 1, 1, p.inputs.q.shape[2], dk, K, io)
    h = la.Handle(1, 1, dk, K, io=w.io, flags=la.LA_FLAG_IDENTITY_PHI)
    o, _, _ = run_gpu_prefill(h, w, p.inputs, chunk)
    h.close()
    rec = o[0, 0, p.read0:p.read0 + K]
    ref = oracle_recall(p)
    tol = 1e-4 if io == "fp32" else 2e-2
    assert slice_rel_err(rec[None, None], ref[None, None]) <= tol
    e = mean_error(rec, p.target)
    assert abs(e - np.sqrt((K - 1) / dk)) <= 0.1 * np.sqrt((K - 1) / dk)


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["gla", "gdn"])
@pytest.mark.parametrize("chunk", [64, 1])
def test_gpu_below_capacity_and_rewrite(variant, chunk):
    torch = pytest.importorskip("torch")
    import gated_delta_rule_causal_gb300 as la
    from _helpers import run_gpu_prefill

    la.build()
    d = 64
    flags = la.LA_FLAG_IDENTITY_PHI if variant == "gla" else 0
    for rewrite in (False, True):
        p = W.recall_probe(variant, d, d, d, keys="orthonormal", rewrite=rewrite, io="bf16", seed=7)
        w = W.Workload("recall_probe", variant, 1, 1, p.inputs.q.shape[2], d, d, "bf16")
        h = la.Handle(1, 1, d, d, io="bf16", flags=flags)
        o, _, _ = run_gpu_prefill(h, w, p.inputs, chunk)
        h.close()
        rec = o[0, 0, p.read0:p.read0 + d]
        want = p.target + (np.eye(d) if (rewrite and variant == "gla") else 0.0)
        # bf16 keys are orthonormal to about 4e-3, so the recall is exact to
        # that order: far below the O(1) errors of the other cases.
        assert mean_error(rec, want) <= 0.05
