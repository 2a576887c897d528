"""The seeded generator: determinism, rounding and the stated distributions."""
import numpy as np
import pytest
import torch

import workloads as W


def test_bf16_rounding_matches_torch():
    r = np.random.default_rng(0)
    x = np.concatenate([r.standard_normal(100000) * 10.0 ** r.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 1e-30, 3.0e38])])
    bits = W.f64_to_bf16_bits(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = W.bf16_bits_to_f64(bits)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_draw_is_deterministic_and_seeded():
    w = W.small(W.GDN_B2H16_T8192_D128, B=1, H=2, T=33)
    a, b, c = W.draw(w, 0), W.draw(w, 0), W.draw(w, 1)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.gate, b.gate)
    assert not np.array_equal(a.q, c.q)


def test_gdn_keys_are_unit_and_gates_in_range():
    w = W.small(W.GDN_B2H16_T8192_D128, B=1, H=4, T=256)
    x = W.draw(w, 3)
    n = np.linalg.norm(W.as_f64(x.k), axis=-1)
    assert np.all(np.abs(n - 1.0) < 1e-2)                 # unit before bf16 rounding
    assert x.gate.shape == (1, 4, 256) and x.beta.shape == (1, 4, 256)
    assert np.all((x.gate > 0) & (x.gate < 1)) and np.all((x.beta > 0) & (x.beta < 1))
    assert 0.95 < float(np.mean(x.gate)) < 0.99            # sigmoid(N(4,1))
    assert 0.4 < float(np.mean(x.beta)) < 0.6              # sigmoid(N(0,1))


def test_gla_gate_per_channel_and_scale():
    w = W.small(W.GLA_B4H16_T4096_D128, B=1, H=2, T=128)
    x = W.draw(w, 0)
    assert x.gate.shape == (1, 2, 128, 128) and x.gate.dtype == np.float32
    assert abs(np.std(W.as_f64(x.q)) - 1 / np.sqrt(128)) < 0.01


def test_decode_steps_regenerate_independently():
    w = W.GDN_DECODE_N256H16_D128.with_(B=4)
    s3a = W.draw_decode_step(w, 3, seed=5)
    s3b = W.draw_decode_step(w, 3, seed=5)
    s4 = W.draw_decode_step(w, 4, seed=5)
    assert np.array_equal(s3a.v, s3b.v) and not np.array_equal(s3a.v, s4.v)
    st = W.draw_decode_state(w, seed=5)
    assert st.shape == (4 * 16 * 128 * 128,) and abs(np.std(st) - 0.02) < 1e-3
