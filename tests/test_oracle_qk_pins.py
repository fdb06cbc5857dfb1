"""Pins for the oracle's RMSNorm and rotary embedding (the q/k path).

RMSNorm and rotary position embeddings are two of the forward pass's
mechanisms ("Make the Engine Talk", 1.3).  Pinned by hand-derived values
(tests/golden/hand_worked.json), closed forms, and, for RoPE, an independent
formulation as complex multiplication.
"""
import json
import math
import os

import numpy as np
import pytest

from paged_kv_gqa_06_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_rmsnorm_hand_worked(oracle_mod):
    c = json.load(open(GOLDEN))["rmsnorm_cases"][0]
    y = oracle_mod.rmsnorm(_bits([c["x"]]), _bits(c["w"]), c["eps"])
    np.testing.assert_allclose(y[0], np.array(c["expected_over_sqrt2"]) * math.sqrt(2), rtol=0, atol=1e-15)


def test_rmsnorm_closed_forms(oracle_mod):
    x = _bits(np.full((3, 64), [[0.5], [-2.0], [8.0]]))
    y = oracle_mod.rmsnorm(x, None, 0.0)
    np.testing.assert_allclose(y, np.sign(W.bf16_bits_to_f32(x)), rtol=0, atol=1e-15)   # constant rows -> +-1
    eps = 1e-6
    y = oracle_mod.rmsnorm(x, None, eps)
    c = W.bf16_bits_to_f32(x)[:, :1].astype(np.float64)
    np.testing.assert_allclose(y, np.broadcast_to(c / np.sqrt(c * c + eps), y.shape), rtol=0, atol=1e-15)
    r = np.random.default_rng(1).standard_normal((5, 128)).astype(np.float32)
    w = _bits(np.random.default_rng(2).standard_normal(128))
    a = oracle_mod.rmsnorm(_bits(r), w, 0.0)
    b = oracle_mod.rmsnorm(_bits(4 * r), w, 0.0)         # exact power-of-two scaling drops out
    np.testing.assert_allclose(a, b, rtol=1e-15, atol=0)
    ms = np.mean(oracle_mod.rmsnorm(_bits(r), None, 0.0) ** 2, axis=1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-14)       # unit mean square


def test_rope_hand_worked(oracle_mod):
    c = json.load(open(GOLDEN))["rope_cases"][0]
    y = oracle_mod.rope(np.array([c["x"]], dtype=np.float64), [c["pos"]], c["theta"])
    want = [math.cos(1), -math.sin(0.01), math.sin(1), math.cos(0.01)]
    np.testing.assert_allclose(y[0], want, rtol=0, atol=1e-15)


def _rope_complex(x, pos, theta):
    """The same rotation as complex multiplication of z_i = x_i + j x_{i+D/2}."""
    D = x.shape[-1]
    h = D // 2
    z = x[..., :h] + 1j * x[..., h:]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * np.arange(h) / D)
    z = z * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("D", [2, 64, 128])
def test_rope_equals_complex_rotation(oracle_mod, D):
    rng = np.random.default_rng(D)
    x = rng.standard_normal((6, D))
    pos = np.array([0, 1, 7, 1000, 16383, 131071])
    y = oracle_mod.rope(x, pos, 1e6)
    np.testing.assert_allclose(y, _rope_complex(x, pos, 1e6), rtol=0, atol=1e-9)
    assert np.array_equal(y[0], x[0])                                        # position 0: identity
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_depends_only_on_relative_position(oracle_mod):
    rng = np.random.default_rng(9)
    q, k = rng.standard_normal((2, 128))
    for m, n, t in [(5, 2, 10), (100, 99, 1000), (7, 7, 40000)]:
        a = oracle_mod.rope(q[None], [m], 1e6)[0] @ oracle_mod.rope(k[None], [n], 1e6)[0]
        b = oracle_mod.rope(q[None], [m + t], 1e6)[0] @ oracle_mod.rope(k[None], [n + t], 1e6)[0]
        assert abs(a - b) < 1e-9


def test_bf16_round_is_nearest_even(oracle_mod):
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 1e-3, 3.14159, -0.1, 65280.0, 65408.0])
    got = oracle_mod.bf16_round(x)
    import torch
    ref = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
