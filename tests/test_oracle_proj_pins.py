"""Pins of the oracle's dense neighbours of the forward (input projection,
gated RMS norm, output projection) against facts other than themselves (CPU
only): exact selections by 0/1 weights, a hand-computed product, torch's
silu, and closed forms of the norm that a per-head / per-token slip breaks."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def test_in_proj_selects_columns_with_unit_weights():
    rng = np.random.default_rng(0)
    T, D = 5, 12
    h = rng.standard_normal((T, D))
    eye = np.eye(D)
    x, z, b, a = oracle.in_proj(h, eye[:6], eye[6:10], eye[10:11], eye[11:12])
    np.testing.assert_array_equal(x, h[:, :6])
    np.testing.assert_array_equal(z, h[:, 6:10])
    np.testing.assert_array_equal(b, h[:, 10:11])
    np.testing.assert_array_equal(a, h[:, 11:12])


def test_in_proj_hand_computed():
    h = np.array([[1.0, 2.0, -1.0]])
    w = np.array([[1.0, 0.0, 2.0], [0.5, -1.0, 3.0]])  # rows are output features
    x, z, b, a = oracle.in_proj(h, w, w[:1], w[1:], w)
    np.testing.assert_array_equal(x, [[-1.0, -4.5]])
    np.testing.assert_array_equal(z, [[-1.0]])
    np.testing.assert_array_equal(b, [[-4.5]])


def test_out_proj_flattens_heads_in_order():
    o = np.arange(2 * 2 * 3, dtype=np.float64).reshape(2, 2, 3)  # [T][Hv][dv]
    w = np.zeros((1, 6))
    w[0, 4] = 1.0  # head 1, channel 1
    y = oracle.out_proj(o, w)
    np.testing.assert_array_equal(y[:, 0], o[:, 1, 1])


def test_gated_rmsnorm_closed_forms():
    rng = np.random.default_rng(1)
    T, H, dv = 3, 2, 8
    # a head of constant value c: o / rms = sign(c) / sqrt(1 + eps / c^2)
    o = np.zeros((T, H, dv))
    o[:, 0, :] = 3.0
    o[:, 1, :] = -0.5
    z = np.full((T, H, dv), 40.0)  # silu(40) = 40 to fp64 precision
    w = np.ones(dv)
    eps = 1e-6
    y = oracle.gated_rmsnorm(o, z, w, eps)
    np.testing.assert_allclose(y[:, 0], 40.0 / np.sqrt(1 + eps / 9.0), rtol=1e-14)
    np.testing.assert_allclose(y[:, 1], -40.0 / np.sqrt(1 + eps / 0.25), rtol=1e-14)
    # a zero gate closes the output
    np.testing.assert_array_equal(oracle.gated_rmsnorm(o, np.zeros_like(z), w, eps), 0.0)
    # each head is normalised on its own: scaling one head leaves the other unchanged
    o2 = rng.standard_normal((T, H, dv))
    z2 = rng.standard_normal((T, H, dv))
    w2 = rng.standard_normal(dv)
    base = oracle.gated_rmsnorm(o2, z2, w2, 0.0)
    o3 = o2.copy()
    o3[:, 1] *= 1000.0
    np.testing.assert_allclose(oracle.gated_rmsnorm(o3, z2, w2, 0.0), base, rtol=1e-12)


def test_gated_rmsnorm_equals_torch_pieces():
    """RMS over the d_v channels of each head, times the weight and torch's silu."""
    rng = np.random.default_rng(2)
    o = rng.standard_normal((4, 3, 16))
    z = rng.standard_normal((4, 3, 16)) * 3
    w = rng.standard_normal(16)
    ot = torch.from_numpy(o)
    ref = ot * torch.rsqrt(ot.pow(2).mean(-1, keepdim=True) + 1e-5) * torch.from_numpy(w)
    ref = ref * F.silu(torch.from_numpy(z))
    np.testing.assert_allclose(oracle.gated_rmsnorm(o, z, w, 1e-5), ref.numpy(), rtol=1e-12,
                               atol=1e-14)


@pytest.mark.parametrize("wrong", ["all_heads", "no_eps"])
def test_planted_norm_mistakes_are_caught(wrong):
    rng = np.random.default_rng(3)
    o = rng.standard_normal((2, 2, 4)) * np.array([1.0, 50.0])[None, :, None]
    z = rng.standard_normal((2, 2, 4))
    w = np.ones(4)
    good = oracle.gated_rmsnorm(o, z, w, 0.5)
    if wrong == "all_heads":
        rs = 1 / np.sqrt(np.mean(o * o, axis=(1, 2), keepdims=True) + 0.5)
    else:
        rs = 1 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    bad = o * rs * w * (z / (1 + np.exp(-z)))
    assert not np.allclose(good, bad, rtol=1e-6)
