"""Pins of the oracle's projections around the attention (RMSNorm + QKV
projection with RoPE; output projection + residual), against facts fixed
outside the oracle: a hand-worked RMSNorm row, closed forms (constant rows,
scale invariance, one-hot inputs, zero weights, position 0), library
routines in double (torch's rms_norm, numpy's matrix product), and RoPE
written independently as a complex rotation.  Nothing here touches the GPU.
"""
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_golden_rmsnorm_row():
    vals = {}
    for line in open(os.path.join(GOLDEN, "rmsnorm_c2_worked.txt")):
        if line.strip() and not line.startswith("#"):
            name, expr = line.split()
            vals[name] = float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt}))
    got = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), eps=0.0)[0]
    np.testing.assert_allclose(got, [vals["xn0"], vals["xn1"]], rtol=1e-15)


def test_rmsnorm_matches_torch_in_double():
    x, g = _rand((37, 96), 1), _rand(96, 2)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g),
                                       eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, g, eps=1e-5), ref, rtol=1e-13, atol=1e-13)


def test_rmsnorm_closed_forms():
    g = _rand(16, 3)
    # a constant row c: mean(x^2) = c^2, so xn = c / sqrt(c^2 + eps) * g
    for c in (-2.5, 0.75):
        got = oracle.rmsnorm(np.full((1, 16), c), g, eps=1e-3)[0]
        np.testing.assert_allclose(got, c / math.sqrt(c * c + 1e-3) * g, rtol=1e-14)
    # scale invariance without eps
    x = _rand((5, 16), 4)
    np.testing.assert_allclose(oracle.rmsnorm(7.0 * x, g, eps=0.0), oracle.rmsnorm(x, g, eps=0.0),
                               rtol=1e-13)


def test_linear_matches_numpy_and_picks_weight_columns():
    a, w = _rand((9, 24), 5), _rand((40, 24), 6)
    np.testing.assert_allclose(oracle.linear(a, w), a @ w.T, rtol=1e-12, atol=1e-12)
    onehot = np.zeros((1, 24))
    onehot[0, 7] = 1.0
    np.testing.assert_array_equal(oracle.linear(onehot, w)[0], w[:, 7])


def _rope_complex(x, positions, base):
    """RoPE as a complex rotation (rotate-half pairing): z_i = x_i + i x_{i+D/2}
    turned by exp(i m theta_i); written independently of the oracle."""
    D = x.shape[-1]
    half = D // 2
    theta = base ** (-(2.0 * np.arange(half)) / D)
    z = x[..., :half] + 1j * x[..., half:]
    z = z * np.exp(1j * np.outer(positions, theta))
    return np.concatenate([z.real, z.imag], axis=-1)


def test_qkv_rope_against_an_independent_composition():
    B, T, H, D = 2, 5, 3, 8
    C = H * D
    x, g, w = _rand((B * T, C), 7), _rand(C, 8), _rand((3 * C, C), 9, 0.2)
    q, k, v = oracle.qkv_rope(x, g, w, B, T, H, D, base=500.0, eps=1e-5)
    xn = torch.nn.functional.rms_norm(torch.from_numpy(x), (C,), torch.from_numpy(g),
                                      eps=1e-5).numpy()
    y = xn @ w.T
    pos = np.tile(np.arange(T), B)
    for h in range(H):
        cols = slice(h * D, (h + 1) * D)
        np.testing.assert_allclose(q[:, cols], _rope_complex(y[:, cols], pos, 500.0), atol=1e-12)
        np.testing.assert_allclose(k[:, cols],
                                   _rope_complex(y[:, C + h * D:C + (h + 1) * D], pos, 500.0),
                                   atol=1e-12)
    np.testing.assert_allclose(v, y[:, 2 * C:], atol=1e-12)
    # position 0 of each sequence is not rotated
    for b in range(B):
        np.testing.assert_allclose(q[b * T], y[b * T, :C], atol=1e-13)
        np.testing.assert_allclose(k[b * T], y[b * T, C:2 * C], atol=1e-13)


def test_qkv_rope_preserves_per_head_norms():
    B, T, H, D = 1, 9, 2, 16
    C = H * D
    x, g, w = _rand((T, C), 10), _rand(C, 11), _rand((3 * C, C), 12, 0.3)
    q, k, _ = oracle.qkv_rope(x, g, w, B, T, H, D)
    y = oracle.linear(oracle.rmsnorm(x, g), w)
    for h in range(H):
        cols = slice(h * D, (h + 1) * D)
        np.testing.assert_allclose(np.linalg.norm(q[:, cols], axis=1),
                                   np.linalg.norm(y[:, cols], axis=1), rtol=1e-13)


def test_out_proj_residual_closed_forms():
    N, C = 6, 20
    o, w, r = _rand((N, C), 13), _rand((C, C), 14), _rand((N, C), 15)
    np.testing.assert_array_equal(oracle.out_proj_residual(o, np.zeros((C, C)), r), r)
    np.testing.assert_allclose(oracle.out_proj_residual(o, w, r), r + o @ w.T, rtol=1e-12,
                               atol=1e-12)
    onehot = np.zeros((1, C))
    onehot[0, 3] = 1.0
    np.testing.assert_allclose(oracle.out_proj_residual(onehot, w, r[:1])[0], r[0] + w[:, 3],
                               rtol=1e-15)
