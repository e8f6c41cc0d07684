"""Parity of the projections around the attention (RMSNorm + QKV projection
with RoPE in the epilogue; output projection + residual) with the CPU oracle.

Tolerance: the kernel rounds x_norm to bf16 before the projection and the
outputs to bf16 after it (each a relative rounding of at most 2^-9), and
accumulates in fp32, so against the double-precision oracle the relative L2
error of each output is of the order of 2^-9; the bar is 1e-2.  rstd is fp32
(relative error bar 1e-5).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _inputs(B, T, H, seed):
    g = torch.Generator().manual_seed(seed)
    C = H * 64
    x = torch.randn((B * T, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((C,), generator=g) * 0.1 + 1.0).to(torch.bfloat16)
    wq = (torch.randn((3 * C, C), generator=g) / C ** 0.5).to(torch.bfloat16)
    return x, w, wq


@pytest.mark.parametrize("B,T,H", [(2, 200, 4), (1, 130, 8)])
def test_rmsnorm_qkv_rope_small_full(na, B, T, H):
    x, g, w = _inputs(B, T, H, 3 + T)
    q, k, v, xn, rstd = na.ne_rmsnorm_qkv_rope(x.cuda(), g.cuda(), w.cuda(), T)
    assert na.ne_attn_get_device_status() == 0
    C = H * 64
    rq, rk, rv = oracle.qkv_rope(x, g, w, B, T, H, 64, base=10000.0, eps=1e-5)
    rxn = oracle.rmsnorm(x, g, eps=1e-5)
    errs = {n: rel_l2(a.reshape(B * T, C).double().cpu().numpy(), b)
            for n, a, b in (("q", q, rq), ("k", k, rk), ("v", v, rv), ("x_norm", xn, rxn))}
    xd = x.double().numpy()
    rr = 1.0 / np.sqrt((xd * xd).mean(axis=1) + 1e-5)
    errs["rstd"] = float(np.max(np.abs(rstd.double().cpu().numpy() - rr) / rr))
    print("\n[proj] qkv", B, T, H, ", ".join(f"{n}={e:.2e}" for n, e in errs.items()))
    assert errs["rstd"] <= 1e-5, errs
    assert all(e <= TOL for n, e in errs.items() if n != "rstd"), errs


def test_rmsnorm_qkv_rope_gpt2s_sequences(na):
    """GPT-2-small shape (B=8, T=1024, C=768): two whole sequences against the oracle."""
    B, T, H = 8, 1024, 12
    x, g, w = _inputs(B, T, H, 11)
    q, k, v, _, _ = na.ne_rmsnorm_qkv_rope(x.cuda(), g.cuda(), w.cuda(), T)
    assert na.ne_attn_get_device_status() == 0
    C = H * 64
    for b in (0, B - 1):
        rows = slice(b * T, (b + 1) * T)
        rq, rk, rv = oracle.qkv_rope(x[rows], g, w, 1, T, H, 64)
        for n, a, r in (("q", q, rq), ("k", k, rk), ("v", v, rv)):
            err = rel_l2(a[b].reshape(T, C).double().cpu().numpy(), r)
            assert err <= TOL, (b, n, err)


@pytest.mark.parametrize("N,C", [(300, 256), (8192, 768)])
def test_out_proj_residual(na, N, C):
    g = torch.Generator().manual_seed(N + C)
    o = torch.randn((N, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((C, C), generator=g) / C ** 0.5).to(torch.bfloat16)
    r = torch.randn((N, C), generator=g).to(torch.bfloat16)
    y = na.ne_out_proj_residual(o.cuda(), w.cuda(), r.cuda())
    assert na.ne_attn_get_device_status() == 0
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(0).integers(0, N, 128)]))
    ref = oracle.out_proj_residual(o[rows], w, r[rows])
    err = rel_l2(y[rows].double().cpu().numpy(), ref)
    print(f"\n[proj] out_proj N={N} C={C} rel_l2={err:.2e}")
    assert err <= TOL, err


def test_zero_weight_gives_the_residual_bitwise(na):
    N, C = 256, 512
    r = torch.randn((N, C)).to(torch.bfloat16).cuda()
    o = torch.randn((N, C)).to(torch.bfloat16).cuda()
    y = na.ne_out_proj_residual(o, torch.zeros((C, C), dtype=torch.bfloat16).cuda(), r)
    assert torch.equal(y, r)
