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


def _rotate_bf16(x, T, H):
    """The bf16 operands RoPE produces in the attention kernels (oracle mode 1),
    per head, positions 0..T-1 in each sequence: [B, T, H, 64] bf16."""
    B = x.shape[0]
    out = np.empty(tuple(x.shape))
    for b in range(B):
        for h in range(H):
            out[b, :, h] = oracle.rope(x[b, :, h].double().numpy(), base=10000.0, mode=1)
    return torch.from_numpy(out).to(torch.bfloat16)


def test_rotated_attention_matches_the_rotating_one(na):
    """ne_attn_fwd_rotated on q', k' = the bf16 rotations gives bitwise the O,
    LSE of ne_attn_fwd on q, k; ne_attn_bwd_rotated gives dv bitwise and dq',
    dk' whose un-rotation matches the oracle's dq, dk."""
    from causal_self_attention_gb300.inputs import make_custom
    from parity import GRAD_TOL, packed_view
    inp = make_custom(2, 300, 3, seed=61)
    B, T, H = 2, 300, 3
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    qr, kr = _rotate_bf16(inp["q"], T, H).cuda(), _rotate_bf16(inp["k"], T, H).cuda()
    o, lse = na.ne_attn_fwd(q, k, v)
    o2, lse2 = na.ne_attn_fwd_rotated(qr, kr, v)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    dq, dk, dv = na.ne_attn_bwd(q, k, v, o, do, lse)
    dqr, dkr, dv2 = na.ne_attn_bwd_rotated(qr, kr, v, o2, do, lse2)
    assert na.ne_attn_get_device_status() == 0
    assert torch.equal(dv, dv2)
    (cq, ck, cv, cdo), cu = packed_view(inp)
    ref = oracle.attention(cq, ck, cv, cdo, cu, base=10000.0, scale=inp["scale"], mode=0)
    for name, g in (("dq", dqr), ("dk", dkr)):
        gr = g.double().cpu().numpy()
        back = np.empty_like(gr)
        for b in range(B):
            for h in range(H):
                back[b, :, h] = oracle.rope_transpose(gr[b, :, h], base=10000.0)
        err = rel_l2(back.reshape(B * T, H, 64), ref[name])
        assert err <= GRAD_TOL, (name, err)


def test_attention_block_chain(na):
    """RMSNorm + QKV + RoPE -> attention on q', k' -> output projection +
    residual, against the oracle's composition of the same steps (one layer's
    attention block, as the pages' transformer layer runs it)."""
    B, T, H = 1, 256, 4
    C = H * 64
    x, g, w = _inputs(B, T, H, 71)
    gen = torch.Generator().manual_seed(72)
    wo = (torch.randn((C, C), generator=gen) / C ** 0.5).to(torch.bfloat16)
    q, k, v, _, _ = na.ne_rmsnorm_qkv_rope(x.cuda(), g.cuda(), w.cuda(), T)
    o, _ = na.ne_attn_fwd_rotated(q, k, v)
    y = na.ne_out_proj_residual(o.reshape(B * T, C), wo.cuda(), x.cuda())
    assert na.ne_attn_get_device_status() == 0
    rq, rk, rv = oracle.qkv_rope(x, g, w, B, T, H, 64)
    # attention on the (double) rotated operands: base irrelevant at mode 0 with
    # rotation already applied -- express it as attention with RoPE undone:
    # the oracle's attention takes un-rotated q, k, so un-rotate q', k' first.
    uq = np.stack([oracle.rope_transpose(rq[:, h * 64:(h + 1) * 64]) for h in range(H)], axis=1)
    uk = np.stack([oracle.rope_transpose(rk[:, h * 64:(h + 1) * 64]) for h in range(H)], axis=1)
    att = oracle.attention(uq, uk, rv.reshape(T, H, 64), None, [0, T], base=10000.0,
                           scale=0.125, mode=0)
    ref = oracle.out_proj_residual(att["o"].reshape(T, C), wo, x)
    err = rel_l2(y.double().cpu().numpy(), ref)
    print(f"\n[proj] attention block chain rel_l2={err:.2e}")
    assert err <= TOL, err
