"""Decode attention over a KV cache (ne_attn_decode) against the CPU oracle.

A decode of sequence b at position m = pos[b] is row m of the causal
attention of that sequence's first m + 1 tokens, so the oracle evaluates that
one query row (bf16 rotated operands, mode 1, as for the training forward)
over the cached keys and values.  Bars: O max abs error <= 1e-2 (the kernel
writes bf16), LSE abs error <= 1e-3.  Cases: ragged positions including 0 and
the last cache row, the two named decode workloads (every sequence and head),
agreement with the training forward's last row, and a position outside the
cache (reported, never read).  ne_attn_decode_rotated on a cache of rotated
keys (rotated by the oracle's mode-1 rule, the bf16 values the kernels
multiply) gives bit for bit the results of ne_attn_decode on the un-rotated
cache, and meets the oracle's bars."""
import numpy as np
import pytest
import torch

import oracle
from causal_self_attention_gb300.inputs import make_custom, make_decode
from parity import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _oracle_decode(inp, heads=None):
    """(o [B, H, D], lse [B, H]) of the oracle for every sequence (and the
    given heads, default all)."""
    B, H, D = inp["B"], inp["H"], inp["D"]
    heads = range(H) if heads is None else heads
    o = np.full((B, H, D), np.nan)
    lse = np.full((B, H), np.nan)
    for b in range(B):
        L = int(inp["pos"][b]) + 1
        q = torch.zeros((L, H, D), dtype=torch.bfloat16)
        q[L - 1] = inp["q"][b]
        k = inp["k_cache"][b, :L]
        v = inp["v_cache"][b, :L]
        res = oracle.attention_sampled(q, k, v, None, [0, L], [(0, h, [L - 1], []) for h in heads],
                                       base=inp["rope_base"], scale=inp["scale"], mode=1)
        for h, r in zip(heads, res):
            o[b, h] = r["o"][0]
            lse[b, h] = r["lse"][0]
    return o, lse


def _run(na, inp):
    q, kc, vc, pos = (inp[n].cuda() for n in ("q", "k_cache", "v_cache", "pos"))
    out, lse = na.ne_attn_decode(q, kc, vc, pos, inp["rope_base"], inp["scale"])
    assert na.ne_attn_get_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(na, inp, heads=None):
    out, lse = _run(na, inp)
    ro, rl = _oracle_decode(inp, heads)
    sel = np.isfinite(rl)
    o_err = float(np.max(np.abs(out[sel] - ro[sel])))
    l_err = float(np.max(np.abs(lse[sel] - rl[sel])))
    print(f"\n[decode] {inp['name']} B{inp['B']} H{inp['H']} Tmax{inp['Tmax']}: "
          f"o_max_abs={o_err:.3e} lse_max_abs={l_err:.3e}")
    assert o_err <= O_TOL and l_err <= LSE_TOL, (o_err, l_err)


def test_decode_ragged_positions(na):
    _check(na, make_decode(B=5, H=3, Tmax=600, positions=[0, 1, 255, 256, 599], seed=5))


@pytest.mark.parametrize("name", ["decode1k", "decode16k"])
def test_decode_named_workloads(na, name):
    _check(na, make_decode(name))


def test_decode_is_the_training_forward_last_row(na):
    inp = make_custom(2, 1000, 3, seed=17)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o32, lse = na.ne_attn_fwd(q, k, v, out_f32=True)
    pos = torch.full((2,), 999, dtype=torch.int32, device="cuda")
    od, ld = na.ne_attn_decode(q[:, 999].contiguous(), k, v, pos)
    assert na.ne_attn_get_device_status() == 0
    assert torch.allclose(od.float(), o32[:, 999], atol=1e-2, rtol=0)
    assert torch.allclose(ld, lse[:, :, 999], atol=1e-4, rtol=0)


def test_decode_position_outside_the_cache_is_reported(na):
    inp = make_decode(B=2, H=2, Tmax=64, positions=[10, 64], seed=9)
    q, kc, vc, pos = (inp[n].cuda() for n in ("q", "k_cache", "v_cache", "pos"))
    out, lse = na.ne_attn_decode(q, kc, vc, pos)
    assert na.ne_attn_get_device_status() == 7  # NE_ERR_BAD_SEQLEN
    assert torch.all(out[1] == 0) and torch.all(torch.isinf(lse[1]))
    ro, rl = _oracle_decode(dict(inp, B=1, pos=inp["pos"][:1]))
    assert np.max(np.abs(out[0].float().cpu().numpy() - ro[0])) <= O_TOL


def _rotate_cache(kc):
    """Oracle mode-1 rotation of a cache ``[B, Tmax, H, 64]``: row n at
    position n."""
    B, _, H, _ = kc.shape
    out = np.empty(kc.shape, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            out[b, :, h] = oracle.rope(kc[b, :, h].double().numpy(), base=10000.0, mode=1)
    return torch.from_numpy(out).to(torch.bfloat16)


def _rotate_queries(q, pos):
    """Oracle mode-1 rotation of ``q`` ``[B, H, 64]``, row b at position pos[b]."""
    B, H, D = q.shape
    out = np.empty((B, H, D))
    for b in range(B):
        m = int(pos[b])
        x = np.zeros((m + 1, D))
        for h in range(H):
            x[m] = q[b, h].double().numpy()
            out[b, h] = oracle.rope(x, base=10000.0, mode=1)[m]
    return torch.from_numpy(out).to(torch.bfloat16)


@pytest.mark.parametrize("case", ["ragged", "decode1k", "decode16k"])
def test_rotated_cache_decode_equals_the_rotating_one(na, case):
    inp = (make_decode(B=5, H=3, Tmax=600, positions=[0, 1, 255, 256, 599], seed=21)
           if case == "ragged" else make_decode(case))
    q, kc, vc, pos = (inp[n].cuda() for n in ("q", "k_cache", "v_cache", "pos"))
    qr = _rotate_queries(inp["q"], inp["pos"]).cuda()
    krc = _rotate_cache(inp["k_cache"]).cuda()
    o1, l1 = na.ne_attn_decode(q, kc, vc, pos, inp["rope_base"], inp["scale"])
    o2, l2 = na.ne_attn_decode_rotated(qr, krc, vc, pos, inp["scale"])
    assert na.ne_attn_get_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    if case == "ragged":
        ro, rl = _oracle_decode(inp)
        assert np.max(np.abs(o2.float().cpu().numpy() - ro)) <= O_TOL
        assert np.max(np.abs(l2.cpu().numpy() - rl)) <= LSE_TOL


def test_rotated_cache_decode_reports_a_position_outside_the_cache(na):
    inp = make_decode(B=2, H=2, Tmax=64, positions=[10, 64], seed=23)
    qr, kc, vc, pos = (inp[n].cuda() for n in ("q", "k_cache", "v_cache", "pos"))
    out, lse = na.ne_attn_decode_rotated(qr, kc, vc, pos)
    assert na.ne_attn_get_device_status() == 7  # NE_ERR_BAD_SEQLEN
    assert torch.all(out[1] == 0) and torch.all(torch.isinf(lse[1]))
