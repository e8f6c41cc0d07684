"""The training pair: ne_attn_fwd_train rotates q and k once and hands the
rotated operands q' = R(m) q, k' = R(n) k to ne_attn_bwd_train.

What is checked: q', k' are exactly the bf16 operands RoPE gives under the
forward's fp32 rule (oracle mode 1); O and LSE are bitwise those of
ne_attn_fwd; the backward from q', k' returns the gradients w.r.t. the
un-rotated q, k that ne_attn_bwd returns (dk, dv bitwise; dq to the order of
its fp32 accumulation, relative L2 <= 1e-3, as between two calls of
ne_attn_bwd) and meets the oracle's bar (relative L2 <= 2e-2).  Shapes: a
single row, short ragged sequences (T 63, 129, 300), a case from 2048 positions on (where ne_attn_fwd itself
rotates the keys in a separate pass), the GPT-2-small training shape, and a
packed variable-length batch.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_self_attention_gb300.inputs import make_custom, make_inputs
from parity import GRAD_TOL, packed_view, rel_l2

pytestmark = pytest.mark.gpu
DQ_TOL = 1e-3


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _rotated_rows(x, cu, H):
    """Oracle mode-1 rotation of packed rows ``[N, H, 64]``, positions from 0
    in each sequence: the bf16 values the kernels multiply."""
    xd = x.double().numpy()
    out = np.empty_like(xd)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            if b > a:
                out[a:b, h] = oracle.rope(xd[a:b, h], base=10000.0, mode=1)
    return torch.from_numpy(out).to(torch.bfloat16)


def _same_gradients(got, ref):
    for t in got:
        assert torch.isfinite(t.float()).all()
    assert torch.equal(got[1], ref[1]), "dk"
    assert torch.equal(got[2], ref[2]), "dv"
    err = rel_l2(got[0].double().cpu().numpy(), ref[0].double().cpu().numpy())
    assert err <= DQ_TOL, ("dq", err)
    return err


@pytest.mark.parametrize("case", ["one_row", "t63", "t129", "ragged", "long", "gpt2s"])
def test_training_pair_matches_the_plain_pair(na, case):
    # one_row .. t129: fewer (row, head) pairs than the streamed preprocess
    # has CTAs, chunks of a few pairs, and a last query tile of one row.
    inp = {"one_row": lambda: make_custom(1, 1, 1, seed=88),
           "t63": lambda: make_custom(3, 63, 5, seed=89),
           "t129": lambda: make_custom(1, 129, 2, seed=90),
           "ragged": lambda: make_custom(2, 300, 3, seed=91),
           "long": lambda: make_custom(1, 2300, 2, seed=92),
           "gpt2s": lambda: make_inputs("gpt2s")}[case]()
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    B, T, H, D = q.shape
    o, lse = na.ne_attn_fwd(q, k, v)
    o2, lse2, qr, kr = na.ne_attn_fwd_train(q, k, v)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    (cq, ck, _, _), cu = packed_view(inp)
    if case != "gpt2s":  # the rotation itself, against the oracle, bit for bit
        assert torch.equal(qr.cpu().reshape(-1, H, D), _rotated_rows(cq, cu, H))
        assert torch.equal(kr.cpu().reshape(-1, H, D), _rotated_rows(ck, cu, H))
    ref = na.ne_attn_bwd(q, k, v, o, do, lse)
    got = na.ne_attn_bwd_train(qr, kr, v, o2, do, lse2)
    assert na.ne_attn_get_device_status() == 0
    err = _same_gradients(got, ref)
    print(f"\n[train] {case}: O, LSE, dk, dv bitwise equal; dq rel L2 {err:.1e}")


def test_training_pair_meets_the_oracle_bar(na):
    inp = make_custom(2, 300, 3, seed=93)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    H, D = inp["H"], inp["D"]
    o, lse, qr, kr = na.ne_attn_fwd_train(q, k, v)
    dq, dk, dv = na.ne_attn_bwd_train(qr, kr, v, o, do, lse)
    assert na.ne_attn_get_device_status() == 0
    (cq, ck, cv, cdo), cu = packed_view(inp)
    ref = oracle.attention(cq, ck, cv, cdo, cu, base=inp["rope_base"], scale=inp["scale"], mode=0)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = rel_l2(t.reshape(-1, H, D).double().cpu().numpy(), ref[name])
        assert err <= GRAD_TOL, (name, err)


def test_varlen_training_pair_matches_the_plain_pair(na):
    inp = make_custom(0, 0, 3, seed=94, lengths=[1, 129, 700, 0, 2100, 64])
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    cu, mx = inp["cu_seqlens"].cuda(), inp["max_seqlen"]
    H = inp["H"]
    o, lse = na.ne_attn_varlen_fwd(q, k, v, cu, mx)
    o2, lse2, qr, kr = na.ne_attn_varlen_fwd_train(q, k, v, cu, mx)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    cul = [int(c) for c in inp["cu_seqlens"]]
    assert torch.equal(qr.cpu(), _rotated_rows(inp["q"], cul, H))
    assert torch.equal(kr.cpu(), _rotated_rows(inp["k"], cul, H))
    ref = na.ne_attn_varlen_bwd(q, k, v, o, do, lse, cu, mx)
    got = na.ne_attn_varlen_bwd_train(qr, kr, v, o2, do, lse2, cu, mx)
    assert na.ne_attn_get_device_status() == 0
    _same_gradients(got, ref)


def test_rotation_phase_event_brackets_the_pass(na):
    """The forward phase event lands between the rotation pass and the
    attention kernel: both intervals it splits the call into are positive."""
    inp = make_custom(2, 512, 4, seed=95)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e1.record()  # torch times only events it has seen recorded; the library re-records it
    torch.cuda.synchronize()
    na.ne_attn_set_fwd_phase_event(e1)
    try:
        e0.record()
        na.ne_attn_fwd_train(q, k, v)
        e2.record()
        torch.cuda.synchronize()
    finally:
        na.ne_attn_set_fwd_phase_event(None)
    assert e0.elapsed_time(e1) > 0 and e1.elapsed_time(e2) > 0
