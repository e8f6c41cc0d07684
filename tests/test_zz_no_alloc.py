"""The backward entry point that allocates nothing (ne_attn_bwd_noalloc).

Some callers cannot allocate device memory, nor let a library allocate it on
their behalf: code running under an allocator that must own every byte of the
GPU, a serving process whose memory budget is fixed once it has started, a
plug-in handed tensors but no allocator.  For them the library keeps one fixed
scratch array of its own.  These tests check, through the C ABI, that the
results through that array are those of the ordinary backward (dK and dV
bitwise, dQ up to the order of its fp32 additions) on calls in a row, so that
what one call leaves in the shared array cannot leak into the next; that they
meet the oracle's bar on their own; that a new RoPE base rewrites the table in
stream order, behind earlier work on the caller's stream, and is refused inside
a stream capture; and that problems larger than the array are refused on the
host.

This file is collected last on purpose: a run that stops at the first failure
has then already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from causal_self_attention_gb300.inputs import make_custom, make_inputs
from parity import GRAD_TOL, packed_view, rel_l2

# dQ of the two paths differs only in the order of its fp32 reduce-adds.
DQ_TOL = 1e-3


def test_oversized_problems_are_refused_on_the_host():
    from causal_self_attention_gb300 import build
    lib = ctypes.CDLL(build.build())
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.ne_attn_bwd_noalloc.argtypes = [P] * 6 + [I] * 4 + [F] * 2 + [P] * 4
    fake = P(0x10000)  # never dereferenced: the size check comes first
    args = [fake] * 6

    def call(B, H, T):
        return lib.ne_attn_bwd_noalloc(*args, B, H, T, 64, 10000.0, 0.125, fake, fake, fake, None)

    assert call(1, 1, 16385) == 8  # more positions than the RoPE table holds
    assert call(9, 12, 1024) == 8  # 110592 token-head rows > 108000


def _na():
    from causal_self_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_self_attention_gb300 import ne_attn as na
    return na


def _compare(got, ref, what):
    dq, dk, dv = got
    rq, rk, rv = ref
    assert torch.equal(dk, rk), (what, "dk")
    assert torch.equal(dv, rv), (what, "dv")
    err = rel_l2(dq.double().cpu().numpy(), rq.double().cpu().numpy())
    assert err <= DQ_TOL, (what, "dq", err)
    for t in got:
        assert torch.isfinite(t.float()).all(), what
    return err


@pytest.mark.gpu
def test_noalloc_backward_matches_the_ordinary_backward_twice():
    na = _na()
    # Two calls in a row through the same scratch: the first at the GPT-2-small
    # training shape, the second on a smaller ragged problem.
    for inp in (make_inputs("gpt2s"), make_custom(2, 300, 3, seed=77)):
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
        o, lse = na.ne_attn_fwd(q, k, v)
        ref = na.ne_attn_bwd(q, k, v, o, do, lse)
        got = na.ne_attn_bwd_noalloc(q, k, v, o, do, lse)
        assert na.ne_attn_get_device_status() == 0
        err = _compare(got, ref, inp["name"])
        print(f"\n[noalloc] {inp['name']}: dk, dv bitwise equal; dq rel L2 {err:.2e}")


@pytest.mark.gpu
def test_noalloc_backward_meets_the_oracle_bar():
    na = _na()
    inp = make_inputs("tiny")
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = na.ne_attn_fwd(q, k, v)
    got = na.ne_attn_bwd_noalloc(q, k, v, o, do, lse)
    assert na.ne_attn_get_device_status() == 0
    (cq, ck, cv, cdo), cu = packed_view(inp)
    ref = oracle.attention(cq, ck, cv, cdo, cu, base=inp["rope_base"], scale=inp["scale"], mode=0)
    H, D = inp["H"], inp["D"]
    for name, t in zip(("dq", "dk", "dv"), got):
        err = rel_l2(t.reshape(-1, H, D).double().cpu().numpy(), ref[name])
        assert err <= GRAD_TOL, (name, err)


@pytest.mark.gpu
def test_noalloc_table_rewrite_is_ordered_on_the_callers_stream():
    """Two calls queued back to back on a side stream, the second with another
    RoPE base, behind a long busy kernel: the second call's table rewrite must
    wait for the first call's kernels, and both must match the ordinary path
    at their own base."""
    na = _na()
    inp = make_custom(2, 520, 3, seed=91)
    side = torch.cuda.Stream()
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    bases = (10000.0, 500000.0)
    with torch.cuda.stream(side):
        fw = [na.ne_attn_fwd(q, k, v, rope_base=b, stream=side) for b in bases]
        refs = [na.ne_attn_bwd(q, k, v, o, do, lse, rope_base=b, stream=side)
                for b, (o, lse) in zip(bases, fw)]
    side.synchronize()
    outs = [tuple(torch.empty_like(q) for _ in range(3)) for _ in bases]
    with torch.cuda.stream(side):
        torch.cuda._sleep(100_000_000)  # keeps the stream busy while the calls are enqueued
        for b, (o, lse), (dq, dk, dv) in zip(bases, fw, outs):
            na.ne_attn_bwd_noalloc(q, k, v, o, do, lse, rope_base=b, dq=dq, dk=dk, dv=dv,
                                   stream=side)
    assert na.ne_attn_get_device_status(side) == 0
    for b, got, ref in zip(bases, outs, refs):
        _compare(got, ref, f"base {b}")
    # The two bases give different gradients: the table really changed.
    assert not torch.equal(outs[0][1], outs[1][1])


@pytest.mark.gpu
def test_noalloc_base_change_inside_a_capture_is_refused():
    """A new RoPE base inside a stream capture would capture a copy of a host
    image that later calls rebuild: refused with NE_ERR_UNSUPPORTED, nothing
    enqueued; a call at the base already in the table is captured and replays
    to the eager results."""
    na = _na()
    inp = make_custom(1, 200, 2, seed=92)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = na.ne_attn_fwd(q, k, v, rope_base=10000.0)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    na.ne_attn_bwd_noalloc(q, k, v, o, do, lse, rope_base=10000.0, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (dq, dk, dv)]
    for t in (dq, dk, dv):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(RuntimeError, match="UNSUPPORTED"):
            na.ne_attn_bwd_noalloc(q, k, v, o, do, lse, rope_base=20000.0, dq=dq, dk=dk, dv=dv)
        na.ne_attn_bwd_noalloc(q, k, v, o, do, lse, rope_base=10000.0, dq=dq, dk=dk, dv=dv)
    g.replay()
    torch.cuda.synchronize()
    assert na.ne_attn_get_device_status() == 0
    _compare((dq, dk, dv), ref, "captured at base 10000")
