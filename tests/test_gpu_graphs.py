"""The attention calls captured in a CUDA graph and replayed.

Inside a stream capture the library takes its capture-aware paths: the
backward's workspace and the forward's temporary for rotated keys are
stream-ordered allocations of the captured call itself, a packed batch's
work lists too, and a fixed-length backward whose work schedule has not been
made yet falls back to the snake order; a call that would have to build a
RoPE table is refused.  What is checked: replaying the
graph gives the results of the same calls launched eagerly (O, LSE, dK, dV
bitwise; dQ to the order of its fp32 accumulation, relative L2 <= 1e-3), for
the training pair (replayed twice, with new inputs copied in between), for
the plain pair on a sequence long enough that the forward rotates its keys
in a separate pass, and for a packed variable-length batch; the device
status stays clean.
"""
import pytest
import torch

from causal_self_attention_gb300.inputs import make_custom
from parity import rel_l2

pytestmark = pytest.mark.gpu
DQ_TOL = 1e-3


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _capture(fn):
    """Capture fn() on a side stream; returns the graph and fn's outputs."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        outs = fn()
    torch.cuda.synchronize()
    return g, outs


def _same(got, ref, dq_index):
    for i, (a, b) in enumerate(zip(got, ref)):
        if i == dq_index:
            err = rel_l2(a.double().cpu().numpy(), b.double().cpu().numpy())
            assert err <= DQ_TOL, ("dq", err)
        else:
            assert torch.equal(a, b), i


def test_first_use_of_a_rope_base_inside_a_capture_is_refused(na):
    """A new base needs its table built, which a capture does not allow: the
    call returns NE_ERR_UNSUPPORTED and enqueues nothing; the capture goes on
    and the graph replays the rest of what was captured."""
    inp = make_custom(1, 64, 1, seed=100)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    x = torch.zeros(4, device="cuda")

    def body():
        x.add_(1.0)
        with pytest.raises(RuntimeError, match="UNSUPPORTED"):
            na.ne_attn_fwd(q, k, v, rope_base=12345.0)
        return (x,)

    g, _ = _capture(body)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x, torch.ones(4, device="cuda"))
    assert na.ne_attn_get_device_status() == 0
    na.ne_attn_fwd(q, k, v, rope_base=12345.0)  # outside a capture the table is built


def test_training_step_replays_like_eager_launches(na):
    inp = make_custom(2, 300, 3, seed=101)
    new = make_custom(2, 300, 3, seed=102)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))

    def step():
        o, lse, qr, kr = na.ne_attn_fwd_train(q, k, v)
        dq, dk, dv = na.ne_attn_bwd_train(qr, kr, v, o, do, lse)
        return o, lse, dq, dk, dv

    # A warm-up outside the capture on another shape (the RoPE table, the
    # kernels' launch attributes); this shape's work schedule is not made yet.
    w = make_custom(1, 128, 1, seed=105)
    wq, wk, wv, wdo = (w[n].cuda() for n in ("q", "k", "v", "dout"))
    wo, wl, wqr, wkr = na.ne_attn_fwd_train(wq, wk, wv)
    na.ne_attn_bwd_train(wqr, wkr, wv, wo, wdo, wl)
    na.ne_attn_fwd(q, k, v)
    torch.cuda.synchronize()
    g, outs = _capture(step)
    for src in (inp, new):
        for n, t in (("q", q), ("k", k), ("v", v), ("dout", do)):
            t.copy_(src[n].cuda())
        g.replay()
        torch.cuda.synchronize()
        assert na.ne_attn_get_device_status() == 0
        got = [t.clone() for t in outs]
        ref = step()
        torch.cuda.synchronize()
        _same(got, ref, dq_index=2)


def test_plain_pair_with_a_key_rotation_pass_replays_like_eager_launches(na):
    inp = make_custom(1, 2100, 2, seed=103)  # from 2048 positions on: keys rotated in a pass
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))

    def step():
        o, lse = na.ne_attn_fwd(q, k, v)
        dq, dk, dv = na.ne_attn_bwd(q, k, v, o, do, lse)
        return o, lse, dq, dk, dv

    ref = step()
    torch.cuda.synchronize()
    g, outs = _capture(step)
    g.replay()
    torch.cuda.synchronize()
    assert na.ne_attn_get_device_status() == 0
    _same(outs, ref, dq_index=2)


def test_packed_batch_replays_like_eager_launches(na):
    inp = make_custom(0, 0, 3, seed=104, lengths=[1, 129, 700, 0, 2100, 64])
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    cu, mx = inp["cu_seqlens"].cuda(), inp["max_seqlen"]

    def step():
        o, lse = na.ne_attn_varlen_fwd(q, k, v, cu, mx)
        dq, dk, dv = na.ne_attn_varlen_bwd(q, k, v, o, do, lse, cu, mx)
        return o, lse, dq, dk, dv

    ref = step()
    torch.cuda.synchronize()
    g, outs = _capture(step)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert na.ne_attn_get_device_status() == 0
    _same(outs, ref, dq_index=2)
