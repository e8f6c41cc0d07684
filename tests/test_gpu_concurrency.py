"""Calls in flight on several streams at once, and from several host threads.

The library keeps per-device state (RoPE tables, work schedules) and one
temporary per stream; a call on one stream must neither read another
stream's temporary nor wait for it.  What is checked: the training pair and
the plain pair enqueued alternately on two streams (the backward with and
without a caller workspace), and the plain pair called from two host threads
at once, each on its own stream, give the results of the same calls run one
after the other on one stream (O, LSE, dK, dV bitwise; dQ to the order of its
fp32 accumulation, relative L2 <= 1e-3); the device status stays clean.
"""
import threading

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


def _same(got, ref):
    o, lse, dq, dk, dv = got
    ro, rlse, rdq, rdk, rdv = ref
    assert torch.equal(o, ro) and torch.equal(lse, rlse)
    assert torch.equal(dk, rdk) and torch.equal(dv, rdv)
    assert rel_l2(dq.double().cpu().numpy(), rdq.double().cpu().numpy()) <= DQ_TOL


def _inputs(shapes):
    out = []
    for i, (B, T, H) in enumerate(shapes):
        inp = make_custom(B, T, H, seed=200 + i)
        out.append(tuple(inp[n].cuda() for n in ("q", "k", "v", "dout")))
    return out


def _train(na, q, k, v, do, stream, ws=None):
    o, lse, qr, kr = na.ne_attn_fwd_train(q, k, v, stream=stream)
    dq, dk, dv = na.ne_attn_bwd_train(qr, kr, v, o, do, lse, workspace=ws, stream=stream)
    return o, lse, dq, dk, dv


def _plain(na, q, k, v, do, stream):
    o, lse = na.ne_attn_fwd(q, k, v, stream=stream)
    dq, dk, dv = na.ne_attn_bwd(q, k, v, o, do, lse, stream=stream)
    return o, lse, dq, dk, dv


def test_two_streams_interleaved(na):
    # A long sequence on one stream (its forward uses the stream's temporary
    # for rotated keys), a short batch on the other.
    data = _inputs([(1, 2300, 2), (3, 300, 3)])
    main = torch.cuda.current_stream()
    refs = [_train(na, *d, stream=main) for d in data] + [_plain(na, *d, stream=main) for d in data]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ws = [torch.empty(na.ne_attn_bwd_workspace_bytes(d[0].shape[0] * d[0].shape[1],
                                                     d[0].shape[2]),
                      dtype=torch.uint8, device="cuda") for d in data]
    for s in streams:
        s.wait_stream(main)
    for _ in range(3):
        got = []
        for i, d in enumerate(data):
            with torch.cuda.stream(streams[i]):
                got.append(_train(na, *d, stream=streams[i], ws=ws[i]))
        for i, d in enumerate(data):
            with torch.cuda.stream(streams[i]):
                got.append(_plain(na, *d, stream=streams[i]))
        torch.cuda.synchronize()
        assert na.ne_attn_get_device_status() == 0
        for g, r in zip(got, refs):
            _same(g, r)


def test_two_host_threads(na):
    data = _inputs([(2, 700, 2), (1, 1500, 3)])
    main = torch.cuda.current_stream()
    refs = [_plain(na, *d, stream=main) for d in data]
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def work(i):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(main)
            with torch.cuda.stream(s):
                out = [_plain(na, *data[i], stream=s) for _ in range(5)]
            s.synchronize()
            results[i] = out
        except Exception as ex:  # reported on the main thread
            errors.append(ex)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert na.ne_attn_get_device_status() == 0
    for i in range(2):
        for got in results[i]:
            _same(got, refs[i])
