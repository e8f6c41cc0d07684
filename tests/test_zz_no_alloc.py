"""The backward entry point that allocates nothing (ne_attn_bwd_noalloc).

Some callers cannot allocate device memory, nor let a library allocate it on
their behalf: code running under an allocator that must own every byte of the
GPU, a serving process whose memory budget is fixed once it has started, a
plug-in handed tensors but no allocator.  For them the library keeps one fixed
scratch array of its own; these tests check that the results through it match
the ordinary backward, on two calls in a row (so that what the first call
leaves in the shared array cannot leak into the second), and that problems
larger than the array are refused on the host.

This file is collected last on purpose: a run that stops at the first failure
has then already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from causal_self_attention_gb300.inputs import make_custom, make_inputs
from parity import GRAD_TOL, rel_l2


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


@pytest.mark.gpu
def test_noalloc_backward_matches_the_ordinary_backward_twice():
    from causal_self_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_self_attention_gb300 import ne_attn as na
    # Two calls in a row through the same scratch: the first at the GPT-2-small
    # training shape, the second on a smaller ragged problem.
    for inp in (make_inputs("gpt2s"), make_custom(2, 300, 3, seed=77)):
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
        o, lse = na.ne_attn_fwd(q, k, v)
        ref = na.ne_attn_bwd(q, k, v, o, do, lse)
        got = na.ne_attn_bwd_noalloc(q, k, v, o, do, lse)
        assert na.ne_attn_get_device_status() == 0
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            err = rel_l2(a.double().cpu().numpy(), b.double().cpu().numpy())
            assert err <= GRAD_TOL, (inp["name"], name, err)
            assert np.isfinite(a.float().cpu().numpy()).all()
