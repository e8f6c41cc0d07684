"""Seeded random shapes: fixed-length batches (B 1-6, T from 1 to 2300, H 1-12)
and packed batches (1-7 sequences of 0 to 2200 rows, empty ones included).

What is checked, per shape: the training pair gives the plain pair's O, LSE,
dK, dV bitwise and its dQ to the order of the fp32 accumulation (relative L2
<= 1e-3), with a clean device status; on the smaller shapes both pairs also
meet the oracle's bar (the helpers of the named-workload parity tests).
"""
import random

import pytest
import torch

from causal_self_attention_gb300.inputs import make_custom
from parity import check_full, rel_l2, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _shape(rng, trial, small):
    H = rng.choice([1, 2, 3] if small else [1, 2, 3, 5, 12])
    long = 420 if small else 2200
    if rng.random() < 0.4:
        lengths = [rng.choice([0, 1, rng.randint(1, 130), rng.randint(100, long)])
                   for _ in range(rng.randint(1, 4 if small else 7))]
        if sum(lengths) == 0:
            lengths[0] = 3
        return make_custom(0, 0, H, seed=5000 + trial, lengths=lengths)
    T = rng.choice([1, 2, 63, 64, 65, 127, 128, 129, rng.randint(1, long)] +
                   ([] if small else [rng.randint(1900, 2300)]))
    return make_custom(rng.randint(1, 3 if small else 6), T, H, seed=6000 + trial)


@pytest.mark.parametrize("trial", range(16))
def test_training_pair_equals_plain_pair(na, trial):
    inp = _shape(random.Random(1000 + trial), trial, small=False)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    if "cu_seqlens" in inp:
        cu, mx = inp["cu_seqlens"].cuda(), inp["max_seqlen"]
        o, lse = na.ne_attn_varlen_fwd(q, k, v, cu, mx)
        o2, lse2, qr, kr = na.ne_attn_varlen_fwd_train(q, k, v, cu, mx)
        ref = na.ne_attn_varlen_bwd(q, k, v, o, do, lse, cu, mx)
        got = na.ne_attn_varlen_bwd_train(qr, kr, v, o2, do, lse2, cu, mx)
    else:
        o, lse = na.ne_attn_fwd(q, k, v)
        o2, lse2, qr, kr = na.ne_attn_fwd_train(q, k, v)
        ref = na.ne_attn_bwd(q, k, v, o, do, lse)
        got = na.ne_attn_bwd_train(qr, kr, v, o2, do, lse2)
    assert na.ne_attn_get_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    assert rel_l2(got[0].double().cpu().numpy(), ref[0].double().cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("trial", range(8))
def test_small_random_shapes_meet_the_oracle_bar(na, trial):
    inp = _shape(random.Random(2000 + trial), trial, small=True)
    for train in (False, True):
        check_full(inp, run_gpu(inp, device="cuda", train=train))
