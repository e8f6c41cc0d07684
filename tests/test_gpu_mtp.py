"""Parity of the multi-token prediction head (ne_mtp_head: K linear heads on
the hidden states, head j predicting the token j + 1 positions ahead, softmax
cross-entropy over a 256-way byte vocabulary, analytic dh and dW) with the
CPU oracle evaluated in fp64 on the same bf16 inputs.

Tolerance: the logits are fp32 sums of exact bf16 products (relative error of
order 1e-6 for C <= 768), so the loss and each row's loss agree to ~1e-5; the
bar is 1e-3 (absolute, per row) and 1e-4 relative for the mean.  dlogits are
rounded to bf16 (relative 2^-9) before the two gradient products, and dh is
rounded to bf16 again, so dh and dW carry a relative L2 error of a few 1e-3;
the bar is 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _inputs(M, C, K, seed, ignore=0.2, V=256):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn((M, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((K * V, C), generator=g) * (2.0 / C ** 0.5)).to(torch.bfloat16)
    tg = torch.randint(0, V, (M, K), generator=g, dtype=torch.int32)
    tg[torch.rand((M, K), generator=g) < ignore] = -1
    return h, w, tg


def _check(na, M, C, K, seed, **kw):
    h, w, tg = _inputs(M, C, K, seed, **kw)
    loss, row, dh, dw = na.ne_mtp_head(h.cuda(), w.cuda(), tg.cuda(), K)
    assert na.ne_attn_get_device_status() == 0
    r_loss, r_row, r_dh, r_dw = oracle.mtp_head(h, w, tg.numpy(), K)
    got = float(loss.cpu()[0])
    errs = {
        "loss": abs(got - r_loss) / max(abs(r_loss), 1e-30),
        "row_max_abs": float(np.max(np.abs(row.cpu().double().numpy() - r_row))),
        "dh": rel_l2(dh.cpu().double().numpy(), r_dh),
        "dw": rel_l2(dw.cpu().double().numpy(), r_dw),
    }
    assert torch.isfinite(dh.float()).all() and torch.isfinite(dw).all()
    assert errs["loss"] <= 1e-4, errs
    assert errs["row_max_abs"] <= 1e-3, errs
    assert errs["dh"] <= 1e-2 and errs["dw"] <= 1e-2, errs
    return errs


@pytest.mark.parametrize("M,C,K", [(300, 192, 2), (129, 64, 1), (257, 320, 3)])
def test_mtp_head_small_ragged(na, M, C, K):
    """Ragged token counts (partial 128-row tiles), widths that leave a partial
    256-column tile (and whole 64-column blocks past the end), 1-3 heads."""
    errs = _check(na, M, C, K, seed=M + C + K)
    print(f"\\n[mtp] M={M} C={C} K={K}: {errs}")


def test_mtp_head_gpt2s_shape(na):
    """The GPT-2-small training shape: 8192 tokens of width 768, next token
    and the one after it (K = 2), against the oracle on every row."""
    errs = _check(na, 8192, 768, 2, seed=5)
    print(f"\\n[mtp] gpt2s: {errs}")


def test_mtp_head_without_targets_is_zero(na):
    h, w, tg = _inputs(200, 128, 2, seed=9)
    tg[:] = -1
    loss, row, dh, dw = na.ne_mtp_head(h.cuda(), w.cuda(), tg.cuda(), 2)
    assert na.ne_attn_get_device_status() == 0
    assert float(loss.cpu()[0]) == 0.0
    assert torch.count_nonzero(row) == 0 and torch.count_nonzero(dh) == 0
    assert torch.count_nonzero(dw) == 0


def test_mtp_head_repeatable(na):
    """dh and the row losses are bitwise the same from call to call (no
    atomics on their path); dW (split-K reduce-adds) to its accumulation
    order."""
    h, w, tg = (t.cuda() for t in _inputs(1000, 256, 2, seed=13))
    a = na.ne_mtp_head(h, w, tg, 2)
    b = na.ne_mtp_head(h, w, tg, 2)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert rel_l2(a[3].cpu().double().numpy(), b[3].cpu().double().numpy()) <= 1e-6
