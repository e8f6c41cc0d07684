"""Bring-up checks of each hardware primitive the attention kernels rely on,
against plain host arithmetic: the TMA 128-byte-swizzled tile load, the
in-shared-memory RoPE of a tile (bitwise against the oracle's bf16-operand
rule), and the three tcgen05 MMA operand forms."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ne_attn


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("row0", [0, 200])
def test_tma_tile_swizzle(na, row0):
    n, H, h = 300, 3, 1
    src = _bf16((n, H, 64), 1)
    raw = na.ne_debug_tma_tile(src.cuda(), h, row0).cpu().numpy().view(np.uint16)
    exp = np.zeros(8192, dtype=np.uint16)
    s16 = src.view(torch.int16).numpy().view(np.uint16)
    for r in range(128):
        if row0 + r >= n:
            continue  # out of range rows read as zero
        for c in range(8):
            off = (r * 128 + ((c ^ (r & 7)) * 16)) // 2
            exp[off:off + 8] = s16[row0 + r, h, 8 * c:8 * c + 8]
    np.testing.assert_array_equal(raw, exp)


@pytest.mark.parametrize("pos0", [0, 384, 16256])
def test_rope_tile_bitwise(na, pos0):
    n, H, h = 256, 2, 1
    src = _bf16((n, H, 64), 2, 2.0)
    got = na.ne_debug_rope_tile(src.cuda(), h, 64, pos0).cpu().double().numpy()
    rows = np.zeros((pos0 + 128, 64))
    rows[pos0:] = src[64:192, h].double().numpy()
    ref = oracle.rope(rows, base=10000.0, mode=1)[pos0:]
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("form", [0, 1, 2, 3])
def test_umma_forms(na, form):
    if form == 0:
        a, b = _bf16((128, 64), 3), _bf16((128, 64), 4)
        ref = a.double() @ b.double().T
    elif form == 1:
        a, b = _bf16((128, 128), 5), _bf16((128, 64), 6)
        ref = a.double() @ b.double()
    elif form == 2:
        a, b = _bf16((128, 128), 7), _bf16((128, 64), 8)
        ref = a.double().T @ b.double()
    else:
        a, b = _bf16((128, 128), 9), _bf16((128, 64), 10)
        ref = a.double() @ b.double()
    d = na.ne_debug_umma(form, a.cuda(), b.cuda()).cpu().double()
    assert na.ne_attn_get_device_status() == 0
    err = (d - ref).abs().max().item()
    assert err <= 1e-4 * max(1.0, ref.abs().max().item()), err
