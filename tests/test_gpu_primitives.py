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


def test_pipeline_completes_without_a_drop(na):
    src = _bf16((4 * 128, 2, 64), 11)
    d = na.ne_debug_pipeline(src.cuda(), 4).cpu().double()
    assert na.ne_attn_get_device_status() == 0
    a = src[:, 0].double().reshape(4, 128, 64)
    ref = sum(a[i] @ a[i].T for i in range(4))
    err = (d - ref).abs().max().item()
    assert err <= 1e-4 * ref.abs().max().item(), err


def test_expired_wait_reports_timeout_and_leaves_the_gpu_usable(na):
    """A left-out producer arrive makes the consumer's bounded wait expire
    (limit 1e5 cycles, about 50 us): the kernel reports NE_ERR_TIMEOUT with the
    wait site, drains and exits; the next ordinary calls are correct."""
    src = _bf16((4 * 128, 2, 64), 12)
    na.ne_debug_pipeline(src.cuda(), 4, drop_item=2, wait_limit_cycles=100_000)
    assert na.ne_attn_get_device_status() == 5  # NE_ERR_TIMEOUT
    assert na.ne_attn_last_device_code() == 0x100 + 51
    assert na.ne_attn_get_device_status() == 0  # reading the status cleared it
    test_pipeline_completes_without_a_drop(na)
    from causal_self_attention_gb300.inputs import make_inputs
    from parity import check_full, run_gpu
    inp = make_inputs("tiny")
    check_full(inp, run_gpu(inp))
