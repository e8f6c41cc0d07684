"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small workloads are compared element by element with the full oracle; the
large ones on sampled rows the oracle computes one by one (query rows spread
over the whole sequence; key rows in the tail, where the oracle's dk/dv needs
few query rows).  Edge cases: a single token, ragged tails around the
128-row tile, several batch entries, a packed batch with lengths 1..300, and
the five named workloads.
"""
import numpy as np
import pytest
import torch

from causal_self_attention_gb300.inputs import make_custom, make_inputs
from parity import check_full, check_sampled, packed_view, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from causal_self_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _report(name, errs):
    print(f"\n[parity] {name}: " + ", ".join(f"{k}={v:.3e}" for k, v in errs.items()))


def test_tiny_config_full():
    inp = make_inputs("tiny")
    _report("tiny", check_full(inp, run_gpu(inp)))


@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (2, 1, 3), (1, 63, 2), (2, 65, 1), (1, 129, 3),
                                   (3, 200, 2), (1, 384, 1)])
def test_edge_shapes_full(B, T, H):
    inp = make_custom(B, T, H, seed=100 + T)
    _report(f"B{B} T{T} H{H}", check_full(inp, run_gpu(inp)))


def test_sharp_softmax_full():
    inp = make_custom(2, 300, 2, seed=7, qk_mult=2.0)
    _report("sharp T300", check_full(inp, run_gpu(inp)))


def test_varlen_small_full():
    inp = make_custom(0, 0, 3, seed=11, lengths=[1, 127, 128, 129, 300, 5, 256])
    _report("varlen small", check_full(inp, run_gpu(inp)))


def test_gpt2s_config_full():
    inp = make_inputs("gpt2s")
    _report("gpt2s", check_full(inp, run_gpu(inp)))


def _long_loop_keys(L, rng):
    """Key rows whose gradients sum over the most query tiles: the first key
    tile (rows 0, 1, 127 and a few more), the first row of the second tile, and
    a tile in the middle of the sequence."""
    mid = (L // 2) // 128 * 128
    rows = [0, 1, 127, 128, mid, mid + 1, mid + 127]
    rows += list(rng.integers(0, min(L, 128), 6))
    return [r for r in rows if r < L]


def _picks_fixed(inp, n_q=48, n_k=48, seed=0):
    rng = np.random.default_rng(seed)
    B, T, H = inp["B"], inp["T"], inp["H"]
    picks = []
    for b in range(B):
        for h in range(H):
            if rng.random() > 4.0 / (B * H) and not (b == B - 1 and h == H - 1):
                continue
            qr = np.unique(np.concatenate([[0, 1, 127, 128, T - 1],
                                           rng.integers(0, T, n_q)])).astype(np.int32)
            kr = np.unique(np.concatenate([[T - 1, T - 128, T - 129],
                                           rng.integers(T - 384, T, n_k),
                                           _long_loop_keys(T, rng)])).astype(np.int32)
            picks.append((b, h, qr, kr))
    return picks


def _report_long_loop(name, errs):
    long = {k: v for k, v in errs.items() if "_long" in k}
    print(f"\n[parity] {name} long-loop key rows: " +
          ", ".join(f"{k}={v:.3e}" for k, v in long.items()))


@pytest.mark.parametrize("name", ["byte4k", "long16k"])
def test_long_configs_sampled(name):
    inp = make_inputs(name)
    gpu = run_gpu(inp)
    errs = check_sampled(inp, gpu, _picks_fixed(inp), long_loop_tiles=8)
    _report(name, errs)
    _report_long_loop(name, errs)
    assert "dk_long_rel_l2" in errs


def test_varlen_config_sampled():
    inp = make_inputs("varlen")
    gpu = run_gpu(inp)
    rng = np.random.default_rng(1)
    lengths = [int(L) for L in inp["lengths"]]
    longest = set(np.argsort(lengths)[-2:].tolist())
    picks = []
    for s, L in enumerate(lengths):
        if s % 4 and s not in longest:
            continue
        h = int(rng.integers(inp["H"]))
        qr = np.unique(np.concatenate([[0, L - 1], rng.integers(0, L, 24)])).astype(np.int32)
        kr = [L - 1, max(L - 130, 0)] + list(rng.integers(max(L - 300, 0), L, 24))
        if s in longest:
            kr += _long_loop_keys(L, rng)
        picks.append((s, h, qr, np.unique(np.asarray(kr)).astype(np.int32)))
    errs = check_sampled(inp, gpu, picks, long_loop_tiles=8)
    _report("varlen", errs)
    _report_long_loop("varlen", errs)
    assert "dk_long_rel_l2" in errs


@pytest.mark.parametrize("B,T,H", [(3, 200, 2), (8, 1024, 12)])
def test_varlen_equal_lengths_matches_fixed(B, T, H):
    """A packed batch of equal lengths computes exactly the fixed-length call.
    At the GPT-2-small shape the fixed-length backward deals its units by the
    schedule packed on the host while the packed batch keeps the kernel's
    snake order: which CTA computes a unit must not change dK, dV."""
    from causal_self_attention_gb300 import ne_attn as na
    fixed = make_custom(B, T, H, seed=21)
    packed = dict(fixed)
    D = fixed["D"]
    for n in ("q", "k", "v", "dout"):
        packed[n] = fixed[n].reshape(-1, H, D)
    packed["cu_seqlens"] = torch.arange(0, (B + 1) * T, T, dtype=torch.int32)
    packed["max_seqlen"] = T
    if T == 1024:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        n_units = B * H * (T // 128)
        assert na.ne_debug_schedule(B, H, T, min(sms, n_units)) is not None
    a, b = run_gpu(fixed), run_gpu(packed)
    for n in ("o32", "o16", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    assert torch.allclose(a["dq"].float(), b["dq"].float(), atol=2e-2, rtol=0)


def test_causality_and_isolation_bitwise():
    """Perturbing positions >= t leaves O and LSE of rows < t bitwise unchanged;
    perturbing one packed sequence leaves every other sequence's O, LSE, dK, dV
    bitwise unchanged (no attention weight outside the window)."""
    inp = make_custom(1, 300, 2, seed=31)
    base = run_gpu(inp)
    t = 170
    pert = dict(inp)
    for n in ("q", "k", "v", "dout"):
        x = inp[n].clone()
        x[:, t:] = (x[:, t:].float() * -1.5 + 0.25).to(torch.bfloat16)
        pert[n] = x
    got = run_gpu(pert)
    assert torch.equal(base["o32"][:t], got["o32"][:t])
    assert torch.equal(base["lse"][:, :t], got["lse"][:, :t])

    lengths = [100, 150, 130]
    inp = make_custom(0, 0, 2, seed=32, lengths=lengths)
    base = run_gpu(inp)
    pert = dict(inp)
    a, b = 100, 250  # sequence 1
    for n in ("q", "k", "v", "dout"):
        x = inp[n].clone()
        x[a:b] = (x[a:b].float() * 0.5 - 1.0).to(torch.bfloat16)
        pert[n] = x
    got = run_gpu(pert)
    keep = torch.cat([torch.arange(0, a), torch.arange(b, sum(lengths))])
    for n in ("o32", "dk", "dv"):
        assert torch.equal(base[n][keep], got[n][keep]), n
    assert torch.equal(base["lse"][:, keep], got["lse"][:, keep])


def test_repeated_calls_are_deterministic():
    """O, LSE, dK and dV are bitwise identical across repeated calls (no
    ordering races between the pipeline stages); dQ is accumulated with
    atomics, so it is only required to stay within rounding of itself."""
    from causal_self_attention_gb300 import ne_attn as na
    for inp in (make_custom(1, 129, 3, seed=41), make_inputs("gpt2s")):
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
        ref = None
        for _ in range(3):
            o, lse = na.ne_attn_fwd(q, k, v)
            dq, dk, dv = na.ne_attn_bwd(q, k, v, o, do, lse)
            cur = [t.clone() for t in (o, lse, dk, dv, dq)]
            if ref is None:
                ref = cur
                continue
            for a, b in zip(cur[:4], ref[:4]):
                assert torch.equal(a, b)
            assert torch.allclose(cur[4].float(), ref[4].float(), atol=1e-2, rtol=1e-2)
        assert na.ne_attn_get_device_status() == 0


def test_key_rotation_paths_agree_bitwise():
    """The forward rotates the keys either inside every item that uses them
    (short sequences) or once per call in a pass of its own (from 2048
    positions on); a packed batch called with a small and with a large
    max_seqlen takes the two paths and must give bitwise the same O and LSE."""
    from causal_self_attention_gb300 import ne_attn as na
    inp = make_custom(0, 0, 3, seed=51, lengths=[300, 129, 200])
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"].cuda()
    outs = [na.ne_attn_varlen_fwd(q, k, v, cu, mx, out_f32=f) for mx in (300, 4096)
            for f in (False, True)]
    assert na.ne_attn_get_device_status() == 0
    for a, b in zip(outs[:2], outs[2:]):
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_varlen_sequence_longer_than_max_is_reported():
    """cu_seqlens puts a sequence above max_seqlen: both directions report
    NE_ERR_BAD_SEQLEN, skip that sequence (it is never read past the limit)
    and compute the others exactly as a valid call does -- through the work
    lists compacted on the device, which keep the bad sequence's items so
    that the kernels see and report it.  The training pair's backward (whose
    preprocess streams every packed row without looking at the sequences)
    reports and skips it the same way."""
    from causal_self_attention_gb300 import ne_attn as na
    inp = make_custom(0, 0, 2, seed=77, lengths=[100, 300, 50])
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    cu = inp["cu_seqlens"].cuda()
    o_ref, lse_ref = na.ne_attn_varlen_fwd(q, k, v, cu, 300)
    dq_ref, dk_ref, dv_ref = na.ne_attn_varlen_bwd(q, k, v, o_ref, do, lse_ref, cu, 300)
    assert na.ne_attn_get_device_status() == 0
    o, lse = na.ne_attn_varlen_fwd(q, k, v, cu, 200)
    assert na.ne_attn_get_device_status() == 7  # NE_ERR_BAD_SEQLEN
    dq, dk, dv = na.ne_attn_varlen_bwd(q, k, v, o_ref, do, lse_ref, cu, 200)
    assert na.ne_attn_get_device_status() == 7
    keep = torch.cat([torch.arange(0, 100), torch.arange(400, 450)]).cuda()
    assert torch.equal(o[keep], o_ref[keep])
    assert torch.equal(lse[:, keep], lse_ref[:, keep])
    assert torch.equal(dk[keep], dk_ref[keep]) and torch.equal(dv[keep], dv_ref[keep])
    assert torch.allclose(dq[keep].float(), dq_ref[keep].float(), atol=1e-2, rtol=0)
    assert na.ne_attn_get_device_status() == 0
    _, _, qr, kr = na.ne_attn_varlen_fwd_train(q, k, v, cu, 300)
    assert na.ne_attn_get_device_status() == 0
    dq, dk, dv = na.ne_attn_varlen_bwd_train(qr, kr, v, o_ref, do, lse_ref, cu, 200)
    assert na.ne_attn_get_device_status() == 7
    assert torch.equal(dk[keep], dk_ref[keep]) and torch.equal(dv[keep], dv_ref[keep])
    assert torch.allclose(dq[keep].float(), dq_ref[keep].float(), atol=1e-2, rtol=0)
    assert na.ne_attn_get_device_status() == 0
