"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every check here would fail on a plausible mistake in the oracle: a dropped
term, a wrong sign, a transposed operand, the wrong RoPE pairing or frequency,
a mask off by one, a missing scale, or gradients that skip the rotation.
Nothing here touches the GPU.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_SAFE = {"sin": math.sin, "cos": math.cos, "exp": math.exp, "log": math.log}


def _eval(expr, extra=None):
    ns = dict(_SAFE)
    if extra:
        ns.update(extra)
    return float(eval(expr, {"__builtins__": {}}, ns))


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden)
# --------------------------------------------------------------------------

def test_golden_rope_d4():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "rope_d4_worked.txt"))
             if l.strip() and not l.startswith("#")]
    hdr = {l[0]: l[1] for l in lines if l[0] in ("D", "base", "position")}
    D, base, m = int(hdr["D"]), float(hdr["base"]), int(hdr["position"])
    ins = [list(map(float, l[1:])) for l in lines if l[0] == "input"]
    exps = [[_eval(e) for e in l[1:]] for l in lines if l[0] == "expect"]
    assert len(ins) == len(exps) == D
    for x, e in zip(ins, exps):
        rows = np.zeros((m + 1, D))
        rows[m] = x
        got = oracle.rope(rows, base=base, mode=0)[m]
        np.testing.assert_allclose(got, e, rtol=0, atol=1e-15)


def test_golden_attention_t2_d2():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "attn_t2_d2_worked.txt"))
             if l.strip() and not l.startswith("#")]
    T = int([l for l in lines if l[0] == "T"][0][1])
    D = int([l for l in lines if l[0] == "D"][0][1])
    scale = float([l for l in lines if l[0] == "scale"][0][1])
    arr = {l[0]: np.array(list(map(float, l[1:]))).reshape(T, 1, D)
           for l in lines if l[0] in ("q", "k", "v", "dout")}
    a = 1.0 / (1.0 + math.exp(math.sin(1.0)))
    r = oracle.attention(arr["q"], arr["k"], arr["v"], arr["dout"], [0, T], base=10000.0,
                         scale=scale)
    for l in lines:
        if l[0] != "expect":
            continue
        name, vals = l[1], np.array([_eval(e, {"a": a}) for e in l[2:]])
        got = r[name].reshape(-1)
        np.testing.assert_allclose(got, vals, rtol=0, atol=1e-13, err_msg=name)


# --------------------------------------------------------------------------
# Finite differences (centred, double) through RoPE, as the NanoEuler page
# describes for its own gradients.
# --------------------------------------------------------------------------

def _loss(q, k, v, dout, cu, base, scale):
    r = oracle.attention(q, k, v, None, cu, base=base, scale=scale)
    return float(np.sum(r["o"] * dout))


@pytest.mark.parametrize("T,D,H,base", [(1, 4, 1, 10000.0), (2, 4, 1, 10.0), (5, 8, 2, 10.0),
                                        (8, 8, 1, 10000.0), (8, 4, 1, 3.0)])
def test_finite_difference_gradients(T, D, H, base):
    q, k, v, dout = (_rand((T, H, D), s) for s in range(4))
    scale = 1.0 / math.sqrt(D)
    cu = [0, T]
    r = oracle.attention(q, k, v, dout, cu, base=base, scale=scale)
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, dout, cu, base, scale)
            x[idx] = old - h
            lm = _loss(q, k, v, dout, cu, base, scale)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(r[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_finite_difference_tiny_config_slice():
    """A sample of elements of the T=64, D=64 tiny workload shape, base 10000."""
    T, H, D = 64, 1, 64
    q, k, v, dout = (_rand((T, H, D), 10 + s) for s in range(4))
    scale = 0.125
    cu = [0, T]
    r = oracle.attention(q, k, v, dout, cu, scale=scale)
    rng = np.random.default_rng(5)
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        for _ in range(6):
            idx = (int(rng.integers(T)), 0, int(rng.integers(D)))
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, dout, cu, 10000.0, scale)
            x[idx] = old - h
            lm = _loss(q, k, v, dout, cu, 10000.0, scale)
            x[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(r[name][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_mask():
    T, D = 9, 8
    q, k = _rand((T, D), 1), _rand((T, D), 2)
    P = oracle.probs(q, k, base=10000.0, scale=0.3)
    np.testing.assert_allclose(P.sum(axis=1), np.ones(T), rtol=0, atol=1e-14)
    assert np.all(P[np.triu_indices(T, 1)] == 0.0)
    assert np.all(P[np.tril_indices(T)] > 0.0)


def test_causality_bitwise():
    T, H, D = 12, 2, 8
    q, k, v, dout = (_rand((T, H, D), 20 + s) for s in range(4))
    r0 = oracle.attention(q, k, v, dout, [0, T])
    t = 7
    q2, k2, v2, d2 = (x.copy() for x in (q, k, v, dout))
    for x in (q2, k2, v2, d2):
        x[t:] += _rand(x[t:].shape, 99)
    r1 = oracle.attention(q2, k2, v2, d2, [0, T])
    for name in ("o", "dq"):
        assert np.array_equal(r0[name][:t], r1[name][:t]), name
    assert np.array_equal(r0["lse"][:, :t], r1["lse"][:, :t])


def test_rope_preserves_norm():
    L, D = 300, 64
    x = _rand((L, D), 3)
    xr = oracle.rope(x, base=10000.0)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1),
                               rtol=1e-13)
    # Position 0 is the identity.
    np.testing.assert_array_equal(xr[0], x[0])


def test_rope_relative_position():
    """R(m)q . R(n)k depends only on m - n."""
    L, D = 40, 16
    qv, kv = _rand(D, 4), _rand(D, 5)
    Q = oracle.rope(np.tile(qv, (L, 1)), base=10000.0)
    K = oracle.rope(np.tile(kv, (L, 1)), base=10000.0)
    for delta in (0, 1, 7, 20):
        vals = [Q[m] @ K[m - delta] for m in range(delta, L)]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-11, atol=1e-12)
    # And it is a genuine function of m - n (not constant).
    assert abs(Q[5] @ K[5] - Q[6] @ K[5]) > 1e-3


def test_rope_transpose_is_inverse():
    L, D = 50, 64
    x = _rand((L, D), 6)
    np.testing.assert_allclose(oracle.rope_transpose(oracle.rope(x)), x, atol=1e-12)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_single_position_closed_form():
    H, D = 3, 8
    q, k, v, dout = (_rand((1, H, D), 30 + s) for s in range(4))
    r = oracle.attention(q, k, v, dout, [0, 1], scale=0.5)
    np.testing.assert_allclose(r["o"], v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["lse"][:, 0], 0.5 * np.sum(q[0] * k[0], axis=-1), atol=1e-14)
    # One key: P = 1, dS = 0, so dq = dk = 0 and dv = dO.
    np.testing.assert_allclose(r["dq"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dk"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dv"], dout, atol=1e-15)


def test_zero_query_gives_uniform_weights():
    T, H, D = 10, 2, 8
    q = np.zeros((T, H, D))
    k, v = _rand((T, H, D), 40), _rand((T, H, D), 41)
    r = oracle.attention(q, k, v, None, [0, T])
    m = np.arange(T)
    for h in range(H):
        np.testing.assert_allclose(r["lse"][h], np.log(m + 1), atol=1e-14)
        mean = np.cumsum(v[:, h], axis=0) / (m + 1)[:, None]
        np.testing.assert_allclose(r["o"][:, h], mean, atol=1e-14)


def test_gradient_sum_identities():
    T, H, D = 16, 2, 8
    q, k, v, dout = (_rand((T, H, D), 50 + s) for s in range(4))
    r = oracle.attention(q, k, v, dout, [0, T], want_delta=True)
    # sum_n dv_n = sum_m dO_m (each row of P sums to one).
    np.testing.assert_allclose(r["dv"].sum(axis=0), dout.sum(axis=0), atol=1e-12)
    # D_m = dO_m . O_m.
    np.testing.assert_allclose(r["delta"], np.einsum("thd,thd->ht", dout, r["o"]), atol=1e-12)


def test_equal_rotated_keys_give_zero_dq():
    """If every rotated key is the same vector, every score in a row is equal, so
    sum_n dS_mn k'_n = k' sum_n dS_mn = 0.  The raw keys are R(n)^T c, built here
    with the textbook 2-d rotation (D = 2, theta_0 = 1)."""
    T = 6
    c = np.array([0.7, -1.3])
    k = np.zeros((T, 1, 2))
    for n in range(T):
        cs, sn = math.cos(n), math.sin(n)
        k[n, 0] = [cs * c[0] + sn * c[1], -sn * c[0] + cs * c[1]]
    q, v, dout = _rand((T, 1, 2), 60), _rand((T, 1, 2), 61), _rand((T, 1, 2), 62)
    r = oracle.attention(q, k, v, dout, [0, T], scale=1.0)
    np.testing.assert_allclose(r["dq"], 0.0, atol=1e-13)
    assert np.max(np.abs(r["dk"])) > 1e-3


# --------------------------------------------------------------------------
# Library special case: torch float64 causal SDPA + autograd on rotated inputs
# --------------------------------------------------------------------------

def _torch_rotate(x, base):
    """Rotate-half RoPE with torch ops (test-side, used only to feed SDPA)."""
    L, H, D = x.shape
    half = D // 2
    i = torch.arange(half, dtype=torch.float64)
    theta = base ** (-(2.0 * i) / D)
    ang = torch.arange(L, dtype=torch.float64)[:, None] * theta[None, :]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    x0, x1 = x[..., :half], x[..., half:]
    return torch.cat([x0 * c - x1 * s, x1 * c + x0 * s], dim=-1)


@pytest.mark.parametrize("lengths", [[37], [5, 64, 1, 20]])
def test_against_torch_sdpa_float64(lengths):
    H, D = 3, 16
    N = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
    q, k, v, dout = (_rand((N, H, D), 70 + s) for s in range(4))
    scale = 1.0 / math.sqrt(D)
    r = oracle.attention(q, k, v, dout, cu, scale=scale)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        tq, tk, tv = (torch.tensor(x[a:b], requires_grad=True) for x in (q, k, v))
        qr, kr = _torch_rotate(tq, 10000.0), _torch_rotate(tk, 10000.0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr.transpose(0, 1), kr.transpose(0, 1), tv.transpose(0, 1), is_causal=True,
            scale=scale).transpose(0, 1)
        o.backward(torch.tensor(dout[a:b]))
        np.testing.assert_allclose(r["o"][a:b], o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(r["dq"][a:b], tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(r["dk"][a:b], tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(r["dv"][a:b], tv.grad.numpy(), atol=1e-11)


# --------------------------------------------------------------------------
# Packing, sampling and the bf16-operand mode
# --------------------------------------------------------------------------

def test_varlen_equals_per_sequence_calls():
    lengths = [3, 17, 1, 9]
    H, D = 2, 8
    N = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
    q, k, v, dout = (_rand((N, H, D), 80 + s) for s in range(4))
    r = oracle.attention(q, k, v, dout, cu)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        rs = oracle.attention(q[a:b], k[a:b], v[a:b], dout[a:b], [0, b - a])
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_array_equal(r[name][a:b], rs[name])
        np.testing.assert_array_equal(r["lse"][:, a:b], rs["lse"])


def test_sampled_rows_equal_full():
    T, H, D = 40, 2, 8
    q, k, v, dout = (_rand((T, H, D), 90 + s) for s in range(4))
    full = oracle.attention(q, k, v, dout, [0, T])
    qrows, krows = [0, 13, 39], [2, 30, 39]
    res = oracle.attention_sampled(q, k, v, dout, [0, T], [(0, 1, qrows, krows)])[0]
    np.testing.assert_array_equal(res["o"], full["o"][qrows, 1])
    np.testing.assert_array_equal(res["lse"], full["lse"][1, qrows])
    np.testing.assert_array_equal(res["dq"], full["dq"][qrows, 1])
    np.testing.assert_array_equal(res["dk"], full["dk"][krows, 1])
    np.testing.assert_array_equal(res["dv"], full["dv"][krows, 1])


def _is_bf16(x):
    t = torch.tensor(x, dtype=torch.float64)
    return bool(torch.equal(t.to(torch.bfloat16).to(torch.float64), t))


def test_bf16_operand_mode():
    """mode 1 rounds each rotated element to bf16 after an fp32 rotation; the
    result is bf16-representable and within half a bf16 ulp (plus fp32 error) of
    the double rotation."""
    L, D = 256, 64
    x = torch.randn(L, D, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    xd = oracle.as_f64(x)
    r0 = oracle.rope(xd, mode=0)
    r1 = oracle.rope(xd, mode=1)
    assert _is_bf16(r1)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r0), 1e-30))) - 7)
    assert np.all(np.abs(r1 - r0) <= 0.5 * ulp + 1e-6 * np.abs(r0) + 1e-30)
    # Position 0: cos = 1, sin = 0, so the rotation is exact and so is bf16.
    np.testing.assert_array_equal(r1[0], xd[0])
