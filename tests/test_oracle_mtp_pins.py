"""Pins of the oracle's multi-token prediction head (softmax cross-entropy of K
linear heads, head j predicting the token j + 1 positions ahead) and its
analytic gradients.

Each pin is independent of the oracle's arithmetic:
- a hand-worked case (logits 1, 2, 3), evaluated here from the closed forms;
- zero weights: every logit is 0, so each term is log V exactly, dh = 0 and
  dw has a closed form;
- centred finite differences in double precision, the check the NanoEuler
  Show HN page (paragraph 2) describes for the engine's analytic gradients,
  "including the RoPE and MTP layers";
- invariances: adding one vector to every row of a head leaves the loss and
  the gradients unchanged (softmax shift invariance; the rows of dlogit sum to
  0); permuting the heads permutes dw's blocks and leaves the rest unchanged;
  no targets give a zero loss and zero gradients.
"""
import math

import numpy as np
import pytest

import oracle


def test_hand_worked_case():
    h = np.array([[1.0, 2.0]])
    w = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])  # logits h.w_v = 1, 2, 3
    loss, row, dh, dw = oracle.mtp_head(h, w, [[0]], K=1)
    z = math.exp(1) + math.exp(2) + math.exp(3)
    p = [math.exp(1) / z, math.exp(2) / z, math.exp(3) / z]
    assert loss == pytest.approx(math.log(z) - 1.0, rel=1e-15, abs=1e-15)
    assert row[0, 0] == pytest.approx(math.log(z) - 1.0, rel=1e-15)
    g = [p[0] - 1.0, p[1], p[2]]  # softmax - onehot, n = 1
    np.testing.assert_allclose(dh[0], [g[0] + g[2], g[1] + g[2]], rtol=1e-14)
    np.testing.assert_allclose(dw, [[g[0], 2 * g[0]], [g[1], 2 * g[1]], [g[2], 2 * g[2]]],
                               rtol=1e-14)


def _problem(seed, M=7, C=5, K=2, V=6, ignore=0.25):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((M, C))
    w = rng.standard_normal((K * V, C)) * 0.7
    tg = rng.integers(0, V, size=(M, K)).astype(np.int32)
    tg[rng.random((M, K)) < ignore] = -1
    return h, w, tg, K, V


def test_zero_weights_closed_form():
    h, _, tg, K, V = _problem(3, M=9, C=4, K=3, V=5)
    w = np.zeros((K * V, h.shape[1]))
    loss, row, dh, dw = oracle.mtp_head(h, w, tg, K)
    valid = tg >= 0
    n = int(valid.sum())
    assert loss == pytest.approx(math.log(V), rel=1e-14)
    np.testing.assert_allclose(row[valid], math.log(V), rtol=1e-14)
    assert np.all(row[~valid] == 0.0)
    assert np.all(dh == 0.0)
    # dw_{jV+v} = (1/n) sum_{t with target} (1/V - [y_tj = v]) h_t
    want = np.zeros_like(dw)
    for j in range(K):
        for t in range(h.shape[0]):
            if tg[t, j] < 0:
                continue
            for v in range(V):
                want[j * V + v] += ((1.0 / V) - (1.0 if tg[t, j] == v else 0.0)) * h[t] / n
    np.testing.assert_allclose(dw, want, rtol=1e-13, atol=1e-15)


def test_gradients_match_centred_finite_differences():
    h, w, tg, K, V = _problem(7)
    _, _, dh, dw = oracle.mtp_head(h, w, tg, K)
    eps = 1e-6
    rng = np.random.default_rng(1)
    for _ in range(12):
        i, c = rng.integers(0, h.shape[0]), rng.integers(0, h.shape[1])
        hp, hm = h.copy(), h.copy()
        hp[i, c] += eps
        hm[i, c] -= eps
        fd = (oracle.mtp_head(hp, w, tg, K)[0] - oracle.mtp_head(hm, w, tg, K)[0]) / (2 * eps)
        assert fd == pytest.approx(dh[i, c], rel=1e-6, abs=1e-9)
        r, c = rng.integers(0, w.shape[0]), rng.integers(0, w.shape[1])
        wp, wm = w.copy(), w.copy()
        wp[r, c] += eps
        wm[r, c] -= eps
        fd = (oracle.mtp_head(h, wp, tg, K)[0] - oracle.mtp_head(h, wm, tg, K)[0]) / (2 * eps)
        assert fd == pytest.approx(dw[r, c], rel=1e-6, abs=1e-9)


def test_shift_of_a_heads_rows_changes_nothing():
    h, w, tg, K, V = _problem(11)
    base = oracle.mtp_head(h, w, tg, K)
    u = np.random.default_rng(2).standard_normal(h.shape[1])
    w2 = w.copy()
    w2[V:2 * V] += u  # every row of head 1
    got = oracle.mtp_head(h, w2, tg, K)
    assert got[0] == pytest.approx(base[0], rel=1e-12)
    for a, b in zip(got[1:], base[1:]):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_head_permutation():
    h, w, tg, K, V = _problem(13, K=3)
    base = oracle.mtp_head(h, w, tg, K)
    perm = [2, 0, 1]
    w2 = np.concatenate([w[j * V:(j + 1) * V] for j in perm])
    got = oracle.mtp_head(h, w2, tg[:, perm], K)
    assert got[0] == pytest.approx(base[0], rel=1e-13)
    np.testing.assert_allclose(got[1], base[1][:, perm], rtol=1e-13)
    np.testing.assert_allclose(got[2], base[2], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(got[3], np.concatenate([base[3][j * V:(j + 1) * V] for j in perm]),
                               rtol=1e-12, atol=1e-15)


def test_no_targets_give_zeros():
    h, w, tg, K, V = _problem(17)
    tg[:] = -1
    loss, row, dh, dw = oracle.mtp_head(h, w, tg, K)
    assert loss == 0.0 and np.all(row == 0) and np.all(dh == 0) and np.all(dw == 0)


def test_bad_target_is_refused():
    h, w, tg, K, V = _problem(19)
    tg[0, 0] = V
    with pytest.raises(ValueError):
        oracle.mtp_head(h, w, tg, K)
