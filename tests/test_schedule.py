"""CPU checks of the persistent backward's work schedule (ne_debug_schedule,
host code of the library): for a fixed-length batch the backward's units (one
key tile of one sequence and head each) are packed on the host instead of
dealt in a snake order.

What is checked, for the shapes of the named workloads, ragged lengths and
grids smaller than the unit count:
  - the table is a partition: every unit index exactly once, offsets
    non-decreasing, each CTA's units in increasing index order (the kernel's
    longest-first order);
  - its busiest CTA, counted in steps plus a per-unit overhead across the
    range the packer assumes, is no busier than the snake order's (computed
    here independently from the definition of a unit's steps);
  - at the GPT-2-small shape it is measurably better.
"""
import ctypes

import pytest

G_SM = 152
# (nseq, H, T)
SHAPES = {"gpt2s": (8, 12, 1024), "byte4k": (2, 12, 4096), "long16k": (1, 12, 16384),
          "ragged": (3, 5, 700), "short": (4, 2, 129), "one_tile": (6, 4, 100)}
OVERHEAD = (1.0, 1.5, 2.0)  # steps per unit


@pytest.fixture(scope="module")
def na():
    from causal_self_attention_gb300 import build, ne_attn
    build.build()
    return ne_attn


def _steps(nseq, H, T):
    """Steps of unit r in the kernel's longest-first order: key tile
    j = r // (nseq H) meets the query tiles i >= j, one step each."""
    n_tiles = -(-T // 128)
    return [n_tiles - r // (nseq * H) for r in range(n_tiles * nseq * H)]


def _snake(n, G):
    bins = [[] for _ in range(G)]
    k = 0
    while k * G < n:
        for c in range(G):
            r = k * G + ((G - 1 - c) if k & 1 else c)
            if r < n:
                bins[c].append(r)
        k += 1
    return bins


def _worst(bins, w):
    worst = 0.0
    for c in OVERHEAD:
        mean = sum(x + c for x in w) / len(bins)
        worst = max(worst, max(sum(w[i] + c for i in b) for b in bins) / mean)
    return worst


def _bins(tab, G):
    offs, units = tab
    return [units[offs[c]:offs[c + 1]] for c in range(G)]


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("G", [G_SM, 37])
def test_schedule_is_a_partition_no_worse_than_the_snake(na, shape, G):
    nseq, H, T = SHAPES[shape]
    w = _steps(nseq, H, T)
    G = min(G, len(w))
    tab = na.ne_debug_schedule(nseq, H, T, G)
    if tab is None:  # the snake order is kept
        return
    offs, units = tab
    assert len(offs) == G + 1 and offs[0] == 0 and offs[-1] == len(w)
    assert all(a <= b for a, b in zip(offs, offs[1:]))
    assert sorted(units) == list(range(len(w)))
    bins = _bins(tab, G)
    for b in bins:
        assert b == sorted(b)
    assert _worst(bins, w) <= _worst(_snake(len(w), G), w) + 1e-9


def test_schedule_balances_the_gpt2_small_backward(na):
    nseq, H, T = SHAPES["gpt2s"]
    w = _steps(nseq, H, T)
    tab = na.ne_debug_schedule(nseq, H, T, G_SM)
    assert tab is not None
    got = _worst(_bins(tab, G_SM), w)
    snake = _worst(_snake(len(w), G_SM), w)
    print(f"\n[schedule] gpt2s backward: busiest CTA / mean {got:.3f} (snake {snake:.3f})")
    assert got <= 1.07 < snake


def test_schedule_rejects_bad_arguments(na):
    buf = (ctypes.c_int * 16)()
    L = na.lib()
    assert L.ne_debug_schedule(0, 1, 128, 1, buf, 16) == -1
    assert L.ne_debug_schedule(1, 1, 0, 1, buf, 16) == -1
    assert L.ne_debug_schedule(8, 12, 1024, 152, buf, 16) == -1  # table longer than out
    assert L.ne_debug_schedule(1, 1, 128, 1, None, 0) == -1
