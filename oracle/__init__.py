"""CPU oracle for causal self-attention with RoPE, forward and backward, for
the projections around it (RMSNorm + QKV projection with RoPE; output
projection + residual), and for a multi-token prediction head with its
softmax cross-entropy loss and analytic gradients.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  The product library never
does, and this package never imports the product: the two share no code.

The arithmetic lives in ``ne_attn_oracle.c`` (plain C, double precision,
OpenMP over rows).  This module only builds that file, loads it with ctypes and
marshals numpy arrays in and out; it adds no arithmetic of its own.

Layout convention (same as the library's public one, chosen so a fixed-length
batch is a packed batch with equal lengths): tokens are rows of a
``[tokens, heads, D]`` array; a fixed-length batch ``[B, T, H, D]`` is viewed
as ``[B*T, H, D]`` with sequence boundaries ``cu_seqlens = [0, T, 2T, ...]``.
LSE and D_m come back as ``[heads, tokens]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ne_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libne_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libne_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.ne_oracle_rope.argtypes = [dp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, ctypes.c_int, dp]
        lib.ne_oracle_rope.restype = ctypes.c_int
        lib.ne_oracle_rope_transpose.argtypes = [dp, ctypes.c_longlong, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, dp]
        lib.ne_oracle_rope_transpose.restype = ctypes.c_int
        lib.ne_oracle_attention_head.argtypes = [
            dp, dp, dp, dp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_double, ctypes.c_int, ip, ctypes.c_int, ip, ctypes.c_int,
            dp, dp, dp, dp, dp, dp]
        lib.ne_oracle_attention_head.restype = ctypes.c_int
        lib.ne_oracle_probs.argtypes = [dp, dp, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_int, dp]
        lib.ne_oracle_probs.restype = ctypes.c_int
        lib.ne_oracle_rmsnorm.argtypes = [dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_double, dp]
        lib.ne_oracle_rmsnorm.restype = ctypes.c_int
        lib.ne_oracle_linear.argtypes = [dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
        lib.ne_oracle_linear.restype = ctypes.c_int
        lib.ne_oracle_qkv_rope.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                           dp, dp, dp]
        lib.ne_oracle_qkv_rope.restype = ctypes.c_int
        lib.ne_oracle_out_proj_residual.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int, dp]
        lib.ne_oracle_out_proj_residual.restype = ctypes.c_int
        lib.ne_oracle_mtp_head.argtypes = [dp, dp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, dp, dp, dp, dp]
        lib.ne_oracle_mtp_head.restype = ctypes.c_int
        lib.ne_oracle_num_threads.argtypes = []
        lib.ne_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _dptr(a, offset: int = 0):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    assert 0 <= offset <= a.size
    return ctypes.cast(a.ctypes.data + 8 * int(offset), ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    assert a.dtype == np.int32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def as_f64(x) -> np.ndarray:
    """A torch tensor (any float dtype, CPU) or array as a contiguous float64 array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def num_threads() -> int:
    return int(_load().ne_oracle_num_threads())


def rope(x: np.ndarray, base: float = 10000.0, mode: int = 0) -> np.ndarray:
    """Rotate rows of ``x`` ``[L, D]`` at positions 0..L-1."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    L, D = x.shape
    out = np.empty_like(x)
    if _load().ne_oracle_rope(_dptr(x), D, L, D, float(base), int(mode), _dptr(out)) != 0:
        raise ValueError("ne_oracle_rope: bad arguments")
    return out


def rope_transpose(g: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """Apply R(m)^T to rows of ``g`` ``[L, D]`` at positions 0..L-1."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    L, D = g.shape
    out = np.empty_like(g)
    if _load().ne_oracle_rope_transpose(_dptr(g), D, L, D, float(base), _dptr(out)) != 0:
        raise ValueError("ne_oracle_rope_transpose: bad arguments")
    return out


def probs(q: np.ndarray, k: np.ndarray, base: float = 10000.0, scale: float | None = None,
          mode: int = 0) -> np.ndarray:
    """Full causal probability matrix ``P[L, L]`` of one head (``q``, ``k``: ``[L, D]``)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    L, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    P = np.empty((L, L), dtype=np.float64)
    if _load().ne_oracle_probs(_dptr(q), _dptr(k), D, L, D, float(base), float(scale),
                               int(mode), _dptr(P)) != 0:
        raise ValueError("ne_oracle_probs: bad arguments")
    return P


def head(q, k, v, dout, offset, L, D, stride, base, scale, mode, qrows, krows,
         want_o=True, want_lse=True, want_delta=False, want_dq=True, want_dkdv=True):
    """One (sequence, head).  ``q``, ``k``, ``v``, ``dout`` are contiguous float64
    arrays; row 0 of that sequence and head starts ``offset`` elements into each,
    and consecutive rows are ``stride`` elements apart."""
    lib = _load()
    qrows = np.ascontiguousarray(qrows, dtype=np.int32)
    krows = np.ascontiguousarray(krows, dtype=np.int32)
    nq, nk = len(qrows), len(krows)
    bwd = dout is not None
    o = np.empty((nq, D)) if want_o else None
    lse = np.empty(nq) if want_lse else None
    delta = np.empty(nq) if (want_delta and bwd) else None
    dq = np.empty((nq, D)) if (want_dq and bwd) else None
    dk = np.empty((nk, D)) if (want_dkdv and bwd) else None
    dv = np.empty((nk, D)) if (want_dkdv and bwd) else None
    rc = lib.ne_oracle_attention_head(
        _dptr(q, offset), _dptr(k, offset), _dptr(v, offset),
        _dptr(dout, offset) if bwd else None, int(stride), int(L), int(D),
        float(base), float(scale), int(mode), _iptr(qrows), nq, _iptr(krows), nk,
        _dptr(o), _dptr(lse), _dptr(delta), _dptr(dq), _dptr(dk), _dptr(dv))
    if rc != 0:
        raise ValueError("ne_oracle_attention_head: bad arguments")
    return dict(o=o, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv)


def attention(q, k, v, dout=None, cu_seqlens=None, base: float = 10000.0,
              scale: float | None = None, mode: int = 0, want_delta: bool = False):
    """Full forward (and backward when ``dout`` is given) of a packed batch.

    ``q``, ``k``, ``v``, ``dout``: ``[N, H, D]`` (float64, or anything ``as_f64``
    takes); ``cu_seqlens``: ``nseq + 1`` sequence offsets (default: one sequence).
    Returns a dict with ``o``, ``dq``, ``dk``, ``dv`` ``[N, H, D]`` and ``lse``
    (and ``delta`` when asked) ``[H, N]``.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    dout = as_f64(dout) if dout is not None else None
    N, H, D = q.shape
    if cu_seqlens is None:
        cu_seqlens = [0, N]
    cu = [int(c) for c in cu_seqlens]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = dict(o=np.zeros((N, H, D)), lse=np.zeros((H, N)))
    if want_delta and dout is not None:
        out["delta"] = np.zeros((H, N))
    if dout is not None:
        out.update(dq=np.zeros((N, H, D)), dk=np.zeros((N, H, D)), dv=np.zeros((N, H, D)))
    for s in range(len(cu) - 1):
        t0, L = cu[s], cu[s + 1] - cu[s]
        if L <= 0:
            continue
        rows = np.arange(L, dtype=np.int32)
        for h in range(H):
            r = head(q, k, v, dout, (t0 * H + h) * D, L, D, H * D, base, scale, mode, rows, rows if dout is not None else [],
                     want_delta=want_delta)
            out["o"][t0:t0 + L, h] = r["o"]
            out["lse"][h, t0:t0 + L] = r["lse"]
            if dout is not None:
                out["dq"][t0:t0 + L, h] = r["dq"]
                out["dk"][t0:t0 + L, h] = r["dk"]
                out["dv"][t0:t0 + L, h] = r["dv"]
                if want_delta:
                    out["delta"][h, t0:t0 + L] = r["delta"]
    return out


def attention_sampled(q, k, v, dout, cu_seqlens, picks, base: float = 10000.0,
                      scale: float | None = None, mode: int = 0):
    """Selected outputs only, for sizes too large for the full oracle.

    ``picks``: list of ``(seq, head, qrows, krows)``; query rows get O, LSE, dq,
    key rows get dk, dv (rows local to the sequence).  Returns a list of dicts in
    the same order.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    dout = as_f64(dout) if dout is not None else None
    N, H, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = [int(c) for c in cu_seqlens]
    res = []
    for (s, h, qrows, krows) in picks:
        t0, L = cu[s], cu[s + 1] - cu[s]
        res.append(head(q, k, v, dout, (t0 * H + h) * D, L, D, H * D, base, scale, mode, qrows,
                        krows if dout is not None else []))
    return res


# ---------------------------------------------------------------- projections

def rmsnorm(x, g, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm of the rows of ``x`` ``[N, C]`` with weight ``g`` ``[C]``."""
    x, g = as_f64(x), as_f64(g)
    N, C = x.shape
    out = np.empty_like(x)
    if _load().ne_oracle_rmsnorm(_dptr(x), _dptr(g), N, C, float(eps), _dptr(out)) != 0:
        raise ValueError("ne_oracle_rmsnorm: bad arguments")
    return out


def linear(a, w) -> np.ndarray:
    """``a [N, K] . w[M, K]^T`` (weights in the [out, in] convention)."""
    a, w = as_f64(a), as_f64(w)
    N, K = a.shape
    M = w.shape[0]
    y = np.empty((N, M))
    if _load().ne_oracle_linear(_dptr(a), _dptr(w), N, K, M, _dptr(y)) != 0:
        raise ValueError("ne_oracle_linear: bad arguments")
    return y


def qkv_rope(x, g, w, B: int, T: int, H: int, D: int = 64, base: float = 10000.0,
             eps: float = 1e-5):
    """QKV projection with RoPE of a fixed-length batch: ``x [B*T, H*D]``,
    ``g [H*D]``, ``w [3*H*D, H*D]``.  Returns ``(q', k', v)``, each ``[B*T, H*D]``."""
    x, g, w = as_f64(x), as_f64(g), as_f64(w)
    C = H * D
    outs = [np.empty((B * T, C)) for _ in range(3)]
    if _load().ne_oracle_qkv_rope(_dptr(x), _dptr(g), _dptr(w), B, T, H, D, float(base),
                                  float(eps), *(_dptr(o) for o in outs)) != 0:
        raise ValueError("ne_oracle_qkv_rope: bad arguments")
    return tuple(outs)


def out_proj_residual(o, w, r) -> np.ndarray:
    """``r + o . w^T`` for ``o``, ``r`` ``[N, C]``, ``w`` ``[C, C]``."""
    o, w, r = as_f64(o), as_f64(w), as_f64(r)
    N, C = o.shape
    y = np.empty((N, C))
    if _load().ne_oracle_out_proj_residual(_dptr(o), _dptr(w), _dptr(r), N, C, _dptr(y)) != 0:
        raise ValueError("ne_oracle_out_proj_residual: bad arguments")
    return y


def mtp_head(h, w, targets, K: int):
    """Multi-token prediction head with softmax cross-entropy: ``h [M, C]``,
    ``w [K*V, C]`` (head j in rows j*V .. j*V+V-1), ``targets [M, K]`` int
    (-1: no target).  Returns ``(loss, row_loss [M, K], dh [M, C], dw [K*V, C])``."""
    h, w = as_f64(h), as_f64(w)
    tg = np.ascontiguousarray(np.asarray(targets, dtype=np.int32))
    M, C = h.shape
    V = w.shape[0] // K
    assert w.shape == (K * V, C) and tg.shape == (M, K)
    loss = np.zeros(1)
    row_loss = np.empty((M, K))
    dh = np.empty((M, C))
    dw = np.empty((K * V, C))
    if _load().ne_oracle_mtp_head(_dptr(h), _dptr(w), _iptr(tg), M, C, K, V, _dptr(loss),
                                  _dptr(row_loss), _dptr(dh), _dptr(dw)) != 0:
        raise ValueError("ne_oracle_mtp_head: bad arguments")
    return float(loss[0]), row_loss, dh, dw

