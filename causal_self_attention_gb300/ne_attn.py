"""ctypes binding of ``libne_attn.so`` (C ABI: include/ne_attn.h, include/ne_attn_debug.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Torch supplies device memory and streams.  Each
function keeps the C name; tensors replace raw pointers and the sizes are read
from their shapes.  A nonzero status raises :class:`NeAttnError`.  There is no
fallback: if the library is missing, or the device is not an sm_103 GPU, the
call fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

NE_OK = 0
STATUS_NAMES = {0: "NE_OK", 1: "NE_ERR_INVALID_ARG", 2: "NE_ERR_UNSUPPORTED",
                3: "NE_ERR_MISALIGNED", 4: "NE_ERR_CUDA", 5: "NE_ERR_TIMEOUT", 6: "NE_ERR_OOM",
                7: "NE_ERR_BAD_SEQLEN", 8: "NE_ERR_TOO_LARGE"}

EXPORTED = ("ne_attn_fwd", "ne_attn_fwd_f32out", "ne_attn_bwd", "ne_attn_bwd_workspace_bytes",
            "ne_attn_bwd_noalloc", "ne_attn_decode", "ne_attn_decode_rotated",
            "ne_attn_decode_workspace_bytes",
            "ne_attn_varlen_fwd", "ne_attn_varlen_fwd_f32out", "ne_attn_varlen_bwd",
            "ne_attn_set_bwd_phase_events", "ne_attn_get_device_status",
            "ne_attn_last_device_code", "ne_status_string",
            "ne_attn_release", "ne_debug_tma_tile", "ne_debug_rope_tile", "ne_debug_umma",
            "ne_debug_pipeline", "ne_rmsnorm_qkv_rope", "ne_out_proj_residual",
            "ne_attn_fwd_rotated", "ne_attn_bwd_rotated", "ne_attn_fwd_train",
            "ne_attn_bwd_train", "ne_attn_varlen_fwd_train", "ne_attn_varlen_bwd_train",
            "ne_attn_set_fwd_phase_event", "ne_mtp_head", "ne_mtp_head_workspace_bytes",
            "ne_debug_schedule")


class NeAttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load the library (built in-tree by ``causal_self_attention_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m causal_self_attention_gb300.build`")
    L = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "ne_attn_fwd": [P, P, P, I, I, I, I, F, F, P, P, P],
        "ne_attn_fwd_f32out": [P, P, P, I, I, I, I, F, F, P, P, P],
        "ne_attn_bwd": [P, P, P, P, P, P, I, I, I, I, F, F, P, P, P, P, Z, P],
        "ne_attn_bwd_noalloc": [P, P, P, P, P, P, I, I, I, I, F, F, P, P, P, P],
        "ne_attn_varlen_fwd": [P, P, P, P, I, I, I, I, I, F, F, P, P, P],
        "ne_attn_varlen_fwd_f32out": [P, P, P, P, I, I, I, I, I, F, F, P, P, P],
        "ne_attn_varlen_bwd": [P, P, P, P, P, P, P, I, I, I, I, I, F, F, P, P, P, P, Z, P],
        "ne_attn_decode": [P, P, P, P, I, I, I, I, F, F, P, P, P, Z, P],
        "ne_attn_decode_rotated": [P, P, P, P, I, I, I, I, F, P, P, P, Z, P],
        "ne_attn_set_bwd_phase_events": [P, P],
        "ne_attn_get_device_status": [P],
        "ne_attn_last_device_code": [],
        "ne_attn_release": [],
        "ne_debug_tma_tile": [P, I, I, I, I, P, P],
        "ne_debug_rope_tile": [P, I, I, I, I, I, F, P, P],
        "ne_debug_umma": [I, P, P, P, P],
        "ne_debug_pipeline": [P, I, I, I, I, ctypes.c_longlong, P, P],
        "ne_rmsnorm_qkv_rope": [P, P, P, I, I, I, I, F, F, P, P, P, P, P, P],
        "ne_out_proj_residual": [P, P, P, I, I, P, P],
        "ne_attn_fwd_rotated": [P, P, P, I, I, I, I, F, P, P, P],
        "ne_attn_bwd_rotated": [P, P, P, P, P, P, I, I, I, I, F, P, P, P, P, Z, P],
        "ne_attn_fwd_train": [P, P, P, I, I, I, I, F, F, P, P, P, P, P],
        "ne_attn_bwd_train": [P, P, P, P, P, P, I, I, I, I, F, F, P, P, P, P, Z, P],
        "ne_attn_varlen_fwd_train": [P, P, P, P, I, I, I, I, I, F, F, P, P, P, P, P],
        "ne_attn_varlen_bwd_train": [P, P, P, P, P, P, P, I, I, I, I, I, F, F, P, P, P, P, Z,
                                     P],
        "ne_attn_set_fwd_phase_event": [P],
        "ne_mtp_head": [P, P, P, I, I, I, I, P, P, P, P, P, Z, P],
        "ne_debug_schedule": [I, I, I, I, P, I],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = None if name == "ne_attn_release" else I
    L.ne_attn_bwd_workspace_bytes.argtypes = [I, I, I]
    L.ne_attn_bwd_workspace_bytes.restype = Z
    L.ne_mtp_head_workspace_bytes.argtypes = [I, I, I]
    L.ne_mtp_head_workspace_bytes.restype = Z
    L.ne_attn_decode_workspace_bytes.argtypes = [I, I, I]
    L.ne_attn_decode_workspace_bytes.restype = Z
    L.ne_status_string.argtypes = [I]
    L.ne_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(name, rc):
    if rc != NE_OK:
        raise NeAttnError(name, rc)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def ne_status_string(status: int) -> str:
    return lib().ne_status_string(int(status)).decode()


def ne_attn_bwd_workspace_bytes(n_tot: int, H: int, D: int = 64) -> int:
    return int(lib().ne_attn_bwd_workspace_bytes(int(n_tot), int(H), int(D)))


def ne_attn_fwd(q, k, v, rope_base=10000.0, scale=None, out=None, lse=None, out_f32=False,
                stream=None):
    """Forward on ``[B, T, H, 64]`` bf16 tensors.  Returns ``(out, lse)``;
    ``lse`` is ``[B, H, T]`` fp32, ``out`` bf16 (fp32 with ``out_f32``)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, T, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device=q.device)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    fn = lib().ne_attn_fwd_f32out if out_f32 else lib().ne_attn_fwd
    _check("ne_attn_fwd", fn(_ptr(q), _ptr(k), _ptr(v), B, H, T, D, float(rope_base),
                             float(scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def ne_attn_bwd(q, k, v, out, dout, lse, rope_base=10000.0, scale=None, dq=None, dk=None,
                dv=None, workspace=None, stream=None):
    """Backward on ``[B, T, H, 64]`` tensors.  Returns ``(dq, dk, dv)`` (bf16).
    ``workspace``: a CUDA uint8 tensor of ``ne_attn_bwd_workspace_bytes`` bytes,
    or None (stream-ordered temporary inside the library)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, T, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_bwd", lib().ne_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), B, H, T, D,
        float(rope_base), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        ws_bytes, _stream(stream)))
    return dq, dk, dv


def ne_attn_bwd_noalloc(q, k, v, out, dout, lse, rope_base=10000.0, scale=None, dq=None,
                        dk=None, dv=None, stream=None):
    """Backward on ``[B, T, H, 64]`` tensors that allocates no device memory:
    for callers that cannot allocate (the library's fixed scratch array is used
    instead of a workspace; see include/ne_attn.h for its limits and for why
    overlapping calls race).  ``dq``, ``dk``, ``dv`` must be passed in by such
    callers; they are only created here when omitted.  Returns ``(dq, dk, dv)``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, T, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check("ne_attn_bwd_noalloc", lib().ne_attn_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), B, H, T, D,
        float(rope_base), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
    return dq, dk, dv


def ne_attn_varlen_fwd(q, k, v, cu_seqlens, max_seqlen, rope_base=10000.0, scale=None,
                       out=None, lse=None, out_f32=False, stream=None):
    """Forward on packed ``[N_tot, H, 64]`` tensors; ``cu_seqlens`` int32 CUDA
    ``[nseq + 1]``.  Returns ``(out, lse)`` with ``lse`` ``[H, N_tot]``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    N, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device=q.device)
    if lse is None:
        lse = torch.empty((H, N), dtype=torch.float32, device=q.device)
    fn = lib().ne_attn_varlen_fwd_f32out if out_f32 else lib().ne_attn_varlen_fwd
    _check("ne_attn_varlen_fwd", fn(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens),
                                    cu_seqlens.numel() - 1, N, int(max_seqlen), H, D,
                                    float(rope_base), float(scale), _ptr(out), _ptr(lse),
                                    _stream(stream)))
    return out, lse


def ne_attn_varlen_bwd(q, k, v, out, dout, lse, cu_seqlens, max_seqlen, rope_base=10000.0,
                       scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of :func:`ne_attn_varlen_fwd`.  Returns ``(dq, dk, dv)``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    N, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_varlen_bwd", lib().ne_attn_varlen_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, N, int(max_seqlen), H, D, float(rope_base), float(scale),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, _stream(stream)))
    return dq, dk, dv


def ne_attn_fwd_rotated(qr, kr, v, scale=None, out=None, lse=None, stream=None):
    """Forward on pre-rotated ``q' = R(m) q``, ``k' = R(n) k`` (``[B, T, H, 64]``
    bf16).  Returns ``(out, lse)``."""
    for t, n in ((qr, "qr"), (kr, "kr"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, T, H, D = qr.shape
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(qr) if out is None else out
    lse = torch.empty((B, H, T), dtype=torch.float32, device=qr.device) if lse is None else lse
    _check("ne_attn_fwd_rotated", lib().ne_attn_fwd_rotated(
        _ptr(qr), _ptr(kr), _ptr(v), B, H, T, D, float(scale), _ptr(out), _ptr(lse),
        _stream(stream)))
    return out, lse


def ne_attn_bwd_rotated(qr, kr, v, out, dout, lse, scale=None, dqr=None, dkr=None, dv=None,
                        workspace=None, stream=None):
    """Backward of :func:`ne_attn_fwd_rotated`.  Returns ``(dqr, dkr, dv)``: the
    gradients w.r.t. q', k' (the rotated frame) and v."""
    for t, n in ((qr, "qr"), (kr, "kr"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, T, H, D = qr.shape
    scale = D ** -0.5 if scale is None else scale
    dqr = torch.empty_like(qr) if dqr is None else dqr
    dkr = torch.empty_like(kr) if dkr is None else dkr
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_bwd_rotated", lib().ne_attn_bwd_rotated(
        _ptr(qr), _ptr(kr), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), B, H, T, D, float(scale),
        _ptr(dqr), _ptr(dkr), _ptr(dv), _ptr(workspace), ws_bytes, _stream(stream)))
    return dqr, dkr, dv


def ne_rmsnorm_qkv_rope(x, g, w_qkv, T, eps=1e-5, rope_base=10000.0, x_norm=None, rstd=None,
                        q=None, k=None, v=None, stream=None):
    """RMSNorm of ``x`` (``[B*T, C]`` bf16, rows of B sequences of T tokens,
    C = H*64) with weight ``g`` (``[C]`` bf16), then the QKV projection with
    ``w_qkv`` (``[3C, C]`` bf16, [out, in]) and RoPE on q and k in the GEMM's
    epilogue.  Returns ``(q', k', v, x_norm, rstd)``: q', k', v ``[B, T, H, 64]``
    bf16 (the attention's layout), ``x_norm`` ``[B*T, C]`` bf16, ``rstd``
    ``[B*T]`` fp32."""
    for t, n in ((x, "x"), (g, "g"), (w_qkv, "w_qkv")):
        _need(t, torch.bfloat16, n)
    M, C = x.shape
    B, H = M // T, C // 64
    if B * T != M or H * 64 != C or tuple(w_qkv.shape) != (3 * C, C) or g.numel() != C:
        raise ValueError("shapes: x [B*T, H*64], g [H*64], w_qkv [3*H*64, H*64]")
    dev = x.device
    x_norm = torch.empty_like(x) if x_norm is None else x_norm
    rstd = torch.empty(M, dtype=torch.float32, device=dev) if rstd is None else rstd
    q = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device=dev) if q is None else q
    k = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device=dev) if k is None else k
    v = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device=dev) if v is None else v
    _check("ne_rmsnorm_qkv_rope", lib().ne_rmsnorm_qkv_rope(
        _ptr(x), _ptr(g), _ptr(w_qkv), B, T, H, 64, float(eps), float(rope_base), _ptr(x_norm),
        _ptr(rstd), _ptr(q), _ptr(k), _ptr(v), _stream(stream)))
    return q, k, v, x_norm, rstd


def ne_out_proj_residual(o, w_o, residual, y=None, stream=None):
    """``y = residual + o . w_o^T`` for ``o``, ``residual`` ``[N, C]`` bf16 and
    ``w_o`` ``[C, C]`` bf16 ([out, in]).  Returns ``y`` ``[N, C]`` bf16."""
    for t, n in ((o, "o"), (w_o, "w_o"), (residual, "residual")):
        _need(t, torch.bfloat16, n)
    N, C = o.shape
    if tuple(w_o.shape) != (C, C) or tuple(residual.shape) != (N, C):
        raise ValueError("shapes: o, residual [N, C], w_o [C, C]")
    y = torch.empty_like(residual) if y is None else y
    _check("ne_out_proj_residual", lib().ne_out_proj_residual(
        _ptr(o), _ptr(w_o), _ptr(residual), N, C, _ptr(y), _stream(stream)))
    return y


def ne_mtp_head_workspace_bytes(M: int, K: int, V: int = 256) -> int:
    return int(lib().ne_mtp_head_workspace_bytes(M, K, V))


def ne_mtp_head(h, w, targets, K, loss=None, row_loss=None, dh=None, dw=None, workspace=None,
                stream=None):
    """Multi-token prediction head with softmax cross-entropy: ``h [M, C]``
    bf16, ``w [K*256, C]`` bf16, ``targets [M, K]`` int32 (-1: no target).
    Returns ``(loss [1], row_loss [M, K], dh [M, C] bf16, dw [K*256, C] fp32)``."""
    _need(h, torch.bfloat16, "h")
    _need(w, torch.bfloat16, "w")
    _need(targets, torch.int32, "targets")
    M, C = h.shape
    V = w.shape[0] // K
    loss = torch.empty(1, dtype=torch.float32, device=h.device) if loss is None else loss
    row_loss = (torch.empty((M, K), dtype=torch.float32, device=h.device) if row_loss is None
                else row_loss)
    dh = torch.empty_like(h) if dh is None else dh
    dw = torch.empty((K * V, C), dtype=torch.float32, device=h.device) if dw is None else dw
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_mtp_head", lib().ne_mtp_head(
        _ptr(h), _ptr(w), _ptr(targets), M, C, K, V, _ptr(loss), _ptr(row_loss), _ptr(dh),
        _ptr(dw), _ptr(workspace), ws_bytes, _stream(stream)))
    return loss, row_loss, dh, dw


def ne_attn_decode_workspace_bytes(B: int, H: int, Tmax: int) -> int:
    return int(lib().ne_attn_decode_workspace_bytes(int(B), int(H), int(Tmax)))


def ne_attn_decode(q, k_cache, v_cache, pos, rope_base=10000.0, scale=None, out=None, lse=None,
                   workspace=None, stream=None):
    """Decode attention: ``q`` ``[B, H, 64]`` bf16 (the new tokens), ``k_cache``
    / ``v_cache`` ``[B, Tmax, H, 64]`` bf16 (un-rotated), ``pos`` int32 ``[B]``
    on the device (each new token's position; rows 0..pos[b] are attended).
    Returns ``(out [B, H, 64] bf16, lse [B, H] fp32)``."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(pos, torch.int32, "pos")
    B, H, D = q.shape
    Tmax = k_cache.shape[1]
    if tuple(k_cache.shape) != (B, Tmax, H, D) or tuple(v_cache.shape) != (B, Tmax, H, D):
        raise ValueError("k_cache / v_cache must be [B, Tmax, H, D] matching q")
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_decode",
           lib().ne_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos), B, H, Tmax, D,
                                float(rope_base), float(scale), _ptr(out), _ptr(lse),
                                _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse


def ne_attn_decode_rotated(qr, kr_cache, v_cache, pos, scale=None, out=None, lse=None,
                           workspace=None, stream=None):
    """Decode over a cache of rotated keys: ``qr`` ``[B, H, 64]`` bf16 (the new
    tokens' ``q' = R(pos) q``), ``kr_cache`` ``[B, Tmax, H, 64]`` bf16 holding
    ``k'_n = R(n) k_n``, ``v_cache`` likewise, ``pos`` int32 ``[B]`` on the
    device.  Returns ``(out [B, H, 64] bf16, lse [B, H] fp32)``."""
    _need(qr, torch.bfloat16, "qr")
    _need(kr_cache, torch.bfloat16, "kr_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(pos, torch.int32, "pos")
    B, H, D = qr.shape
    Tmax = kr_cache.shape[1]
    if tuple(kr_cache.shape) != (B, Tmax, H, D) or tuple(v_cache.shape) != (B, Tmax, H, D):
        raise ValueError("kr_cache / v_cache must be [B, Tmax, H, D] matching qr")
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(qr) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=qr.device) if lse is None else lse
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_decode_rotated",
           lib().ne_attn_decode_rotated(_ptr(qr), _ptr(kr_cache), _ptr(v_cache), _ptr(pos), B, H,
                                        Tmax, D, float(scale), _ptr(out), _ptr(lse),
                                        _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse


def ne_attn_fwd_train(q, k, v, rope_base=10000.0, scale=None, out=None, lse=None, qr=None,
                      kr=None, stream=None):
    """Training forward on ``[B, T, H, 64]`` bf16 tensors: as :func:`ne_attn_fwd`,
    and also returns the rotated operands it computed once, for the backward.
    Returns ``(out, lse, qr, kr)``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, T, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    qr = torch.empty_like(q) if qr is None else qr
    kr = torch.empty_like(k) if kr is None else kr
    _check("ne_attn_fwd_train", lib().ne_attn_fwd_train(
        _ptr(q), _ptr(k), _ptr(v), B, H, T, D, float(rope_base), float(scale), _ptr(out),
        _ptr(lse), _ptr(qr), _ptr(kr), _stream(stream)))
    return out, lse, qr, kr


def ne_attn_bwd_train(qr, kr, v, out, dout, lse, rope_base=10000.0, scale=None, dq=None,
                      dk=None, dv=None, workspace=None, stream=None):
    """Backward of :func:`ne_attn_fwd_train` from its ``qr``, ``kr``.  Returns
    ``(dq, dk, dv)``: gradients w.r.t. the un-rotated q, k and v."""
    for t, n in ((qr, "qr"), (kr, "kr"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, T, H, D = qr.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(qr) if dq is None else dq
    dk = torch.empty_like(kr) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_bwd_train", lib().ne_attn_bwd_train(
        _ptr(qr), _ptr(kr), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), B, H, T, D,
        float(rope_base), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        ws_bytes, _stream(stream)))
    return dq, dk, dv


def ne_attn_varlen_fwd_train(q, k, v, cu_seqlens, max_seqlen, rope_base=10000.0, scale=None,
                             out=None, lse=None, qr=None, kr=None, stream=None):
    """Training forward on packed ``[N_tot, H, 64]`` tensors.  Returns
    ``(out, lse, qr, kr)`` with ``lse`` ``[H, N_tot]``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    N, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    qr = torch.empty_like(q) if qr is None else qr
    kr = torch.empty_like(k) if kr is None else kr
    _check("ne_attn_varlen_fwd_train", lib().ne_attn_varlen_fwd_train(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), cu_seqlens.numel() - 1, N, int(max_seqlen),
        H, D, float(rope_base), float(scale), _ptr(out), _ptr(lse), _ptr(qr), _ptr(kr),
        _stream(stream)))
    return out, lse, qr, kr


def ne_attn_varlen_bwd_train(qr, kr, v, out, dout, lse, cu_seqlens, max_seqlen,
                             rope_base=10000.0, scale=None, dq=None, dk=None, dv=None,
                             workspace=None, stream=None):
    """Backward of :func:`ne_attn_varlen_fwd_train`.  Returns ``(dq, dk, dv)``."""
    for t, n in ((qr, "qr"), (kr, "kr"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    N, H, D = qr.shape
    scale = D ** -0.5 if scale is None else scale
    dq = torch.empty_like(qr) if dq is None else dq
    dk = torch.empty_like(kr) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ne_attn_varlen_bwd_train", lib().ne_attn_varlen_bwd_train(
        _ptr(qr), _ptr(kr), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, N, int(max_seqlen), H, D, float(rope_base), float(scale),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, _stream(stream)))
    return dq, dk, dv


def ne_attn_set_fwd_phase_event(ev_after_rotation=None) -> None:
    """Record the given torch.cuda.Event between the rotation pass and the
    attention kernel of every following forward that runs such a pass (None: off)."""
    a = ctypes.c_void_p(ev_after_rotation.cuda_event) if ev_after_rotation else None
    _check("ne_attn_set_fwd_phase_event", lib().ne_attn_set_fwd_phase_event(a))


def ne_attn_set_bwd_phase_events(ev_after_preprocess=None, ev_after_main=None) -> None:
    """Record the given torch.cuda.Event objects after the backward's
    preprocess and main kernels of every following backward call (None: off)."""
    a = ctypes.c_void_p(ev_after_preprocess.cuda_event) if ev_after_preprocess else None
    b = ctypes.c_void_p(ev_after_main.cuda_event) if ev_after_main else None
    _check("ne_attn_set_bwd_phase_events", lib().ne_attn_set_bwd_phase_events(a, b))


def ne_attn_get_device_status(stream=None) -> int:
    """Synchronize the stream; return (and clear) the device status code."""
    return int(lib().ne_attn_get_device_status(_stream(stream)))


def ne_attn_last_device_code() -> int:
    return int(lib().ne_attn_last_device_code())


def ne_attn_release() -> None:
    lib().ne_attn_release()


# ------------------------------------------------------------- bring-up entries

def ne_debug_tma_tile(src, h, row0, stream=None):
    """Raw 16 KiB shared-memory image of one TMA-loaded tile (uint8 CUDA tensor)."""
    _need(src, torch.bfloat16, "src")
    n, H, _ = src.shape
    dst = torch.empty(16384, dtype=torch.uint8, device=src.device)
    _check("ne_debug_tma_tile", lib().ne_debug_tma_tile(_ptr(src), n, H, h, row0, _ptr(dst),
                                                        _stream(stream)))
    return dst


def ne_debug_rope_tile(src, h, row0, pos0, rope_base=10000.0, stream=None):
    """The tile after the kernels' in-smem RoPE, un-swizzled: ``[128, 64]`` bf16."""
    _need(src, torch.bfloat16, "src")
    n, H, _ = src.shape
    dst = torch.empty((128, 64), dtype=torch.bfloat16, device=src.device)
    _check("ne_debug_rope_tile", lib().ne_debug_rope_tile(_ptr(src), n, H, h, row0, pos0,
                                                          float(rope_base), _ptr(dst),
                                                          _stream(stream)))
    return dst


def ne_debug_umma(form, a, b, stream=None):
    """One tcgen05 MMA chain; see include/ne_attn_debug.h for the three forms."""
    _need(a, torch.bfloat16, "a")
    _need(b, torch.bfloat16, "b")
    d = torch.empty((128, 128 if form == 0 else 64), dtype=torch.float32, device=a.device)
    _check("ne_debug_umma", lib().ne_debug_umma(int(form), _ptr(a), _ptr(b), _ptr(d),
                                                _stream(stream)))
    return d


def ne_debug_schedule(nseq, H, T, G):
    """The persistent backward's work schedule for a fixed-length batch (host
    only): ``(offsets [G + 1], units)`` as lists, or None when the snake order
    is kept."""
    n = nseq * H * ((T + 127) // 128)
    buf = (ctypes.c_int * (G + 1 + n))()
    m = lib().ne_debug_schedule(int(nseq), int(H), int(T), int(G), buf, len(buf))
    if m < 0:
        raise NeAttnError("ne_debug_schedule", 1)
    if m == 0:
        return None
    return list(buf[:G + 1]), list(buf[G + 1:m])


def ne_debug_pipeline(src, n_items, drop_item=-1, wait_limit_cycles=2_000_000_000, stream=None):
    """Run the bounded-wait pipeline of include/ne_attn_debug.h on ``src``
    (``[n, H, 64]`` bf16).  Returns ``d`` ``[128, 128]`` fp32 (left unwritten
    when the pipeline aborted; read the status with ne_attn_get_device_status)."""
    _need(src, torch.bfloat16, "src")
    n, H, _ = src.shape
    d = torch.zeros((128, 128), dtype=torch.float32, device=src.device)
    _check("ne_debug_pipeline", lib().ne_debug_pipeline(_ptr(src), n, H, int(n_items),
                                                        int(drop_item), int(wait_limit_cycles),
                                                        _ptr(d), _stream(stream)))
    return d
