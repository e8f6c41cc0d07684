"""CPU checks of the boundary: the library builds for sm_103a, loads, and
exports every function include/*.h declares; host-side argument checks return
their status codes before anything touches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ne_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from causal_self_attention_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("ne_attn_fwd", "ne_attn_bwd", "ne_attn_varlen_fwd", "ne_attn_varlen_bwd",
                 "ne_attn_bwd_workspace_bytes", "ne_attn_get_device_status", "ne_status_string",
                 "ne_attn_release"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from causal_self_attention_gb300 import ne_attn
    assert set(_declared()) <= set(ne_attn.EXPORTED)


def test_status_strings_and_workspace(lib):
    lib.ne_status_string.restype = ctypes.c_char_p
    assert lib.ne_status_string(0) == b"NE_OK"
    assert lib.ne_status_string(5) == b"NE_ERR_TIMEOUT"
    lib.ne_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    ws = lib.ne_attn_bwd_workspace_bytes(8192, 12, 64)
    # fp32 dQ' accumulator, fp32 D, bf16 q' and k' (all multiples of 256 here)
    assert ws == 8192 * 12 * 64 * 4 + 8192 * 12 * 4 + 2 * 8192 * 12 * 64 * 2
    assert lib.ne_attn_bwd_workspace_bytes(8192, 12, 128) == 0


def test_argument_errors_return_before_any_launch(lib):
    P = ctypes.c_void_p
    lib.ne_attn_fwd.argtypes = [P, P, P] + [ctypes.c_int] * 4 + [ctypes.c_float] * 2 + [P, P, P]
    fake = P(0x10000)  # never dereferenced: every case below fails its host check first
    # null pointer
    assert lib.ne_attn_fwd(None, fake, fake, 1, 1, 64, 64, 10000.0, 0.125, fake, fake, None) == 1
    # unsupported head dimension
    assert lib.ne_attn_fwd(fake, fake, fake, 1, 1, 64, 128, 10000.0, 0.125, fake, fake, None) == 2
    # non-positive size
    assert lib.ne_attn_fwd(fake, fake, fake, 0, 1, 64, 64, 10000.0, 0.125, fake, fake, None) == 1
    # 2^31 (row, head) pairs: beyond the 32-bit pair indexes of the kernels
    assert lib.ne_attn_fwd(fake, fake, fake, 1, 4096, 1 << 19, 64, 10000.0, 0.125, fake, fake,
                           None) == 1
    # misaligned tensor pointer
    assert lib.ne_attn_fwd(P(0x10002), fake, fake, 1, 1, 64, 64, 10000.0, 0.125, fake, fake,
                           None) == 3
    # bad rope base
    assert lib.ne_attn_fwd(fake, fake, fake, 1, 1, 64, 64, -1.0, 0.125, fake, fake, None) == 1


def test_training_pair_argument_errors_return_before_any_launch(lib):
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.ne_attn_fwd_train.argtypes = [P, P, P, I, I, I, I, F, F, P, P, P, P, P]
    lib.ne_attn_bwd_train.argtypes = [P, P, P, P, P, P, I, I, I, I, F, F, P, P, P, P, Z, P]
    fake = P(0x10000)  # never dereferenced: every case below fails its host check first

    def fwd(qr=fake, kr=fake, base=10000.0):
        return lib.ne_attn_fwd_train(fake, fake, fake, 1, 1, 64, 64, base, 0.125, fake, fake, qr,
                                     kr, None)

    assert fwd(qr=None) == 1          # the rotated outputs are required
    assert fwd(kr=None) == 1
    assert fwd(kr=P(0x10004)) == 3    # and 16-byte aligned
    assert fwd(base=0.0) == 1         # the pass needs a valid rope base

    def bwd(qr=fake, base=10000.0, ws=None, ws_bytes=0):
        return lib.ne_attn_bwd_train(qr, fake, fake, fake, fake, fake, 1, 1, 64, 64, base, 0.125,
                                     fake, fake, fake, ws, ws_bytes, None)

    assert bwd(qr=None) == 1
    assert bwd(base=float("nan")) == 1  # dq, dk are returned un-rotated: the base is used
    assert bwd(ws=fake, ws_bytes=16) == 1


def test_mtp_head_argument_errors_return_before_any_launch(lib):
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.ne_mtp_head.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, Z, P]
    lib.ne_mtp_head_workspace_bytes.argtypes = [I, I, I]
    lib.ne_mtp_head_workspace_bytes.restype = Z
    fake = P(0x10000)  # never dereferenced: every case below fails its host check first

    def call(h=fake, M=300, C=192, K=2, V=256, ws=None, ws_bytes=0):
        return lib.ne_mtp_head(h, fake, fake, M, C, K, V, fake, fake, fake, fake, ws, ws_bytes,
                               None)

    assert call(h=None) == 1
    assert call(M=0) == 1
    assert call(V=512) == 2       # one 256-wide tile per head
    assert call(C=100) == 2       # rows must be 16-byte multiples
    assert call(h=P(0x10008)) == 3
    assert call(ws=fake, ws_bytes=16) == 1
    # dlogits bf16 [M, K*V] rounded up to 256 bytes, then 256 bytes of accumulators
    assert lib.ne_mtp_head_workspace_bytes(300, 2, 256) == 307200 + 256
    assert lib.ne_mtp_head_workspace_bytes(0, 2, 256) == 0


def test_decode_argument_errors_return_before_any_launch(lib):
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.ne_attn_decode.argtypes = [P, P, P, P, I, I, I, I, F, F, P, P, P, Z, P]
    lib.ne_attn_decode_workspace_bytes.restype = Z
    lib.ne_attn_decode_workspace_bytes.argtypes = [I, I, I]
    fake = P(0x10000)  # never dereferenced: every case below fails its host check first

    def call(q=fake, pos=fake, B=2, H=3, Tmax=100, D=64, base=10000.0, scale=0.125, ws=None,
             ws_bytes=0):
        return lib.ne_attn_decode(q, fake, fake, pos, B, H, Tmax, D, base, scale, fake, fake, ws,
                                  ws_bytes, None)

    assert call(q=None) == 1
    assert call(pos=None) == 1
    assert call(D=128) == 2
    assert call(Tmax=0) == 1
    assert call(scale=0.0) == 1
    assert call(q=P(0x10008)) == 3
    assert call(ws=fake, ws_bytes=16) == 1  # too small
    # workspace: one (m, l, o[64]) partial of 68 floats per 256-key chunk per (b, h)
    assert lib.ne_attn_decode_workspace_bytes(2, 3, 1000) == 2 * 3 * 4 * 68 * 4
    assert lib.ne_attn_decode_workspace_bytes(0, 3, 1000) == 0


def test_rotated_decode_argument_errors_return_before_any_launch(lib):
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.ne_attn_decode_rotated.argtypes = [P, P, P, P, I, I, I, I, F, P, P, P, Z, P]
    fake = P(0x10000)  # never dereferenced: every case below fails its host check first

    def call(qr=fake, kr=fake, B=2, H=3, Tmax=100, D=64, scale=0.125, out=fake, ws=None,
             ws_bytes=0):
        return lib.ne_attn_decode_rotated(qr, kr, fake, fake, B, H, Tmax, D, scale, out, fake,
                                          ws, ws_bytes, None)

    assert call(qr=None) == 1
    assert call(kr=None) == 1
    assert call(out=None) == 1
    assert call(D=32) == 2
    assert call(B=0) == 1
    assert call(scale=float("nan")) == 1
    assert call(kr=P(0x10004)) == 3
    assert call(ws=fake, ws_bytes=16) == 1
