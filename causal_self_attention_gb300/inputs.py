"""Seeded synthetic inputs for causal RoPE self-attention.

This module holds no arithmetic of the attention method: it only draws random
numbers.  It is the one module that both the CUDA path's tests/benchmark and the
CPU oracle's callers use, so that both sides see the same bytes.

Workloads (the pages name no dataset; these synthetic N(0,1) tensors stand in
for the GPT-2-small training shape -- 12 heads, width 768, so head dimension
64 -- on the techinfos.ro NanoEuler article, section "Arhitectură și tehnologii
folosite", and for the byte-level long contexts of "Tiny Hackable CUDA",
section 1):

=========  =====================================  ====================================
name       shape                                   notes
=========  =====================================  ====================================
tiny       B=1, H=2, T=64, D=64                    oracle-sized check
gpt2s      B=8, H=12, T=1024, D=64                 GPT-2-small training shape
byte4k     B=2, H=12, T=4096, D=64                 q and k scaled by 2.0 (sharper softmax)
long16k    B=1, H=12, T=16384, D=64                long-sequence stress
varlen     32 sequences, L ~ U[64, 2048], H=12     packed with cu_seqlens
=========  =====================================  ====================================

Decode workloads (one new token per sequence against a KV cache, the
generation path of the NanoEuler Show HN page and "Tiny Hackable CUDA",
section 7): ``make_decode`` draws q ``[B, H, D]`` and the un-rotated caches
``[B, Tmax, H, D]`` (N(0,1), bf16) from ``manual_seed(2000 + index)`` in the
order q, k, v; ``pos`` holds each sequence's position (the last cache row
unless given).

==========  ==============================  ============================
decode1k    B=8, H=12, Tmax=1024, D=64      end of a GPT-2-small context
decode16k   B=8, H=12, Tmax=16384, D=64     end of a long byte-level context
==========  ==============================  ============================

Recipe: ``torch.Generator('cpu').manual_seed(1000 + index)``; draw order:
sequence lengths (varlen only, ``randint(64, 2049, (32,))``), then q, k, v, dO as
float32 ``randn``, each rounded to bf16 (round to nearest even).  byte4k
multiplies q and k by 2.0 before rounding, which is exact.  Fixed-length
tensors are ``[B, T, H, D]``; varlen tensors are ``[N_tot, H, D]`` with int32
``cu_seqlens`` of length ``nseq + 1``.
"""
from __future__ import annotations

import torch

CONFIG_NAMES = ("tiny", "gpt2s", "byte4k", "long16k", "varlen")

CONFIGS = {
    "tiny": dict(B=1, H=2, T=64, D=64, qk_mult=1.0),
    "gpt2s": dict(B=8, H=12, T=1024, D=64, qk_mult=1.0),
    "byte4k": dict(B=2, H=12, T=4096, D=64, qk_mult=2.0),
    "long16k": dict(B=1, H=12, T=16384, D=64, qk_mult=1.0),
    "varlen": dict(nseq=32, H=12, D=64, lmin=64, lmax=2048, qk_mult=1.0),
}

DECODE_NAMES = ("decode1k", "decode16k")
DECODE_CONFIGS = {
    "decode1k": dict(B=8, H=12, Tmax=1024, D=64),
    "decode16k": dict(B=8, H=12, Tmax=16384, D=64),
}

ROPE_BASE = 10000.0


def seed_of(name: str) -> int:
    return 1000 + CONFIG_NAMES.index(name)


def make_inputs(name: str, seed: int | None = None) -> dict:
    """Draw the inputs of workload ``name`` on the CPU.

    Returns a dict with bf16 CPU tensors ``q``, ``k``, ``v``, ``dout``; for
    fixed-length workloads also ``B``, ``T``; for varlen ``cu_seqlens``
    (int32 CPU tensor), ``lengths``, ``max_seqlen``; and ``H``, ``D``,
    ``scale`` (1/sqrt(D)), ``rope_base``.
    """
    cfg = CONFIGS[name]
    g = torch.Generator("cpu").manual_seed(seed_of(name) if seed is None else seed)
    H, D = cfg["H"], cfg["D"]
    out = dict(name=name, H=H, D=D, scale=1.0 / D ** 0.5, rope_base=ROPE_BASE)
    if name == "varlen":
        lengths = torch.randint(cfg["lmin"], cfg["lmax"] + 1, (cfg["nseq"],), generator=g)
        cu = torch.zeros(cfg["nseq"] + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
        shape = (int(cu[-1]), H, D)
        out.update(cu_seqlens=cu, lengths=[int(x) for x in lengths],
                   max_seqlen=int(lengths.max()))
    else:
        shape = (cfg["B"], cfg["T"], H, D)
        out.update(B=cfg["B"], T=cfg["T"])
    for key in ("q", "k", "v", "dout"):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if key in ("q", "k") and cfg["qk_mult"] != 1.0:
            x = x * cfg["qk_mult"]
        out[key] = x.to(torch.bfloat16)
    return out


def make_custom(B: int, T: int, H: int, D: int = 64, seed: int = 0, qk_mult: float = 1.0,
                lengths=None) -> dict:
    """Same recipe for an arbitrary shape (edge-case tests).  With ``lengths``
    the tensors are packed ``[sum(lengths), H, D]`` and ``B``/``T`` are ignored."""
    g = torch.Generator("cpu").manual_seed(seed)
    out = dict(name="custom", H=H, D=D, scale=1.0 / D ** 0.5, rope_base=ROPE_BASE)
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths), 0).to(torch.int32)
        shape = (int(cu[-1]), H, D)
        out.update(cu_seqlens=cu, lengths=lengths, max_seqlen=max(lengths) if lengths else 0)
    else:
        shape = (B, T, H, D)
        out.update(B=B, T=T)
    for key in ("q", "k", "v", "dout"):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if key in ("q", "k") and qk_mult != 1.0:
            x = x * qk_mult
        out[key] = x.to(torch.bfloat16)
    return out


def make_decode(name: str | None = None, B: int = 0, H: int = 0, Tmax: int = 0, D: int = 64,
                positions=None, seed: int | None = None) -> dict:
    """Inputs of a decode step: ``q`` ``[B, H, D]``, ``k_cache``/``v_cache``
    ``[B, Tmax, H, D]`` (bf16, CPU) and ``pos`` (int32 ``[B]``, CPU).  Either a
    named workload or explicit sizes; ``positions`` defaults to Tmax - 1."""
    if name is not None:
        cfg = DECODE_CONFIGS[name]
        B, H, Tmax, D = cfg["B"], cfg["H"], cfg["Tmax"], cfg["D"]
        seed = 2000 + DECODE_NAMES.index(name) if seed is None else seed
    g = torch.Generator("cpu").manual_seed(0 if seed is None else seed)
    out = dict(name=name or "custom", B=B, H=H, Tmax=Tmax, D=D, scale=1.0 / D ** 0.5,
               rope_base=ROPE_BASE)
    out["q"] = torch.randn((B, H, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    for key in ("k_cache", "v_cache"):
        out[key] = torch.randn((B, Tmax, H, D), generator=g,
                               dtype=torch.float32).to(torch.bfloat16)
    if positions is None:
        positions = [Tmax - 1] * B
    out["pos"] = torch.tensor([int(x) for x in positions], dtype=torch.int32)
    return out
