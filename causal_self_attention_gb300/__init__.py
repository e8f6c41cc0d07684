"""GB300-native causal self-attention with fused RoPE (forward and backward).

The compute lives in ``libne_attn.so`` (hand-written sm_103a CUDA behind the C
ABI in ``include/ne_attn.h``); :mod:`causal_self_attention_gb300.ne_attn` is a
thin ctypes binding with the same names, taking torch CUDA tensors for device
memory and streams.  Importing this package does not load the library; the
first call does, and fails loudly if it has not been built.
"""
from .inputs import CONFIGS, CONFIG_NAMES, make_inputs  # noqa: F401

__all__ = ["CONFIGS", "CONFIG_NAMES", "make_inputs"]
