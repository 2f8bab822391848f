"""GB300-native packed varlen non-causal attention with a fused q/k prologue.

The compute path is the C-ABI library ``libh3attn.so`` (``include/h3attn.h``,
sources under ``csrc/``); ``h3attn`` is its thin ctypes binding.
"""
from . import build  # noqa: F401
