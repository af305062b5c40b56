"""Token-level early exit on one GB300: exit gate, compaction, exit scatter, KV
fill and the Exit River, as hand-written CUDA for sm_103a behind the C ABI in include/tee.h.

The Python side only marshals arguments; see ``ops``.
"""
from . import _lib  # noqa: F401
from .ops import (DecodeStep, ExitRiver, KVFill, Workspace, cache_layout, exit_compact, exit_compact_scatter,  # noqa: F401
                  exit_gate, exit_gate_compact_scatter, exit_scatter, kv_fill, ridge_fit)

__all__ = ["exit_gate", "exit_compact", "exit_compact_scatter", "exit_gate_compact_scatter", "exit_scatter", "ridge_fit", "kv_fill", "KVFill", "ExitRiver", "DecodeStep", "Workspace",
           "cache_layout"]
