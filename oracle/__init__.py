"""CPU oracle for the token early-exit step (test infrastructure, not product).

A plain, slow, obviously correct restatement of what the three source pages
define, written as single-threaded C++17 loops in float64
(``oracle/tee_oracle.cpp``: no BLAS, no threads, no SIMD intrinsics), reached
from Python through ctypes by the thin modules of this package, which only
marshal arrays. It covers River-LLM's state-transition cosine gate, TIDE's
RMSNorm router gate with its compaction and exit scatter, RidgeFill's KV fill
(per-layer linear map, that layer's own RMSNorm and K/V projection, RoPE on K,
store into the backbone's cache slot), RidgeFill's closed-form ridge fit, and
River-LLM's Exit River (the W4A16 copies of the remaining decoder layers).
Inputs stored in bf16/fp16/fp32 are widened to float64 exactly; nothing is
rounded on the way except where a page fixes a precision (the exit decision,
taken in fp32 like the kernels the TIDE notes describe).

``oracle.numpy_ref`` is an independent float64 numpy restatement of the same
definitions, kept only so that a test can cross-check the two.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arms may import this package. The CUDA library never calls it,
and it shares no code, table or constant with the CUDA path.

Every function here is pinned by the ``-m "not gpu"`` tests against closed
forms, invariants, brute force and hand-worked examples; none is marked
"parity unpinned".
"""
from .gate import (cosine_similarity, cosine_gate, router_probability, router_gate,
                   earliest_exit, layer_ops)  # noqa: F401
from .compact import stable_partition, gather_rows, exit_scatter  # noqa: F401
from .fill import dequant_int4, rms_norm, rope_rotate_half, fill_rows, kv_fill  # noqa: F401
from .ridge import ridge_fit  # noqa: F401
from .river import silu, attention, exit_layer, exit_river  # noqa: F401
