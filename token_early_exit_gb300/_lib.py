"""ctypes view of libtee.so (the C ABI declared in include/tee.h).

Loading fails loudly when the library has not been built: there is no
fallback path. Build it with ``python -m token_early_exit_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtee.so")

TEE_OK, TEE_ERR_INVALID_ARG, TEE_ERR_UNSUPPORTED, TEE_ERR_CUDA, TEE_ERR_WORKSPACE, TEE_ERR_DEVICE = range(6)
TEE_F32, TEE_F16, TEE_BF16 = 0, 1, 2
TEE_GATE_COSINE, TEE_GATE_ROUTER = 0, 1
TEE_RULE_PER_TOKEN, TEE_RULE_BATCH_ALL = 0, 1
TEE_W_DENSE, TEE_W_INT4 = 0, 1
(TEE_DEVERR_NONE, TEE_DEVERR_ROW, TEE_DEVERR_POS, TEE_DEVERR_SEQ, TEE_DEVERR_COUNT, TEE_DEVERR_DEST,
 TEE_DEVERR_TIMEOUT) = range(7)
WS_HEADER_BYTES = 256


class GateDesc(ctypes.Structure):
    _fields_ = [("mode", c_int32), ("rule", c_int32), ("dtype", c_int32), ("d", c_int32),
                ("bottleneck", c_int32), ("threshold", c_float), ("eps", c_float)]


TEE_FILL_EARLY_WEIGHTS = 1
TEE_FILL_GENERIC = 2
TEE_RIVER_ATTN_BY_PAIR = 1
TEE_RIVER_ATTN_BY_CHUNK = 2
TEE_FILL_WRITE_K = 1
TEE_FILL_WRITE_V = 2


class FillDesc(ctypes.Structure):
    _fields_ = [("d", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32), ("rope_base", c_float),
                ("eps", c_float), ("dtype", c_int32), ("wfmt", c_int32), ("group", c_int32), ("flags", c_int32)]


class FillLayer(ctypes.Structure):
    _fields_ = [("w_map", c_void_p), ("gamma", c_void_p), ("wk", c_void_p), ("wv", c_void_p),
                ("k_scale", c_void_p), ("k_zero", c_void_p), ("v_scale", c_void_p), ("v_zero", c_void_p),
                ("cache_layer", c_int32), ("writes", c_int32),
                ("k_bias", c_void_p), ("v_bias", c_void_p), ("k_norm", c_void_p)]


class CacheLayout(ctypes.Structure):
    _fields_ = [("s_layer", c_int64), ("s_seq", c_int64), ("s_head", c_int64), ("s_pos", c_int64),
                ("n_layers", c_int32), ("n_seq", c_int32), ("n_heads", c_int32), ("max_pos", c_int32)]


class W4(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scale", c_void_p), ("zero", c_void_p)]


class RiverDesc(ctypes.Structure):
    _fields_ = [("d", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("d_ff", c_int32), ("rope_base", c_float), ("eps", c_float), ("group", c_int32), ("flags", c_int32)]


class RiverLayer(ctypes.Structure):
    _fields_ = [("attn_norm", c_void_p), ("ffn_norm", c_void_p), ("wq", W4), ("wk", W4), ("wv", W4), ("wo", W4),
                ("wg", W4), ("wu", W4), ("wd", W4), ("cache_layer", c_int32), ("reserved", c_int32)]


class StepBuffers(ctypes.Structure):
    _fields_ = [("h_prev", c_void_p), ("h_cur", c_void_p), ("pos", c_void_p), ("seq", c_void_p), ("score", c_void_p),
                ("mask", c_void_p), ("flag", c_void_p), ("cont_rows", c_void_p), ("exit_rows", c_void_p),
                ("cont_pos", c_void_p), ("exit_pos", c_void_p), ("h_cont", c_void_p), ("out", c_void_p),
                ("n_out", c_int64), ("counts", c_void_p), ("ws", c_void_p), ("ws_bytes", c_size_t)]


_P = c_void_p
SIGNATURES = {
    "tee_version": (c_char_p, []),
    "tee_status_string": (c_char_p, [c_int]),
    "tee_last_cuda_error": (c_int, []),
    "tee_workspace_init": (c_int, [_P, c_size_t, _P]),
    "tee_get_device_error": (c_int, [_P, POINTER(c_int32), POINTER(c_int32), _P]),
    "tee_clear_device_error": (c_int, [_P, _P]),
    "tee_check_wait_timeout": (c_int, [_P, ctypes.c_uint32, _P]),
    "tee_launch_count": (ctypes.c_uint64, []),
    "tee_exit_gate_workspace_size": (c_size_t, [POINTER(GateDesc), c_int32]),
    "tee_exit_gate": (c_int, [POINTER(GateDesc), c_int32, _P, c_int64, _P, c_int64, _P, _P, _P, _P, _P,
                              _P, _P, _P, _P, c_size_t, _P]),
    "tee_exit_gate_router_static_max_bytes": (c_size_t, []),
    "tee_exit_gate_router_static": (c_int, [POINTER(GateDesc), c_int32, _P, c_int64, _P, _P, _P, _P, _P, _P, _P,
                                            _P, _P]),
    "tee_exit_gate_router_static_device_error": (c_int, [POINTER(c_int32), POINTER(c_int32), _P]),
    "tee_exit_gate_router_static_clear_error": (c_int, [_P]),
    "tee_exit_compact_workspace_size": (c_size_t, [c_int32]),
    "tee_exit_compact": (c_int, [c_int32, _P, _P, _P, c_int64, c_int32, c_int32, _P, _P, _P, _P, _P, c_int64,
                                 _P, _P, c_size_t, _P]),
    "tee_exit_compact_scatter": (c_int, [c_int32, _P, _P, _P, c_int64, c_int32, c_int32, _P, _P, _P, _P, _P,
                                         c_int64, _P, c_int64, c_int64, _P, _P, c_size_t, _P]),
    "tee_exit_gate_compact_scatter_workspace_size": (c_size_t, [POINTER(GateDesc), c_int32]),
    "tee_exit_gate_compact_scatter": (c_int, [POINTER(GateDesc), c_int32, _P, c_int64, _P, c_int64, _P, _P, _P, _P,
                                              _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, c_int64, _P, c_int64,
                                              c_int64, _P, _P, c_size_t, _P]),
    "tee_ridge_fit_workspace_size": (c_size_t, [c_int32, c_int32, c_int32]),
    "tee_ridge_fit": (c_int, [c_int32, c_int32, c_int32, _P, c_int64, _P, c_int64, c_int32, c_float, _P, c_int64, _P,
                              c_size_t, _P]),
    "tee_exit_river_prep_size": (c_size_t, [POINTER(RiverDesc), c_int32, c_int32]),
    "tee_exit_river_prepare": (c_int, [POINTER(RiverDesc), c_int32, POINTER(RiverLayer), c_int32, _P, c_size_t, _P]),
    "tee_exit_river_workspace_size": (c_size_t, [POINTER(RiverDesc), c_int32, c_int32]),
    "tee_exit_river": (c_int, [POINTER(RiverDesc), c_int32, POINTER(RiverLayer), _P, c_size_t, c_int32, _P, _P,
                               c_int64, c_int32, _P, _P, _P, _P, _P, POINTER(CacheLayout), _P, c_int64, _P,
                               c_size_t, _P]),
    "tee_exit_scatter_workspace_size": (c_size_t, [c_int32]),
    "tee_exit_scatter": (c_int, [c_int32, _P, _P, _P, _P, c_int64, _P, c_int64, c_int64, c_int32, c_int32, _P,
                                 c_float, _P, c_size_t, _P]),
    "tee_decode_step_create": (c_int, [POINTER(GateDesc), c_int32, POINTER(FillDesc), c_int32, POINTER(FillLayer), _P,
                                       c_size_t, _P, _P, POINTER(CacheLayout), POINTER(StepBuffers), POINTER(_P)]),
    "tee_decode_step_run_host": (c_int, [_P, c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "tee_decode_step_destroy": (None, [_P]),
    "tee_kv_fill_prep_size": (c_size_t, [POINTER(FillDesc), c_int32, c_int32]),
    "tee_kv_fill_prepare": (c_int, [POINTER(FillDesc), c_int32, POINTER(FillLayer), c_int32, _P, c_size_t, _P]),
    "tee_kv_fill_workspace_size": (c_size_t, [POINTER(FillDesc), c_int32, c_int32]),
    "tee_kv_fill": (c_int, [POINTER(FillDesc), c_int32, POINTER(FillLayer), _P, c_size_t, c_int32, _P, _P,
                            c_int64, c_int32, _P, _P, c_int32, _P, _P, _P, POINTER(CacheLayout), _P, c_size_t,
                            _P]),
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library with argument types set; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m token_early_exit_gb300.build` "
                           "(the CUDA library is the only implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class TeeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load()
        msg = lib.tee_status_string(status).decode()
        if status == TEE_ERR_CUDA:
            msg += f" (cudaError {lib.tee_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != TEE_OK:
        raise TeeError(fn, status)
