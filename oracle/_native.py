"""Loader of the C++ oracle library (test infrastructure, not product).

Compiles ``oracle/tee_oracle.cpp`` with the host C++ compiler into
``oracle/liboracle.so`` when the library is missing or older than its
source (plain ``-O2``, single-threaded, no BLAS, FMA contraction off so that
x86 and Arm hosts give the same float64 results), then binds its entry points
with ctypes. Nothing here computes: every function of the oracle runs in the
C++ library.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tee_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
CXXFLAGS = ["-O3", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-Wall"]
ABI_VERSION = 1

_P = ctypes.c_void_p
_I = ctypes.c_int64
_D = ctypes.c_double
SIGNATURES = {
    "oc_abi_version": (ctypes.c_int, []),
    "oc_cosine_similarity": (None, [_I, _I, _P, _P, _P]),
    "oc_decide": (ctypes.c_int, [_I, _P, _D, ctypes.c_int, _P, _P]),
    "oc_router_probability": (None, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _D, _P]),
    "oc_earliest_exit": (None, [_I, _P, _I, _P, _D, _I, _I, _P]),
    "oc_layer_ops": (_I, [_I, _P]),
    "oc_stable_partition": (None, [_I, _P, _P, _P, _P, _P, _P, _P]),
    "oc_gather_rows": (None, [_I, _I, _P, _P, _P]),
    "oc_exit_scatter": (None, [_I, _I, _P, _P, _P, _P, _D, _P]),
    "oc_dequant_int4": (None, [_I, _I, _I, _P, _P, _P, _P]),
    "oc_rms_norm": (None, [_I, _I, _P, _P, _D, _P]),
    "oc_rope_rotate_half": (None, [_I, _I, _P, _P, _D, _P]),
    "oc_fill_rows": (None, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _D, _D, _P, _P]),
    "oc_ridge_fit": (ctypes.c_int, [_I, _I, _I, _P, _P, _D, _P]),
    "oc_silu": (None, [_I, _P, _P]),
    "oc_attention": (None, [_I, _I, _I, _P, _P, _P, _I, _I, _P, _P, _P]),
    "oc_exit_layer": (None, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P,
                             _D, _D, _P]),
}

_lock = threading.Lock()
_lib = None


def _cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand:
            return cand
    raise RuntimeError("no C++ compiler found: the oracle is C++ and needs one (g++)")


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    """Compile the oracle library if needed; returns its path."""
    if not force and up_to_date():
        return LIB
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([_cxx(), *CXXFLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C++ oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            if L.oc_abi_version() != ABI_VERSION:
                raise RuntimeError("stale oracle library: rebuild oracle/liboracle.so")
            _lib = L
    return _lib


# ---- marshalling helpers

def f64(x) -> np.ndarray:
    """C-contiguous float64 copy (or view) of x; torch tensors are widened exactly."""
    if hasattr(x, "detach"):
        x = x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64, order="C")


def i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64, order="C")


def u8(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.uint8, order="C")


def ptr(a):
    """Address of a contiguous numpy array, or None for None."""
    return None if a is None else ctypes.c_void_p(a.ctypes.data)
