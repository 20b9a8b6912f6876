"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Nothing here computes attention or block metadata: this module only draws
numbers (``gen.c``) and lays them out in the input formats that the
block-sparse forward consumes (``configs.py``).  Both sides of every parity
check take their inputs from here, so they see bit-identical bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libbsgen.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into libbsgen.so next to it (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.tmp.{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11",
                    "-o", tmp, _SRC, "-lm", "-lpthread"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            for name, ptr in (("bsgen_normal_bf16", ctypes.c_void_p),
                              ("bsgen_uniform01", ctypes.c_void_p),
                              ("bsgen_u64", ctypes.c_void_p)):
                fn = getattr(lib, name)
                fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                               ctypes.c_int64, ptr, ctypes.c_int]
                fn.restype = None
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16_into(ptr: int, n: int, seed: int, stream: int, offset: int = 0) -> None:
    """Write n bf16 N(0,1) deviates (as raw uint16 bits) to host address ptr."""
    _load().bsgen_normal_bf16(seed, stream, offset, n, ctypes.c_void_p(ptr), _threads())


def normal_bf16(shape, seed: int, stream: int) -> np.ndarray:
    """bf16 N(0,1) deviates as a uint16 array of raw bf16 bits."""
    out = np.empty(shape, dtype=np.uint16)
    normal_bf16_into(out.ctypes.data, out.size, seed, stream)
    return out


def uniform01(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    _load().bsgen_uniform01(seed, stream, offset, out.size, ctypes.c_void_p(out.ctypes.data),
                            _threads())
    return out


def u64(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.uint64)
    _load().bsgen_u64(seed, stream, offset, out.size, ctypes.c_void_p(out.ctypes.data),
                      _threads())
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits to float32 (a bit shift, no rounding)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


from .configs import CONFIGS, Workload, make_workload  # noqa: E402,F401
