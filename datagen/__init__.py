"""Seeded synthetic inputs (Philox-4x32-10) shared by the CUDA path and the oracle.

This module holds none of the tensor-relational-algebra arithmetic: it maps
(seed, tensor id, element index) to a number, as documented in ``philox.c``.
Arrays are produced on the host as numpy arrays (fp32 as ``float32``, bf16 as
raw ``uint16`` bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox.c")
_LIB = os.path.join(_HERE, "libdatagen.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``philox.c`` into ``libdatagen.so`` with the host gcc (OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u32, i64, dbl, vp = ctypes.c_uint32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.dg_philox4x32_10.argtypes = [vp, vp, vp]
        for name in ("dg_fill_uniform_f32", "dg_fill_normal_f32", "dg_fill_uniform_bf16", "dg_fill_normal_bf16"):
            getattr(lib, name).argtypes = [u32, u32, i64, dbl, dbl, vp]
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def philox4x32_10(counter, key):
    """One Philox-4x32-10 block: 4 uint32 counter words, 2 uint32 key words -> 4 uint32."""
    lib = _load()
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.dg_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def _fill(name, dtype, shape, seed, tensor, a, b):
    lib = _load()
    out = np.empty(shape, dtype=dtype)
    getattr(lib, name)(seed, tensor, out.size, float(a), float(b), out.ctypes.data)
    return out


def uniform_f32(shape, seed: int, tensor: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    return _fill("dg_fill_uniform_f32", np.float32, shape, seed, tensor, lo, hi)


def normal_f32(shape, seed: int, tensor: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    return _fill("dg_fill_normal_f32", np.float32, shape, seed, tensor, mu, sigma)


def uniform_bf16(shape, seed: int, tensor: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16)."""
    return _fill("dg_fill_uniform_bf16", np.uint16, shape, seed, tensor, lo, hi)


def normal_bf16(shape, seed: int, tensor: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16)."""
    return _fill("dg_fill_normal_bf16", np.uint16, shape, seed, tensor, mu, sigma)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (a bit shift, no arithmetic)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
