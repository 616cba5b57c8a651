"""Seeded synthetic inputs, shared by the oracle tests, the CUDA parity tests and the bench.

Every value is a pure function of ``(seed, tensor_id, index)`` (a splitmix64
counter generator feeding Box-Muller in double precision).  This module holds
none of the verify method's arithmetic; it only draws numbers and hands back
numpy arrays.  bf16 tensors are returned as ``uint16`` bit patterns.

Tensor ids are plain integers; :func:`tid` derives stable ids from names so
that every workload recipe reads as ``normal_bf16(seed, tid("layer3.w_in"), ...)``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` with gcc (OpenMP) next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_normal_f64.argtypes = [u64, u64, dbl, dbl, vp, i64]
        lib.synth_normal_f32.argtypes = [u64, u64, dbl, dbl, vp, i64]
        lib.synth_normal_bf16.argtypes = [u64, u64, dbl, dbl, vp, i64]
        lib.synth_uniform_i32.argtypes = [u64, u64, ctypes.c_int32, ctypes.c_int32, vp, i64]
        lib.synth_words.argtypes = [u64, u64, vp, i64]
        _lib = lib
    return _lib


def tid(name: str) -> int:
    """Stable 63-bit tensor id from a name."""
    return int.from_bytes(hashlib.sha256(name.encode()).digest()[:8], "little") >> 1


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal_f64(seed: int, tensor_id: int, shape, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _load().synth_normal_f64(seed, tensor_id, mean, sigma, _ptr(out), out.size)
    return out


def normal_f32(seed: int, tensor_id: int, shape, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, tensor_id, mean, sigma, _ptr(out), out.size)
    return out


def normal_bf16(seed: int, tensor_id: int, shape, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, sigma^2) samples."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, tensor_id, mean, sigma, _ptr(out), out.size)
    return out


def uniform_i32(seed: int, tensor_id: int, shape, lo: int, hi: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.int32)
    _load().synth_uniform_i32(seed, tensor_id, lo, hi, _ptr(out), out.size)
    return out


def words(seed: int, tensor_id: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_words(seed, tensor_id, _ptr(out), n)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
