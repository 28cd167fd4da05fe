"""Seeded synthetic inputs shared by the engine's tests, the benchmark and the CPU oracle.

This package draws random numbers (SplitMix64, counter-based; see synth.c) and
arranges them into the shapes of the decoder's inputs.  It holds none of the
decoder's arithmetic: no packing, no dequantisation, no normalisation.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile synth.c into libsynth.so next to it (gcc + OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            u64, i64, i32, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            vp = ctypes.c_void_p
            lib.synth_raw_state.argtypes = [u64, i64, vp]
            lib.synth_raw_state.restype = None
            lib.synth_raw_u64.argtypes = [u64, u64, i64, vp]
            lib.synth_randint_i8.argtypes = [u64, u64, i64, i32, i32, vp]
            lib.synth_randint_i32.argtypes = [u64, u64, i64, i32, i32, vp]
            lib.synth_uniform_f32.argtypes = [u64, u64, i64, f32, f32, vp]
            lib.synth_normal_f32.argtypes = [u64, u64, i64, f32, f32, vp]
            lib.synth_f32_to_bf16.argtypes = [i64, vp, vp]
            lib.synth_permutation.argtypes = [u64, u64, i64, vp]
            for f in (lib.synth_raw_u64, lib.synth_randint_i8, lib.synth_randint_i32,
                      lib.synth_uniform_f32, lib.synth_normal_f32, lib.synth_f32_to_bf16,
                      lib.synth_permutation):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def raw_state(state, n):
    out = np.empty(n, dtype=np.uint64)
    _load().synth_raw_state(state, n, _ptr(out))
    return out


def raw_u64(seed, tid, n):
    out = np.empty(n, dtype=np.uint64)
    _load().synth_raw_u64(seed, tid, n, _ptr(out))
    return out


def randint_i8(seed, tid, n, lo, hi):
    out = np.empty(n, dtype=np.int8)
    _load().synth_randint_i8(seed, tid, n, lo, hi, _ptr(out))
    return out


def randint_i32(seed, tid, n, lo, hi):
    out = np.empty(n, dtype=np.int32)
    _load().synth_randint_i32(seed, tid, n, lo, hi, _ptr(out))
    return out


def uniform_f32(seed, tid, n, a, b):
    out = np.empty(n, dtype=np.float32)
    _load().synth_uniform_f32(seed, tid, n, a, b, _ptr(out))
    return out


def normal_f32(seed, tid, n, mean, std):
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, n, mean, std, _ptr(out))
    return out


def f32_to_bf16(a):
    """Round fp32 values to bfloat16 storage (RNE); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().synth_f32_to_bf16(a.size, _ptr(a), _ptr(out))
    return out


def bf16_to_f32(b):
    """bfloat16 bit patterns -> fp32 values (exact widening)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def permutation(seed, tid, n):
    out = np.empty(n, dtype=np.int32)
    _load().synth_permutation(seed, tid, n, _ptr(out))
    return out
