"""Seeded synthetic inputs (counter-based SplitMix64 + Irwin-Hall normals).

Shared by the tests, the benchmark and the oracle's callers.  Holds no MoE
arithmetic: only random draws, bf16 rounding of the drawn values and the
workload shapes.  The C source is ``synth/synth.c``; it is compiled on first
use (or by ``__graft_entry__.build()``) into ``synth/libsynth.so``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_SRC_GPU = os.path.join(_HERE, "synth_gpu.cu")
_LIB_GPU = os.path.join(_HERE, "libsynth_gpu.so")
_lock = threading.Lock()
_lib = None
_lib_gpu = None

# stream tags: the first element of every stream key
TAG_WEIGHT = 1   # (layer, expert, matrix 0=gate 1=up 2=down)
TAG_ROUTER = 2   # (layer)
TAG_BIAS = 3     # (layer)
TAG_X = 4        # (step, layer)
TAG_NOISE = 5    # (step, layer)
TAG_DRIFT = 6    # (step, layer)


def build(force: bool = False) -> str:
    """Compile libsynth.so with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def build_gpu(force: bool = False) -> str:
    """Compile the device twin of the normal draws (synth_gpu.cu) with nvcc."""
    if force or not os.path.exists(_LIB_GPU) or os.path.getmtime(_LIB_GPU) < os.path.getmtime(_SRC_GPU):
        cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC",
               "-shared", "-o", _LIB_GPU + ".tmp", _SRC_GPU]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_GPU + ".tmp", _LIB_GPU)
    return _LIB_GPU


def lib_gpu():
    global _lib_gpu
    with _lock:
        if _lib_gpu is None:
            build_gpu()
            L = ctypes.CDLL(_LIB_GPU)
            u64, i64 = ctypes.c_uint64, ctypes.c_int64
            for f in (L.synth_gpu_normal_f32, L.synth_gpu_normal_bf16):
                f.argtypes = [u64, u64, i64, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
                f.restype = ctypes.c_int
            L.synth_gpu_residual_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_void_p,
                                                  ctypes.c_void_p]
            L.synth_gpu_residual_bf16.restype = ctypes.c_int
            _lib_gpu = L
    return _lib_gpu


def normal_f32_device(k: int, n: int, sigma: float, out_ptr: int, stream_ptr: int = 0, start: int = 0):
    """The same draws as normal_f32, written by a GPU kernel into device memory."""
    rc = lib_gpu().synth_gpu_normal_f32(k, start, n, sigma, out_ptr, stream_ptr)
    if rc:
        raise RuntimeError(f"synth_gpu_normal_f32 failed ({rc})")


def normal_bf16_device(k: int, n: int, sigma: float, out_ptr: int, stream_ptr: int = 0, start: int = 0):
    rc = lib_gpu().synth_gpu_normal_bf16(k, start, n, sigma, out_ptr, stream_ptr)
    if rc:
        raise RuntimeError(f"synth_gpu_normal_bf16 failed ({rc})")


def residual_bf16_device(y_ptr: int, noise_ptr: int, n: int, out_ptr: int, stream_ptr: int = 0):
    """out = bf16(float(y) + noise) on the device (bf16 y, fp32 noise, n elements): the
    next layer's input of the chained-layer workloads, one kernel on `stream_ptr`."""
    rc = lib_gpu().synth_gpu_residual_bf16(y_ptr, noise_ptr, n, out_ptr, stream_ptr)
    if rc:
        raise RuntimeError(f"synth_gpu_residual_bf16 failed ({rc})")


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
            L.synth_key.restype = u64
            L.synth_key.argtypes = [u64] * 5
            L.synth_draw.restype = u64
            L.synth_draw.argtypes = [u64, u64]
            L.synth_normal_f32.argtypes = [u64, u64, i64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
            L.synth_normal_bf16.argtypes = [u64, u64, i64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
            L.synth_permutation.argtypes = [u64, i32, ctypes.c_void_p]
            L.synth_zipf_bias.argtypes = [u64, i32, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p]
            _lib = L
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def key(seed: int, tag: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    return int(lib().synth_key(seed, tag, a, b, c))


def normal_f32(k: int, n: int, sigma: float, start: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    lib().synth_normal_f32(k, start, n, sigma, out.ctypes.data, _threads())
    return out


def normal_bf16(k: int, n: int, sigma: float, start: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0,1) draws, rounded to nearest even."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    lib().synth_normal_bf16(k, start, n, sigma, out.ctypes.data, _threads())
    return out


def permutation(k: int, n: int) -> np.ndarray:
    pi = np.empty(n, dtype=np.int32)
    lib().synth_permutation(k, n, pi.ctypes.data)
    return pi


def zipf_bias(k: int, n: int, s: float) -> tuple[np.ndarray, np.ndarray]:
    """(bias[e] = log p_rank(e), rank[e]) for a Zipf(s) popularity law over n experts."""
    bias = np.empty(n, dtype=np.float32)
    rank = np.empty(n, dtype=np.int32)
    lib().synth_zipf_bias(k, n, s, bias.ctypes.data, rank.ctypes.data)
    return bias, rank


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)
