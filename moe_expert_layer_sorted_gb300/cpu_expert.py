"""Binding of cpu_expert.c: the SwiGLU FFN of one host-resident expert on the
host CPU, the comparison against reading that expert in place over the GPU's
host link.  Not a path of the library (which has no CPU fallback): only the
benchmark's comparison and its test use it."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpu_expert.c")
_LIB = os.path.join(_HERE, "libmoe_cpu_expert.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """gcc -O3 (no fast-math: the compiler may vectorise the independent partial sums only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O3", "-fPIC", "-shared", "-pthread", "-fno-fast-math", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            L.cpu_expert_ffn.argtypes = [P, P, i32, i32, i32, i32, i32, P, i32, P, i32]
            L.cpu_expert_ffn.restype = i32
            _lib = L
    return _lib


def expert_ffn(codes, scales, H: int, I: int, bits: int, group: int, scale_dtype: int,
               x_bf16: np.ndarray, threads: int = 1) -> np.ndarray:
    """o [T][H] fp32 for tokens x_bf16 [T][H] (uint16 bf16 bits); codes/scales: host arrays
    (gate, up, down) in the canonical format."""
    codes = [np.ascontiguousarray(c) for c in codes]
    scales = [np.ascontiguousarray(s) for s in scales]
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    out = np.empty((T, H), dtype=np.float32)
    cp = (ctypes.c_void_p * 3)(*[c.ctypes.data for c in codes])
    sp = (ctypes.c_void_p * 3)(*[s.ctypes.data for s in scales])
    rc = lib().cpu_expert_ffn(cp, sp, H, I, bits, group, scale_dtype, x.ctypes.data, T, out.ctypes.data,
                              int(threads))
    if rc != 0:
        raise ValueError("cpu_expert_ffn: unsupported shape or arguments")
    return out
