"""CPU oracle of the tiered MoE layer (ctypes wrapper over ``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Imported by tests/, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg; the library never imports it, and it
never imports the library.  See ``moe_oracle.c`` for the definitions each
function follows and the passages they cite.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SC_F32, SC_BF16, SC_F16 = 0, 1, 2
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile liboracle.so: IEEE fp32/fp64, no fast-math, no FMA contraction
    (fmaf in the router logits is explicit)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class _Expert(ctypes.Structure):
    _fields_ = [("codes", _P * 3), ("scales", _P * 3)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            i32, i64 = ctypes.c_int, ctypes.c_int64
            L.oracle_quantize.argtypes = [_P, i32, i32, i32, i32, i32, _P, _P]
            L.oracle_dequantize.argtypes = [_P, _P, i32, i32, i32, i32, i32, _P]
            L.oracle_router_logits.argtypes = [_P, i32, i32, _P, i32, _P, _P]
            L.oracle_topk.argtypes = [_P, i32, i32, i32, _P, _P]
            L.oracle_topk.restype = None
            L.oracle_permute.argtypes = [_P, i32, i32, i32, _P, _P, _P, _P]
            L.oracle_permute.restype = None
            L.oracle_expert_ffn.argtypes = [_P, _P, _P, i32, i32, _P, _P]
            L.oracle_expert_ffn.restype = None
            L.oracle_layer_forward.argtypes = [ctypes.POINTER(_Expert), i32, i32, i32, i32, i32,
                                               i32, i32, _P, i32, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _P, _P]
            L.oracle_layer_forward_tokens.argtypes = [ctypes.POINTER(_Expert), i32, i32, i32, i32,
                                                      i32, i32, i32, _P, i32, _P, _P, _P, i32, _P]
            L.oracle_cache_sim.argtypes = [i32, i32, i64, i32, _P, i32, i32, _P, _P, _P, _P, _P]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def scale_itemsize(dtype: int) -> int:
    return 4 if dtype == SC_F32 else 2


def quantize(w: np.ndarray, bits: int, group: int, dtype: int):
    """fp32 [rows][cols] -> (canonical packed codes uint8, scales [rows][cols/group] raw)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    codes = np.zeros(rows * cols * bits // 8, dtype=np.uint8)
    scales = np.zeros(rows * (cols // group), dtype=np.float32 if dtype == SC_F32 else np.uint16)
    rc = lib().oracle_quantize(_ptr(w), rows, cols, bits, group, dtype, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError(f"oracle_quantize failed ({rc})")
    return codes, scales.reshape(rows, cols // group)


def dequantize(codes, scales, rows: int, cols: int, bits: int, group: int, dtype: int) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float32)
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rc = lib().oracle_dequantize(_ptr(codes), _ptr(scales), rows, cols, bits, group, dtype, _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequantize failed ({rc})")
    return out


def router_logits(x_bf16: np.ndarray, wr_bf16: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    wr = np.ascontiguousarray(wr_bf16, dtype=np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    if lib().oracle_router_logits(_ptr(x), T, H, _ptr(wr), E, _ptr(b), _ptr(out)):
        raise ValueError("router logits need H % 256 == 0")
    return out


def topk(logits: np.ndarray, k: int):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().oracle_topk(_ptr(lg), T, E, k, _ptr(idx), _ptr(w))
    return idx, w


def permute(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    lib().oracle_permute(_ptr(idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv))
    return counts, offsets, perm, inv


def expert_ffn(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, x: np.ndarray) -> np.ndarray:
    wg = np.ascontiguousarray(wg, dtype=np.float32)
    wu = np.ascontiguousarray(wu, dtype=np.float32)
    wd = np.ascontiguousarray(wd, dtype=np.float32)
    I, H = wg.shape
    xd = np.ascontiguousarray(x, dtype=np.float64)
    o = np.empty(H, dtype=np.float64)
    lib().oracle_expert_ffn(_ptr(wg), _ptr(wu), _ptr(wd), H, I, _ptr(xd), _ptr(o))
    return o


class QuantExpert:
    """Canonical codes and scales of one expert (gate, up, down) on the host."""

    def __init__(self, codes, scales):
        self.codes = [np.ascontiguousarray(c) for c in codes]
        self.scales = [np.ascontiguousarray(s) for s in scales]

    def _c(self):
        e = _Expert()
        for m in range(3):
            e.codes[m] = self.codes[m].ctypes.data
            e.scales[m] = self.scales[m].ctypes.data
        return e


def _experts_array(experts):
    arr = (_Expert * len(experts))()
    for i, ex in enumerate(experts):
        if ex is None:
            arr[i] = _Expert()
        else:
            arr[i] = ex._c()
    return arr


def layer_forward(experts, H: int, I: int, k: int, bits: int, group: int, dtype: int,
                  x_bf16: np.ndarray, wr_bf16: np.ndarray, bias: np.ndarray | None) -> dict:
    """Full layer on T tokens.  `experts` is a list of E QuantExpert (None allowed
    for experts that are never routed).  Returns a dict of every intermediate."""
    E = len(experts)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    wr = np.ascontiguousarray(wr_bf16, dtype=np.uint16)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = dict(
        logits=np.empty((T, E), np.float32), idx=np.empty((T, k), np.int32),
        w=np.empty((T, k), np.float64), counts=np.empty(E, np.int32),
        offsets=np.empty(E + 1, np.int32), perm=np.empty(T * k, np.int32),
        inv=np.empty(T * k, np.int32), y=np.empty((T, H), np.float64))
    arr = _experts_array(experts)
    rc = lib().oracle_layer_forward(arr, E, H, I, k, bits, group, dtype, _ptr(x), T, _ptr(wr),
                                    _ptr(b), _ptr(out["logits"]), _ptr(out["idx"]), _ptr(out["w"]),
                                    _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
                                    _ptr(out["inv"]), _ptr(out["y"]))
    if rc:
        raise ValueError(f"oracle_layer_forward failed ({rc})")
    return out


def layer_forward_tokens(experts, H: int, I: int, k: int, bits: int, group: int, dtype: int,
                         x_bf16: np.ndarray, wr_bf16: np.ndarray, bias, tok) -> np.ndarray:
    """y [n][H] (fp64) for the listed tokens only; routing over all T tokens."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    wr = np.ascontiguousarray(wr_bf16, dtype=np.uint16)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    y = np.empty((tok.size, H), np.float64)
    arr = _experts_array(experts)
    rc = lib().oracle_layer_forward_tokens(arr, len(experts), H, I, k, bits, group, dtype, _ptr(x), T,
                                           _ptr(wr), _ptr(b), _ptr(tok), tok.size, _ptr(y))
    if rc:
        raise ValueError(f"oracle_layer_forward_tokens failed ({rc})")
    return y


def cache_sim(L: int, E: int, C: int, access: np.ndarray, aging_period: int = 0) -> dict:
    """access: int32 [steps][L][maxd] distinct experts per (step, layer), -1 padded."""
    acc = np.ascontiguousarray(access, dtype=np.int32)
    steps, L2, maxd = acc.shape
    assert L2 == L
    hits = np.empty((steps, L), np.int32)
    misses = np.empty((steps, L), np.int32)
    adm = ctypes.c_int64(0)
    evi = ctypes.c_int64(0)
    owner = np.empty(max(C, 1), np.int32)
    rc = lib().oracle_cache_sim(L, E, C, steps, _ptr(acc), maxd, aging_period, _ptr(hits),
                                _ptr(misses), ctypes.addressof(adm), ctypes.addressof(evi),
                                _ptr(owner))
    if rc:
        raise ValueError(f"oracle_cache_sim failed ({rc})")
    return dict(hits=hits, misses=misses, admissions=adm.value, evictions=evi.value,
                slot_owner=owner[:C])


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """Round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)
