"""Thin Python binding of the tiered-MoE C ABI (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA library
``libmoe_gb300.so``.  There is no fallback: using the binding on a machine
without the built library raises.  Device buffers are passed as torch CUDA
tensors (or raw integer addresses); host buffers as numpy arrays or pinned
torch CPU tensors.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_OOM", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_STATE", 6: "MOE_ERR_UNSUPPORTED"}
SCALE_F32, SCALE_BF16, SCALE_F16 = 0, 1, 2
RES_HBM, RES_HOST = 0, 1
POLICY_STATIC, POLICY_LFU = 0, 1

# every symbol include/moe.h declares
EXPORTS = ["moe_plan_create", "moe_plan_destroy", "moe_set_router", "moe_update_router_bias",
           "moe_update_router_biases", "moe_debug_fail_next_forward",
           "moe_place_experts", "moe_layer_forward", "moe_layer_forward_residual", "moe_prefill_forward", "moe_layer_forward_host",
           "moe_step_end",
           "moe_cache_stats", "moe_residence_table", "moe_quantize", "moe_probe_bandwidth",
           "moe_route_noalloc", "moe_status_string", "moe_last_error"]

_P = ctypes.c_void_p


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class PlanDesc(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("num_layers", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("weight_bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("scale_dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("cache_policy", ctypes.c_int32), ("device", ctypes.c_int32),
                ("hbm_experts", ctypes.c_int64), ("cache_slots", ctypes.c_int64),
                ("reserved0", ctypes.c_int32), ("aging_period", ctypes.c_int32),
                ("prefill_slots", ctypes.c_int64), ("reserved", ctypes.c_int64 * 3)]


class ExpertWeights(ctypes.Structure):
    _fields_ = [("codes", _P * 3), ("scales", _P * 3)]


class RoutingOut(ctypes.Structure):
    _fields_ = [("logits", _P), ("topk_idx", _P), ("topk_w", _P), ("counts", _P),
                ("offsets", _P), ("perm", _P), ("inv", _P)]


class CacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("accesses", "hits", "misses", "admissions", "evictions", "hbm_bytes",
                 "host_bytes", "fill_bytes", "pairs", "forwards", "router_exact")]


_lib = None


def lib():
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -c 'import __graft_entry__ as g; "
                              f"g.build()'` (the library has no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        i32 = ctypes.c_int
        L.moe_plan_create.argtypes = [ctypes.POINTER(PlanDesc), ctypes.POINTER(_P)]
        L.moe_plan_destroy.argtypes = [_P]
        L.moe_set_router.argtypes = [_P, i32, _P, _P]
        L.moe_update_router_bias.argtypes = [_P, i32, _P, _P]
        L.moe_update_router_biases.argtypes = [_P, i32, i32, _P, _P]
        L.moe_debug_fail_next_forward.argtypes = [_P]
        L.moe_place_experts.argtypes = [_P, i32, i32, i32, _P, ctypes.POINTER(ExpertWeights)]
        L.moe_layer_forward.argtypes = [_P, i32, _P, i32, _P, _P, ctypes.POINTER(RoutingOut)]
        L.moe_layer_forward_residual.argtypes = [_P, i32, _P, i32, _P, _P, _P, _P]
        L.moe_layer_forward_host.argtypes = [_P, i32, _P, i32, _P, _P]
        L.moe_prefill_forward.argtypes = [_P, i32, _P, ctypes.c_int64, _P, _P]
        L.moe_step_end.argtypes = [_P, _P]
        L.moe_cache_stats.argtypes = [_P, i32, ctypes.POINTER(CacheStats), i32]
        L.moe_residence_table.argtypes = [_P, i32, _P]
        L.moe_quantize.argtypes = [_P, i32, i32, i32, i32, i32, _P, _P, _P]
        L.moe_probe_bandwidth.argtypes = [i32, ctypes.c_size_t, i32, ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double)]
        L.moe_route_noalloc.argtypes = [_P, i32, i32, _P, _P, i32, i32, _P, _P, _P]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = [_P]
        _lib = L
    return _lib


def _addr(a) -> int | None:
    """Address of a torch tensor, numpy array, or an int; None stays NULL."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        assert a.flags.c_contiguous
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        assert a.is_contiguous()
        return a.data_ptr()
    raise TypeError(type(a))


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, plan_handle=None):
    if rc != MOE_OK:
        msg = lib().moe_last_error(plan_handle)
        raise MoeError(rc, msg.decode() if msg else "")


class Plan:
    """An MoE layer stack with per-expert placement (see include/moe.h)."""

    def __init__(self, *, num_layers, num_experts, hidden, inter, top_k, weight_bits, group_size,
                 scale_dtype, max_tokens, cache_policy=POLICY_STATIC, hbm_experts=0,
                 cache_slots=0, aging_period=0, prefill_slots=0, device=0):
        d = PlanDesc()
        d.struct_size = ctypes.sizeof(PlanDesc)
        d.num_layers, d.num_experts, d.hidden, d.inter = num_layers, num_experts, hidden, inter
        d.top_k, d.weight_bits, d.group_size, d.scale_dtype = top_k, weight_bits, group_size, scale_dtype
        d.max_tokens, d.cache_policy, d.device = max_tokens, cache_policy, device
        d.hbm_experts, d.cache_slots = hbm_experts, cache_slots
        d.aging_period = aging_period
        d.prefill_slots = prefill_slots
        self.desc = d
        h = _P()
        _check(lib().moe_plan_create(ctypes.byref(d), ctypes.byref(h)))
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_router(self, layer, wr_bf16, bias=None):
        _check(lib().moe_set_router(self._h, layer, _addr(wr_bf16), _addr(bias)), self._h)

    def update_router_bias(self, layer, bias, stream=None):
        _check(lib().moe_update_router_bias(self._h, layer, _addr(bias), _stream(stream)), self._h)

    def debug_fail_next_forward(self):
        """Test hook: the next decode forward's bounded waits run out (see include/moe.h)."""
        _check(lib().moe_debug_fail_next_forward(self._h), self._h)

    def update_router_biases(self, first, bias, stream=None):
        """bias: [count][E] fp32 (host or device) for layers first .. first+count-1."""
        _check(lib().moe_update_router_biases(self._h, first, int(bias.shape[0]), _addr(bias),
                                              _stream(stream)), self._h)

    def place_experts(self, layer, first, weights, residence=None):
        """weights: list of (codes[3], scales[3]) per expert (numpy or torch)."""
        n = len(weights)
        arr = (ExpertWeights * n)()
        for i, (codes, scales) in enumerate(weights):
            for m in range(3):
                arr[i].codes[m] = _addr(codes[m])
                arr[i].scales[m] = _addr(scales[m])
        res = None
        if residence is not None:
            res = np.ascontiguousarray(np.asarray(residence, dtype=np.uint8))
        _check(lib().moe_place_experts(self._h, layer, first, n, _addr(res), arr), self._h)

    def forward(self, layer, x, y, stream=None, dbg: dict | None = None):
        T = x.shape[0]
        ro = None
        if dbg is not None:
            ro = RoutingOut()
            for k, v in dbg.items():
                setattr(ro, k, _addr(v))
            ro = ctypes.byref(ro)
        _check(lib().moe_layer_forward(self._h, layer, _addr(x), T, _addr(y), _stream(stream), ro),
               self._h)

    def forward_residual(self, layer, x, y, residual, out, stream=None):
        """y = the layer's output and out = bf16(y + residual) in one forward (see moe.h):
        residual fp32 [T][H], out bf16 [T][H], on x's device."""
        import torch
        T = x.shape[0]
        assert residual.dtype == torch.float32 and residual.is_contiguous() and tuple(residual.shape) == tuple(x.shape)
        assert out.is_contiguous() and out.element_size() == 2 and tuple(out.shape) == tuple(x.shape)
        assert residual.device == x.device and out.device == x.device
        _check(lib().moe_layer_forward_residual(self._h, layer, _addr(x), T, _addr(y), _addr(residual), _addr(out),
                                                _stream(stream)), self._h)

    def prefill_forward(self, layer, x, y, stream=None):
        """Chunked prefill of a long prompt with the plan's prefill slots (see moe.h)."""
        _check(lib().moe_prefill_forward(self._h, layer, _addr(x), int(x.shape[0]), _addr(y), _stream(stream)),
               self._h)

    def forward_host(self, layer, x_host, y_host, stream=None):
        T = x_host.shape[0]
        _check(lib().moe_layer_forward_host(self._h, layer, _addr(x_host), T, _addr(y_host),
                                            _stream(stream)), self._h)

    def step_end(self, stream=None):
        _check(lib().moe_step_end(self._h, _stream(stream)), self._h)

    def stats(self, layer=-1, reset=False) -> dict:
        st = CacheStats()
        _check(lib().moe_cache_stats(self._h, layer, ctypes.byref(st), int(reset)), self._h)
        return {n: int(getattr(st, n)) for n, _ in CacheStats._fields_}

    def residence(self, layer) -> np.ndarray:
        out = np.empty(self.desc.num_experts, dtype=np.int32)
        _check(lib().moe_residence_table(self._h, layer, out.ctypes.data), self._h)
        return out


def quantize(w, bits, group, scale_dtype, codes, scales, stream=None):
    """GPU quantiser into the canonical format (all device tensors)."""
    rows, cols = w.shape
    _check(lib().moe_quantize(_addr(w), rows, cols, bits, group, scale_dtype, _addr(codes),
                              _addr(scales), _stream(stream)))


def probe_bandwidth(device=0, nbytes=1 << 30, iters=5) -> tuple[float, float]:
    """(host zero-copy read GB/s, HBM read GB/s) measured by the library's probe kernel."""
    h, d = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().moe_probe_bandwidth(device, nbytes, iters, ctypes.byref(h), ctypes.byref(d)))
    return h.value, d.value


def route_noalloc(x, wr, bias, k, topk_idx, topk_w, stream=None):
    """Router logits + top-k without any allocation by the library (see
    moe_route_noalloc in include/moe.h): all buffers are the caller's device
    tensors; work space is a fixed device array inside the library.
    x [T][H] and wr [E][H] hold bf16 (bfloat16 or int16 bit patterns), bias
    [E] float32 or None, topk_idx [T][k] int32 and topk_w [T][k] float32, all
    contiguous and on one CUDA device."""
    import torch
    T, H = x.shape
    E = wr.shape[0]
    bf16_like = (torch.bfloat16, torch.int16)
    assert x.is_cuda and x.is_contiguous() and x.dtype in bf16_like, "x: contiguous bf16 [T][H] on a GPU"
    assert wr.is_contiguous() and wr.dtype in bf16_like and tuple(wr.shape) == (E, H), "wr: contiguous bf16 [E][H]"
    assert topk_idx.is_contiguous() and topk_idx.dtype == torch.int32 and tuple(topk_idx.shape) == (T, k)
    assert topk_w.is_contiguous() and topk_w.dtype == torch.float32 and tuple(topk_w.shape) == (T, k)
    tensors = [x, wr, topk_idx, topk_w]
    if bias is not None:
        assert bias.is_contiguous() and bias.dtype == torch.float32 and tuple(bias.shape) == (E,)
        tensors.append(bias)
    assert all(t.device == x.device for t in tensors), "every buffer on the same device"
    rc = lib().moe_route_noalloc(_addr(x), T, H, _addr(wr), _addr(bias), E, k, _addr(topk_idx),
                                 _addr(topk_w), _stream(stream))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_route_noalloc rejected the call")
