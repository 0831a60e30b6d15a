"""Plans built from the seeded synthetic workloads (used by the tests, the
benchmark and the smoke run).  Inputs come from ``synth``; quantisation and
placement go through the library's own calls (``quantize``,
``Plan.place_experts``)."""
from __future__ import annotations

import numpy as np
import torch

from synth import workloads as W

from . import POLICY_LFU, POLICY_STATIC, RES_HBM, RES_HOST, Plan, quantize

_SC_TORCH = {W.SC_F32: torch.float32, W.SC_BF16: torch.bfloat16, W.SC_F16: torch.float16}


class ExpertQuantiser:
    """Generates an expert's fp32 masters (on the host and uploaded through a
    pinned buffer, or with gpu_gen=True directly on the device by the
    generator's bit-identical device twin) and quantises them on the GPU into
    canonical codes/scales."""

    def __init__(self, wl: W.Workload, device="cuda", gpu_gen: bool = False):
        self.wl = wl
        self.gpu_gen = gpu_gen
        self.dev = torch.device(device)
        n = wl.inter * wl.hidden
        self.host = torch.empty(n, dtype=torch.float32).pin_memory()
        self.dw = torch.empty(n, dtype=torch.float32, device=self.dev)
        self.codes = [torch.empty(wl.codes_bytes(m), dtype=torch.uint8, device=self.dev) for m in range(3)]
        self.scales = [torch.empty(wl.matrix_shape(m)[0] * (wl.matrix_shape(m)[1] // wl.group),
                                   dtype=_SC_TORCH[wl.scale_dtype], device=self.dev) for m in range(3)]

    def expert(self, layer: int, e: int):
        """Device (codes[3], scales[3]) of expert e of `layer`; valid until the next call."""
        wl = self.wl
        for m in range(3):
            r, c = wl.matrix_shape(m)
            if self.gpu_gen:
                import synth
                synth.normal_f32_device(W.key(wl.seed, W.TAG_WEIGHT, layer, e, m), r * c, wl.w_sigma,
                                        self.dw.data_ptr(), torch.cuda.current_stream().cuda_stream)
            else:
                torch.cuda.current_stream().synchronize()  # the pinned buffer is reused
                hv = self.host[: r * c].numpy()
                hv[:] = W.expert_master(wl, layer, e, m).ravel()
                self.dw[: r * c].copy_(self.host[: r * c], non_blocking=True)
            quantize(self.dw[: r * c].view(r, c), wl.bits, wl.group, wl.scale_dtype,
                     self.codes[m], self.scales[m])
        torch.cuda.current_stream().synchronize()
        return self.codes, self.scales


def build_plan(wl: W.Workload, *, max_tokens: int | None = None, layers: int | None = None,
               device: int = 0, all_hbm: bool = False, progress=None,
               gpu_gen: bool = False, aging_period: int = 0, prefill_slots: int = 0):
    """Create a plan for `wl` (first `layers` layers), set its routers and place
    every expert (host-resident ones per the workload; with all_hbm, a static
    plan with every expert in HBM).  Returns (plan, info)."""
    L = wl.layers if layers is None else layers
    T = max(wl.tokens) if max_tokens is None else max_tokens
    lfu = wl.cache_frac > 0 and not all_hbm  # all_hbm: every expert in HBM, no cache
    host_sets = []
    routers = []
    for l in range(L):
        wr, bias, rank = W.router(wl, l)
        routers.append((wr, bias, rank))
        hs = W.host_experts(wl, l, rank) if (wl.host_total and not all_hbm) else np.zeros(0, np.int32)
        host_sets.append(set(int(e) for e in hs))
    n_host = sum(len(s) for s in host_sets)
    plan = Plan(num_layers=L, num_experts=wl.experts, hidden=wl.hidden, inter=wl.inter,
                top_k=wl.top_k, weight_bits=wl.bits, group_size=wl.group,
                scale_dtype=wl.scale_dtype, max_tokens=T,
                cache_policy=POLICY_LFU if lfu else POLICY_STATIC,
                hbm_experts=0 if lfu else L * wl.experts - n_host,
                cache_slots=int(np.floor(wl.cache_frac * L * wl.experts)) if lfu else 0,
                aging_period=aging_period, prefill_slots=prefill_slots, device=device)
    q = ExpertQuantiser(wl, device=f"cuda:{device}", gpu_gen=gpu_gen)
    for l in range(L):
        wr, bias, _ = routers[l]
        plan.set_router(l, wr, bias)
        for e in range(wl.experts):
            codes, scales = q.expert(l, e)
            res = RES_HOST if (lfu or e in host_sets[l]) else RES_HBM
            plan.place_experts(l, e, [(codes, scales)], [res])
        if progress:
            progress(l)
    info = dict(routers=routers, host_sets=host_sets, quantiser=q)
    return plan, info
