"""Benchmark of the tiered MoE layer on GB300.

Default workload: the decode MoE layer (H=4096, I=1024, E=384, top-6, int3
G128 bf16 scales, Zipf(1.0) popularity, the 115 least popular experts in
pinned host memory read over UVA).  One step = one forward at each decode
batch size of that workload (T = 1, 4 and 6 tokens), with a fresh input per
step; the metric is decode tokens/s over the step (11 tokens) and the
weight-stream GB/s against the HBM + host-link roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Timing: CUDA events on the launching stream around
each step (the step's forwards are one CUDA-graph replay); L2 is flushed
(256 MiB written, then 256 MiB read) between steps, outside the timed events.  `--impl reference`
times the CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

BATCHES = (1, 4, 6)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _recorded_traffic(name: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary
    profiles/<name>.md, if the kernel sources hashed there are unchanged
    (else None: counters of an older kernel do not describe this one)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name + ".md")
    try:
        kv = {}
        for line in open(path):
            if line.startswith("- ") and ": " in line:
                key, val = line[2:].split(": ", 1)
                kv[key.strip()] = val.strip()
        h = hashlib.sha1()
        for src in kv["sources"].split(","):
            h.update(open(os.path.join(ROOT, src.strip()), "rb").read())
        if h.hexdigest() != kv["sources_sha1"]:
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def _numa_node(device: int = 0):
    """{"pci_bus_id", "numa_node"} of the GPU (NVML and sysfs); a field is None
    where it cannot be read."""
    out = {"pci_bus_id": None, "numa_node": None}
    try:
        import torch
        pr = torch.cuda.get_device_properties(device)
        bus = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        bus = None
    if bus is None:
        try:
            import pynvml
            pynvml.nvmlInit()
            bus = pynvml.nvmlDeviceGetPciInfo(pynvml.nvmlDeviceGetHandleByIndex(device)).busId
            bus = bus.decode() if isinstance(bus, bytes) else bus
        except Exception:
            return out
    out["pci_bus_id"] = bus
    try:
        for cand in (bus.lower(), bus.lower()[-12:]):  # sysfs names use a 4-digit domain
            path = f"/sys/bus/pci/devices/{cand}/numa_node"
            if os.path.exists(path):
                with open(path) as f:
                    out["numa_node"] = int(f.read().strip())
                break
    except Exception:
        pass
    return out


def _tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class L2Flush:
    """Between timed steps: write 256 MiB (more than the 126 MB L2), then read
    another 256 MiB, so that L2 holds none of the step's weights and only
    clean lines (a write alone would leave ~126 MB of dirty lines whose
    write-back the next timed step would pay)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def gpu_hold(seconds: float = 0.05):
    """Keep the GPU busy for about `seconds` (a sleep kernel on the current
    stream) while the host enqueues the timed steps behind it: the steps then
    run back to back on the GPU, and a pause of the host thread (a driver
    call of the clock sampler, the interpreter) does not show up as idle GPU
    time inside a step's events.  Placed before the first timed event."""
    import torch
    torch.cuda._sleep(int(seconds * 2.1e9))


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons sampled during the timed
    region.  The timed region of a decode step is a few milliseconds, shorter
    than nvidia-smi's sampling period, so the primary sampler is a thread that
    polls NVML's read-only queries (libnvidia-ml, shipped with the driver)
    about every millisecond; nvidia-smi -lms is the fallback."""

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int):
        self.dev = torch_device_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.nvml = None
        self.max_mhz = None

    def _nvml_handle(self):
        import ctypes
        import torch
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        pr = torch.cuda.get_device_properties(self.dev)
        bus = getattr(pr, "pci_bus_id", None)
        if bus is not None:
            dom = getattr(pr, "pci_domain_id", 0)
            dv = getattr(pr, "pci_device_id", 0)
            busid = f"{dom:08x}:{bus:02x}:{dv:02x}.0".encode()
            if L.nvmlDeviceGetHandleByPciBusId_v2(busid, ctypes.byref(h)) == 0:
                return L, h
        if L.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(h)) == 0:
            return L, h
        return None

    def start(self):
        import ctypes
        import threading
        try:
            self.nvml = self._nvml_handle()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            L, h = self.nvml
            mx = ctypes.c_uint(0)
            if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = mx.value
            self.stop_flag = False

            def poll():
                clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
                while not self.stop_flag:
                    if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                            L.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                        self.samples.append((clk.value, rs.value))
                    time.sleep(0.001)
            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            # settle before the timed region: a timed step that overlapped the
            # sampler's first queries was once seen 5x slower
            time.sleep(0.1)
            return
        try:
            self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")
            self.f = open(self.path, "w")
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            sm = [c for c, _ in self.samples]
            reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "samples": len(sm), "source": "nvml", "reasons": reasons}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["no clock source"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "source": "nvidia-smi", "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_step_ms(ms_step: float, ws: int, device=None) -> float:
    """Per-step time of the job when every rank runs one replica of the layer:
    the maximum over the ranks (the job's step ends with its slowest rank)."""
    if ws <= 1:
        return ms_step
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_step], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(tokens_per_rank_step: int, ws: int, ms_step: float) -> float:
    """Whole-job throughput: the tokens every rank processed per step over the job's step time."""
    return ws * tokens_per_rank_step / (ms_step * 1e-3)


_CPU_SAMPLES = {}


def _cpu_sample(wl, tokens: int, seed_base: int):
    """Inputs of the CPU baseline, made before any timing: `tokens`
    single-token layer inputs and, quantised by the oracle, the experts they
    are routed to (quantisation is the placement step, not the forward)."""
    key_ = (wl.name, tokens, seed_base)
    if key_ in _CPU_SAMPLES:
        return _CPU_SAMPLES[key_]
    import concurrent.futures as cf
    import oracle
    from synth import workloads as W
    wr, bias, _ = W.router(wl, 0)
    xs = [W.tokens(wl, seed_base + i, 0, 1) for i in range(tokens)]
    need = set()
    for x in xs:
        idx, _ = oracle.topk(oracle.router_logits(x, wr, bias), wl.top_k)
        need |= set(int(e) for e in np.unique(idx))

    def quant(e):
        q = [oracle.quantize(W.expert_master(wl, 0, e, m), wl.bits, wl.group, wl.scale_dtype)
             for m in range(3)]
        return e, oracle.QuantExpert([c for c, _ in q], [s for _, s in q])

    experts = [None] * wl.experts
    with cf.ThreadPoolExecutor(max(1, os.cpu_count() or 1)) as ex:
        for e, qe in ex.map(quant, sorted(need)):
            experts[e] = qe
    _CPU_SAMPLES[key_] = (wr, bias, xs, experts)
    return _CPU_SAMPLES[key_]


def cpu_baseline(wl, tokens: int, threads: int = 1, seed_base: int = 77):
    """The oracle (plain C, fp32 router logits in the fixed order, fp64 FFN)
    on `tokens` single-token forwards of the workload's layer -- routing over
    all E experts, dequantisation and FFN of the routed experts, combine --
    spread over `threads` host threads (one token per task; the oracle itself
    is single-threaded).  Returns (tokens/s, seconds, sample description)."""
    import concurrent.futures as cf
    import oracle
    wr, bias, xs, experts = _cpu_sample(wl, tokens, seed_base)

    def one(x):
        oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                    wl.scale_dtype, x, wr, bias, [0])

    t0 = time.perf_counter()
    if threads <= 1:
        for x in xs:
            one(x)
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, xs))
    dt = time.perf_counter() - t0
    return tokens / dt, dt, (f"{tokens} single-token forwards of the decode layer on {threads} host "
                             f"thread(s) (routing over all experts + dequantise + fp64 FFN of the routed "
                             f"experts + combine; experts quantised beforehand, untimed)")


def cpu_baselines(wl, seed_base: int = 77) -> dict:
    """The oracle timed on the host at 1 thread and at os.cpu_count() threads."""
    cores = os.cpu_count() or 1
    v1, dt1, s1 = cpu_baseline(wl, 3, 1, seed_base)
    vn, dtn, sn = cpu_baseline(wl, 2 * cores, cores, seed_base + 1000)
    return {"value": vn, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sn,
            "seconds": dtn, "single_thread": {"value": v1, "cores": 1, "sample": s1, "seconds": dt1}}


DECODE_WORKLOAD = ("decode MoE layer: H=4096, I=1024, E=384, top-6, int3 G128 bf16 scales, Zipf(1.0), "
                   "115 least-popular experts in pinned host memory (UVA), 269 in HBM; "
                   "step = forwards at T=1, 4, 6")


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from synth import workloads as W
    wl = W.WORKLOADS["decode"]
    import oracle
    oracle.build()
    import synth
    synth.build()
    cores = os.cpu_count() or 1
    cpu_baseline(wl, cores, cores, seed_base=10)  # warm-up (also builds the sample's experts)
    total_tokens, total_s = 0, 0.0
    for s in range(args.steps):  # each step: a bounded sample of `cores` tokens, one per thread
        v, dt, sample = cpu_baseline(wl, cores, cores, seed_base=10)
        total_tokens += cores
        total_s += dt
    value = total_tokens / total_s
    line = {"impl": "reference", "metric": "MoE decode tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD, "parallelism": f"host CPU, {cores} threads"},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "tokens/s", "cores": cores,
                             "sample": f"bounded sample of the workload per step: {sample}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from moe_expert_layer_sorted_gb300 import harness, probe_bandwidth
    from synth import workloads as W

    wl = W.WORKLOADS["decode"]
    hbm_peak, peak_kind = _peaks()
    link_gbs, hbm_probe = probe_bandwidth(local, 1 << 30, 5)
    plan, info = harness.build_plan(wl, device=local)
    stream = torch.cuda.Stream(dev)
    H = wl.hidden
    pool = 32
    xs = {T: [torch.from_numpy(W.tokens(wl, 5000 + 97 * rank + s, 0, T).view(np.int16).copy())
              .to(dev).view(torch.bfloat16) for s in range(pool)] for T in BATCHES}
    ys = {T: torch.empty(T, H, dtype=torch.bfloat16, device=dev) for T in BATCHES}
    flush = L2Flush(dev)

    with torch.cuda.stream(stream):
        for T in BATCHES:  # first use sets the per-T launch configuration
            plan.forward(0, xs[T][0], ys[T], stream=stream)
    stream.synchronize()
    graphs = []
    use_graph = not args.no_graph
    if use_graph:
        for s in range(pool):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for T in BATCHES:
                    plan.forward(0, xs[T][s], ys[T], stream=torch.cuda.current_stream())
            graphs.append(g)

    def step(s):
        if use_graph:
            graphs[s % pool].replay()
        else:
            for T in BATCHES:
                plan.forward(0, xs[T][s % pool], ys[T], stream=stream)

    with torch.cuda.stream(stream):
        for w in range(args.warmup):
            flush()
            step(w)
    stream.synchronize()
    plan.stats(0, reset=True)
    if ws > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    times = []
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        gpu_hold()
        for i in range(args.steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step(args.warmup + i)
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    ck = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in times]
    ms_step = float(np.mean(ms))
    ms_median, ms_min = float(np.median(ms)), float(np.min(ms))
    ms_p90, ms_max = float(np.percentile(ms, 90)), float(np.max(ms))
    st = plan.stats(0)
    fw = max(st["forwards"], 1)
    hbm_b = st["hbm_bytes"] / args.steps     # per step (3 forwards)
    host_b = st["host_bytes"] / args.steps
    ms_step = replica_step_ms(ms_step, ws, dev)
    tokens_step = sum(BATCHES)
    value = replica_value(tokens_step, ws, ms_step)
    achieved = (hbm_b + host_b) / (ms_step * 1e-3) / 1e9
    roof_s = hbm_b / (hbm_peak * 1e9) + host_b / (link_gbs * 1e9)
    roof_max_s = max(hbm_b / (hbm_peak * 1e9), host_b / (link_gbs * 1e9))  # perfect link/HBM overlap
    eff_peak = (hbm_b + host_b) / roof_s / 1e9

    # per batch size (separate timing of each forward, same protocol)
    per_batch = {}
    for T in BATCHES:
        plan.stats(0, reset=True)
        tt = []
        with torch.cuda.stream(stream):
            for i in range(16):
                flush()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                plan.forward(0, xs[T][i % pool], ys[T], stream=stream)
                b.record(stream)
                tt.append((a, b))
        torch.cuda.synchronize()
        m = float(np.median([a.elapsed_time(b) for a, b in tt]))
        s2 = plan.stats(0)
        hb, ob = s2["hbm_bytes"] / 16, s2["host_bytes"] / 16
        rt = hb / (hbm_peak * 1e9) + ob / (link_gbs * 1e9)
        rtm = max(hb / (hbm_peak * 1e9), ob / (link_gbs * 1e9))
        per_batch[str(T)] = {"tokens_per_s": T / (m * 1e-3), "us_per_forward": m * 1e3,
                             "hbm_MB": hb / 1e6, "host_MB": ob / 1e6,
                             "roofline_us": rt * 1e6, "roofline_frac": rt / (m * 1e-3),
                             "roofline_frac_max_form": rtm / (m * 1e-3)}

    popularity = realised_popularity(plan, wl, info, dev, rank)

    # end to end through the host-buffer entry point (pinned buffers, copies timed),
    # over the same sequence of input sets as the device-timed steps
    xh = {T: [xs[T][s].view(torch.int16).cpu().pin_memory() for s in range(pool)] for T in BATCHES}
    yh = {T: torch.empty(T, H, dtype=torch.int16).pin_memory() for T in BATCHES}
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for T in BATCHES:
                plan.forward_host(0, xh[T][(args.warmup + i) % pool], yh[T], stream=stream)
            b.record(stream)
            b.synchronize()
            e2e_ms.append(a.elapsed_time(b))
    e2e_step = float(np.mean(e2e_ms))
    io_bytes = tokens_step * H * 2

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baselines(wl)

    if rank == 0:
        line = {
            "metric": "MoE decode tokens/s", "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_median": ms_median, "ms_per_step_min": ms_min, "ms_per_step_p90": ms_p90,
            "ms_per_step_max": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; weights N(0,0.02) quantised by the library's GPU quantiser)",
            "config": {"workload": DECODE_WORKLOAD,
                       "tokens_per_step": tokens_step, "l2": "256 MiB written then 256 MiB read between steps, outside the timed events",
                       "cuda_graph": use_graph, "parallelism": "replicas" if ws > 1 else "single GPU"},
            "weight_stream_GBps": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": eff_peak, "unit": "GB/s",
                         "frac": achieved / eff_peak, "traffic": _recorded_traffic("expert_decode_kernel_decode_step"),
                         "traffic_note": "DRAM read+write bytes of one step's three expert-kernel launches "
                                         "(T = 1, 4, 6) from the ncu summary in profiles/, against the step's "
                                         "hbm_bytes_per_step (null when the kernel changed since)",
                         "kernel": "router_logits_kernel + expert_decode_kernel (one step: forwards at T = 1, 4, 6)",
                         "peak_note": f"sum-form roofline: HBM {hbm_peak:.0f} GB/s ({peak_kind}, "
                                      f"MEASURED_PEAKS.json) for HBM bytes + measured host link "
                                      f"{link_gbs:.1f} GB/s for host bytes",
                         "hbm_bytes_per_step": hbm_b, "host_bytes_per_step": host_b,
                         "frac_max_form": roof_max_s / (ms_step * 1e-3)},
            "per_batch": per_batch,
            "popularity": popularity,
            "link": {"host_zero_copy_read_GBps": link_gbs, "hbm_read_probe_GBps": hbm_probe,
                     "gpu": _numa_node(local)},
            "e2e": {"value": ws * tokens_step / (e2e_step * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                    "ms_per_step": e2e_step, "ms_per_step_median": float(np.median(e2e_ms)),
                    "note": "moe_layer_forward_host per batch (copy in, forward, copy out), launched eagerly; "
                            "the same input sets in the same order as the device-timed steps"},
            "gpu_launches": 2 * len(BATCHES) * args.steps,
            "clocks": ck, "wall_s_timed": wall,
            "cpu_baseline": cpu,
        }
    plan.close()
    if rank == 0 and not args.no_prefill:
        # the prefill layer (tensor-core path) in the same run, as an extra key
        pre = prefill_measure(args, steps=max(5, min(args.steps, 20)), warmup=3, cpu=not args.no_cpu)
        line["prefill"] = pre
    if rank == 0 and not args.no_stacks:
        # the 40-layer stack and the cached 48-layer decode in the same run, as extra keys
        line["stack40"] = stack_measure(args)
        line["cached"] = cached_measure(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def realised_popularity(plan, wl, info, dev, rank: int, batches: int = 512, T: int = 6) -> dict:
    """Realised routing of the decode layer over `batches` fresh T-token
    inputs (through the forward's routing outputs): per-expert slot counts
    summarised against the Plackett-Luce Zipf(s) targets of the workload."""
    import torch
    from synth import popularity as P
    from synth import workloads as W
    H, E, k = wl.hidden, wl.experts, wl.top_k
    idx = torch.empty(batches, T, k, dtype=torch.int32, device=dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    xs = torch.from_numpy(np.stack([W.tokens(wl, 90000 + 131 * rank + b, 0, T) for b in range(batches)])
                          .view(np.int16)).to(dev).view(torch.bfloat16)
    plan.stats(0, reset=True)
    for b in range(batches):
        plan.forward(0, xs[b], y, dbg=dict(topk_idx=idx[b]))
    torch.cuda.synchronize()
    st = plan.stats(0, reset=True)
    sel = idx.cpu().numpy().reshape(-1, k)
    _, _, rank_of = info["routers"][0]
    host = np.zeros(E, bool)
    host[list(info["host_sets"][0])] = True
    counts = np.bincount(sel.ravel(), minlength=E)
    by_rank = np.zeros(E, np.int64)
    by_rank[rank_of] = counts
    target = P.plackett_luce_inclusion(E, k, wl.zipf_s)
    n_tok = sel.shape[0]
    top = max(1, E // 100)
    # Zipf exponent fitted to the realised inclusion rates of the top half of the ranks
    r = np.arange(1, E // 2 + 1)
    ok = by_rank[: E // 2] > 0
    slope = float(np.polyfit(np.log(r[ok]), np.log(by_rank[: E // 2][ok] / n_tok), 1)[0]) if ok.sum() > 2 else None
    tgt_slope = float(np.polyfit(np.log(r), np.log(target[: E // 2]), 1)[0])
    n_host = int(host.sum())
    return {
        "tokens": int(n_tok), "forwards": batches, "T": T,
        "host_share_of_slots": float(host[sel].mean()),
        "host_share_target": float(target[E - n_host:].sum() / k),
        "p_any_host_per_token": float(host[sel].any(axis=1).mean()),
        "top1pct_share_of_slots": float(by_rank[:top].sum() / sel.size),
        "top1pct_share_target": float(target[:top].sum() / k),
        "loglog_slope_top_half": slope, "loglog_slope_target": tgt_slope,
        "experts_never_routed": int((counts == 0).sum()),
        "distinct_experts_per_forward": st["accesses"] / max(st["forwards"], 1),
        "host_experts_per_forward": st["misses"] / max(st["forwards"], 1),
        "note": "realised per-expert slot counts of the decode layer's router on fresh N(0,1) inputs, "
                "against the Plackett-Luce Zipf(s) inclusion rates the synthetic router bias is calibrated to"}


def _common_line(args, metric, value, unit, ms, config, extra):
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; weights N(0,0.02) drawn on the GPU by the generator's "
                    "bit-identical device twin and quantised by the library's GPU quantiser)",
            "config": config}
    line.update(extra)
    return line


def run_stack(args):
    print(json.dumps(stack_measure(args)), flush=True)


def stack_measure(args) -> dict:
    """40-layer stack of the decode layer (config "stack40"): each step feeds
    T fresh tokens through all 40 layers, layer l+1 taking bf16(y_l + noise).
    Returns the measurement as a dict (the keys of a bench line)."""
    import torch
    import synth
    from moe_expert_layer_sorted_gb300 import harness, probe_bandwidth
    from synth import workloads as W
    wl = W.WORKLOADS["stack40"]
    dev = torch.device("cuda", 0)
    hbm_peak, peak_kind = _peaks()
    link_gbs, hbm_probe = probe_bandwidth(0, 1 << 30, 5)
    t0 = time.perf_counter()
    plan, info = harness.build_plan(wl, gpu_gen=True)
    build_s = time.perf_counter() - t0
    L, H = wl.layers, wl.hidden
    stream = torch.cuda.Stream(dev)
    nsteps = args.warmup + args.steps
    per_T = {}
    launches = 0
    for T in wl.tokens:
        cs = torch.cuda.current_stream().cuda_stream
        noise = torch.empty(nsteps, L, T, H, dtype=torch.float32, device=dev)
        x0 = torch.empty(nsteps, T, H, dtype=torch.int16, device=dev)
        for st in range(nsteps):
            synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, 1000 + st, 0), T * H, 1.0, x0[st].data_ptr(), cs)
            for l in range(L):
                synth.normal_f32_device(W.key(wl.seed, W.TAG_NOISE, 1000 + st, l), T * H, 1.0,
                                        noise[st, l].data_ptr(), cs)
        torch.cuda.synchronize()
        xs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
        ys = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L)]

        def body(st):
            xs[0].view(torch.int16).copy_(x0[st])
            for l in range(L):
                # layer output and the next layer's input bf16(y_l + noise) in one forward
                plan.forward_residual(l, xs[l], ys[l], noise[st, l], xs[l + 1], stream=torch.cuda.current_stream())

        with torch.cuda.stream(stream):
            body(0)  # per-T launch configuration before capture
        stream.synchronize()
        graphs = []
        for st in range(nsteps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body(st)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for st in range(args.warmup):
                graphs[st].replay()
        stream.synchronize()
        plan.stats(-1, reset=True)
        clocks = ClockSampler(0)
        clocks.start()
        ev = []
        with torch.cuda.stream(stream):
            gpu_hold()
            for st in range(args.warmup, nsteps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graphs[st].replay()
                b.record(stream)
                ev.append((a, b))
        torch.cuda.synchronize()
        ck = clocks.stop()
        ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
        stt = plan.stats(-1)
        hb, ob = stt["hbm_bytes"] / args.steps, stt["host_bytes"] / args.steps
        roof = hb / (hbm_peak * 1e9) + ob / (link_gbs * 1e9)
        roof_max = max(hb / (hbm_peak * 1e9), ob / (link_gbs * 1e9))
        per_T[str(T)] = {"tokens_per_s": T / (ms * 1e-3), "ms_per_step": ms, "hbm_GB_per_step": hb / 1e9,
                         "host_GB_per_step": ob / 1e9, "weight_stream_GBps": (hb + ob) / (ms * 1e-3) / 1e9,
                         "roofline_ms": roof * 1e3, "roofline_frac": roof / (ms * 1e-3),
                         "roofline_frac_max_form": roof_max / (ms * 1e-3), "clocks": ck}
        launches = 2 * L * args.steps  # router, expert kernel (which also writes the next layer's input)
        del graphs
    T_head = str(max(wl.tokens))
    line = _common_line(
        args, "MoE decode tokens/s (40-layer stack)", per_T[T_head]["tokens_per_s"], "tokens/s",
        per_T[T_head]["ms_per_step"],
        {"workload": wl.desc, "tokens_per_step": int(T_head),
         "l2": "no flush: one step streams ~1-4 GB of weights, far above L2", "cuda_graph": True,
         "parallelism": "single GPU"},
        {"per_T": per_T, "setup_s": build_s,
         "link": {"host_zero_copy_read_GBps": link_gbs, "hbm_read_probe_GBps": hbm_probe,
                  "gpu": _numa_node(0)},
         "roofline": {"bound": "hbm", "frac": per_T[T_head]["roofline_frac"],
                      "frac_max_form": per_T[T_head]["roofline_frac_max_form"],
                      "peak_note": f"sum form: HBM {hbm_peak:.0f} GB/s ({peak_kind}) + host link {link_gbs:.1f} GB/s"},
         "gpu_launches": launches, "clocks": per_T[T_head]["clocks"]})
    plan.close()
    return line


def run_cached(args):
    print(json.dumps(cached_measure(args)), flush=True)


def cached_measure(args) -> dict:
    """Cached decode (config "cached"): 48 layers, all experts in pinned host
    memory, LFU cache of 70% of them in HBM, one token per step, router bias
    drifting per step; every step ends with the cache's admission pass.
    Returns the measurement as a dict (the keys of a bench line)."""
    import torch
    import synth
    from moe_expert_layer_sorted_gb300 import harness, probe_bandwidth
    from synth import workloads as W
    wl = W.WORKLOADS["cached"]
    dev = torch.device("cuda", 0)
    hbm_peak, peak_kind = _peaks()
    link_gbs, hbm_probe = probe_bandwidth(0, 1 << 30, 5)
    t0 = time.perf_counter()
    L = args.cached_layers or wl.layers  # fewer layers: small cases for profiler captures
    plan, info = harness.build_plan(wl, gpu_gen=True, layers=L)
    build_s = time.perf_counter() - t0
    H, E, T = wl.hidden, wl.experts, 1
    S = args.cached_steps
    # per-step router biases (the drift random walk, accumulated in fp32 on the host)
    b0 = np.stack([info["routers"][l][1] for l in range(L)]).astype(np.float32)
    drift = np.stack([np.stack([W.bias_drift(wl, st, l) for l in range(L)]) for st in range(S)])
    bias_steps = torch.from_numpy(np.concatenate([b0[None], b0[None] + np.cumsum(drift, axis=0, dtype=np.float32)[:-1]])).to(dev)
    cs = torch.cuda.current_stream().cuda_stream
    noise = torch.empty(S, L, T, H, dtype=torch.float32, device=dev)
    x0 = torch.empty(S, T, H, dtype=torch.int16, device=dev)
    for st in range(S):
        synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, st, 0), T * H, 1.0, x0[st].data_ptr(), cs)
        for l in range(L):
            synth.normal_f32_device(W.key(wl.seed, W.TAG_NOISE, st, l), T * H, 1.0, noise[st, l].data_ptr(), cs)
    torch.cuda.synchronize()
    bias_stage = torch.empty(L, E, dtype=torch.float32, device=dev)
    noise_stage = torch.empty(L, T, H, dtype=torch.float32, device=dev)
    x_stage = torch.empty(T, H, dtype=torch.int16, device=dev)
    xs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
    ys = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    stream = torch.cuda.Stream(dev)

    def body():
        xs[0].view(torch.int16).copy_(x_stage)
        plan.update_router_biases(0, bias_stage, stream=torch.cuda.current_stream())
        for l in range(L):
            plan.forward_residual(l, xs[l], ys[l], noise_stage[l], xs[l + 1], stream=torch.cuda.current_stream())
        plan.step_end(stream=torch.cuda.current_stream())

    def stage(st):
        bias_stage.copy_(bias_steps[st])
        noise_stage.copy_(noise[st])
        x_stage.copy_(x0[st])

    # one eager forward sets the launch configuration; its accounting is
    # consumed by a step end before the timed run (capture itself runs nothing)
    with torch.cuda.stream(stream):
        stage(0)
        plan.forward(0, xs[0], ys[0], stream=stream)
        plan.step_end(stream=stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
    stream.synchronize()
    plan.stats(-1, reset=True)
    half = S // 2
    clocks = ClockSampler(0)
    clocks.start()
    a = torch.cuda.Event(enable_timing=True)
    m = torch.cuda.Event(enable_timing=True)
    m2 = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    st_half = None
    with torch.cuda.stream(stream):
        gpu_hold()
        a.record(stream)
        for st in range(S):
            if st == half:  # counters of the first half: read between the two timed halves
                m.record(stream)
                stream.synchronize()
                st_half = plan.stats(-1)
                gpu_hold()
                m2.record(stream)
            stage(st)
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    total_ms = a.elapsed_time(m) + m2.elapsed_time(b)
    st_all = plan.stats(-1)
    line = _common_line(
        args, "MoE decode tokens/s (cached 48-layer decode)", S / (total_ms * 1e-3), "tokens/s", total_ms / S,
        {"workload": wl.desc.replace("2048 steps", f"{S} steps").replace("48 layers", f"{L} layers"),
         "tokens_per_step": 1,
         "l2": "no flush: a step touches ~440 MB", "cuda_graph": True, "parallelism": "single GPU"},
        {"hit_rate": st_all["hits"] / max(st_all["accesses"], 1),
         "hit_rate_second_half": (st_all["hits"] - st_half["hits"]) / max(st_all["accesses"] - st_half["accesses"], 1),
         "cache": {k: st_all[k] for k in ("accesses", "hits", "misses", "admissions", "evictions",
                                          "hbm_bytes", "host_bytes", "fill_bytes")},
         "weight_stream_GBps": (st_all["hbm_bytes"] + st_all["host_bytes"]) / (total_ms * 1e-3) / 1e9,
         "roofline": {"bound": "hbm", "frac": (st_all["hbm_bytes"] / (hbm_peak * 1e9) + st_all["host_bytes"] / (link_gbs * 1e9)
                                               + st_all["fill_bytes"] / (link_gbs * 1e9)) / (total_ms * 1e-3),
                      "frac_max_form": max(st_all["hbm_bytes"] / (hbm_peak * 1e9),
                                           (st_all["host_bytes"] + st_all["fill_bytes"]) / (link_gbs * 1e9)) / (total_ms * 1e-3),
                      "peak_note": f"sum form: HBM {hbm_peak:.0f} GB/s ({peak_kind}) + host link {link_gbs:.1f} GB/s "
                                   "(misses and cache fills both cross the link)"},
         "second_half_ms_per_step": m2.elapsed_time(b) / (S - half),
         "link": {"host_zero_copy_read_GBps": link_gbs, "hbm_read_probe_GBps": hbm_probe,
                  "gpu": _numa_node(0)},
         "setup_s": build_s, "gpu_launches": (2 * L + 2) * S, "clocks": ck})  # per layer: router, expert kernel (+ next input); step end: 2
    plan.close()
    return line


def prefill_measure(args, steps: int, warmup: int, cpu: bool = True) -> dict:
    """Prefill layer (config "prefill"): T = 8192 tokens through one layer
    (H=4096, I=1024, E=384, top-6, int4 G128 bf16 scales, all experts in HBM).
    Returns the measurement as a dict (the keys of a bench line)."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    from synth import workloads as W
    wl = W.WORKLOADS["prefill"]
    T = args.tokens or wl.tokens[0]
    dev = torch.device("cuda", 0)
    tpeak, tkind = _tensor_peak()
    t0 = time.perf_counter()
    plan, info = harness.build_plan(wl, gpu_gen=True, max_tokens=T)
    build_s = time.perf_counter() - t0
    H, E, k, I = wl.hidden, wl.experts, wl.top_k, wl.inter
    import synth
    pool = 3
    xs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(pool)]
    for i, x in enumerate(xs):
        synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, 500 + i, 0), T * H, 1.0, x.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    y = torch.empty_like(xs[0])
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for w in range(warmup):
            plan.forward(0, xs[w % pool], y, stream=stream)
    stream.synchronize()
    plan.stats(0, reset=True)
    clocks = ClockSampler(0)
    clocks.start()
    ev = []
    with torch.cuda.stream(stream):
        gpu_hold()
        for i in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward(0, xs[i % pool], y, stream=stream)
            b.record(stream)
            ev.append((a, b))
    torch.cuda.synchronize()
    ck = clocks.stop()
    all_ms = [a.elapsed_time(b) for a, b in ev]
    ms = float(np.mean(all_ms))
    flops_ffn = 6.0 * T * k * H * I
    flops_router = 2.0 * T * E * H
    achieved = (flops_ffn + flops_router) / (ms * 1e-3) / 1e12
    st = plan.stats(0)
    # end to end through the host-buffer entry point
    xh = xs[0].view(torch.int16).cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e2e = []
    with torch.cuda.stream(stream):
        for i in range(max(2, steps // 2)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward_host(0, xh, yh, stream=stream)
            b.record(stream)
            b.synchronize()
            e2e.append(a.elapsed_time(b))
    e2e_ms = float(np.mean(e2e))
    plan.close()
    del xs, y
    torch.cuda.empty_cache()
    out = {
        "metric": "MoE prefill tokens/s", "value": T / (ms * 1e-3), "unit": "tokens/s", "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "ms_per_step_median": float(np.median(all_ms)),
        "ms_per_step_min": float(np.min(all_ms)), "dtype": "bf16",
        "config": {"workload": wl.desc, "tokens_per_step": T,
                   "l2": "no flush: a step streams ~2.5 GB of weights, far above L2", "cuda_graph": False},
        "tflops": achieved,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": achieved / tpeak, "traffic": _recorded_traffic("pf_gemm_kernel_prefill_T8192"),
                     "traffic_note": "DRAM read+write bytes of one gate/up GEMM launch (the dominant kernel) from "
                                     "the ncu summary in profiles/ (null when the kernel changed since)",
                     "kernel": "whole prefill forward (router, grouping, tcgen05 gate/up and down GEMMs, combine)",
                     "peak_note": f"dense bf16, {tkind} burst figure; FLOPs = 6*T*k*H*I (expert FFNs) + 2*T*E*H (router)"},
        "cache": {k_: st[k_] for k_ in ("accesses", "hits", "hbm_bytes")},
        "router_exact_per_token": st["router_exact"] / (steps * T),
        "e2e": {"value": T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2},
        "setup_s": build_s, "gpu_launches": 9 * steps,
        "gpu_launches_note": "the library's own kernels; the router's approximate-logit GEMM is a cuBLAS launch "
                             "on top", "clocks": ck}
    if cpu:
        cores = os.cpu_count() or 1
        v, dt, sample = cpu_baseline(wl, 2 * cores, cores, seed_base=600)
        out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": sample.replace("decode layer", "prefill layer (int4)"), "seconds": dt}
    return out


def run_prefill(args):
    m = prefill_measure(args, steps=args.steps, warmup=args.warmup, cpu=not args.no_cpu)
    extra = {k_: v for k_, v in m.items() if k_ not in ("metric", "value", "unit", "ms_per_step", "config",
                                                       "steps", "warmup", "dtype")}
    line = _common_line(args, m["metric"], m["value"], m["unit"], m["ms_per_step"],
                        dict(m["config"], parallelism="single GPU"), extra)
    print(json.dumps(line), flush=True)


def run_cpu_vs_uva(args):
    """The measured comparison of serving a host-resident expert: the GPU reading
    it in place over its host link (the decode forward's extra time against the
    same layer with every expert in HBM) against the host CPU computing the
    expert's FFN (cpu_expert.c, on 1 thread and on every core).  Inputs: T = 1
    decode-layer tokens that route to exactly one host-resident expert."""
    import torch
    from moe_expert_layer_sorted_gb300 import cpu_expert, harness, probe_bandwidth
    from synth import workloads as W
    wl = W.WORKLOADS["decode"]
    link_gbs, _ = probe_bandwidth(0, 1 << 30, 5)
    plan, info = harness.build_plan(wl)
    ref, _ = harness.build_plan(wl, all_hbm=True)
    host = info["host_sets"][0]
    k = wl.top_k
    idx = torch.empty(1, k, dtype=torch.int32, device="cuda")
    picks = []
    for st in range(7000, 9000):
        xb = W.tokens(wl, st, 0, 1)
        x = torch.from_numpy(xb.view(np.int16).copy()).cuda().view(torch.bfloat16)
        y = torch.empty_like(x)
        plan.forward(0, x, y, dbg=dict(topk_idx=idx))
        torch.cuda.synchronize()
        hs = [int(e) for e in idx.cpu().numpy().ravel() if int(e) in host]
        if len(hs) == 1:
            picks.append((xb, x, hs[0]))
        if len(picks) == args.cpu_vs_uva_picks:
            break
    flush = L2Flush("cuda")
    stream = torch.cuda.Stream()

    def fwd_us(p, x):
        y = torch.empty_like(x)
        with torch.cuda.stream(stream):
            p.forward(0, x, y, stream=stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                p.forward(0, x, y, stream=torch.cuda.current_stream())
        stream.synchronize()
        ev = []
        with torch.cuda.stream(stream):  # queued back to back: no idle gaps between the forwards
            for i in range(args.warmup + args.steps):
                flush()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                ev.append((a, b))
        stream.synchronize()
        return float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev[args.warmup:]]))

    cores = os.cpu_count() or 1
    rows = []
    for xb, x, e in picks:
        t_host, t_hbm = fwd_us(plan, x), fwd_us(ref, x)
        codes, scales = info["quantiser"].expert(0, e)
        hc = [c.cpu().numpy() for c in codes]
        hsc = [s.view(torch.int16).cpu().numpy() if s.dtype != torch.float32 else s.cpu().numpy() for s in scales]
        cpu = {}
        for n in (1, cores):
            ts = []
            for _ in range(3):
                t0 = time.perf_counter()
                cpu_expert.expert_ffn(hc, hsc, wl.hidden, wl.inter, wl.bits, wl.group, wl.scale_dtype, xb, threads=n)
                ts.append((time.perf_counter() - t0) * 1e6)
            cpu[n] = float(np.median(ts))
        rows.append({"expert": e, "gpu_forward_us_with_host_expert": t_host, "gpu_forward_us_all_hbm": t_hbm,
                     "gpu_extra_us": t_host - t_hbm, "cpu_expert_us_1_thread": cpu[1],
                     f"cpu_expert_us_{cores}_threads": cpu[cores]})
    med = lambda key: float(np.median([r[key] for r in rows]))
    extra_us = med("gpu_extra_us")
    line = _common_line(
        args, "host-resident expert: GPU in-place read vs CPU compute (extra us per forward)", extra_us, "us",
        med("gpu_forward_us_with_host_expert") / 1e3,
        {"workload": wl.desc + "; T = 1 tokens routed to exactly one host-resident expert",
         "l2": "256 MiB written then 256 MiB read before each timed forward", "cuda_graph": True, "parallelism": "single GPU"},
        {"higher_is_better": False,
         "expert_bytes": 4915200, "link_GBps": link_gbs, "link_time_us": 4915200 / (link_gbs * 1e3),
         "gpu_forward_us_with_host_expert": med("gpu_forward_us_with_host_expert"),
         "gpu_forward_us_all_hbm": med("gpu_forward_us_all_hbm"),
         "cpu_expert_us": {"1": med("cpu_expert_us_1_thread"), str(cores): med(f"cpu_expert_us_{cores}_threads")},
         "cpu_cores": cores, "picks": rows,
         "note": "the CPU figure would replace the link read only if it overlapped the GPU's HBM work "
                 "completely: compare it with gpu_forward_us_all_hbm, not with gpu_extra_us",
         "gpu_launches": 2 * 2 * len(rows) * args.steps})
    print(json.dumps(line), flush=True)
    plan.close()
    ref.close()


def run_prefetch_bound(args):
    """Upper bound of layer-ahead prefetch on the cached 48-layer decode: while
    layer l runs, layer l+1's experts are predicted by layer l+1's router on
    layer l's input (the only hidden state available that early); a prefetch of
    the predicted experts could turn into hits at most the misses of layer l+1
    that the prediction contains.  Counted over the second half of the steps
    (the LFU cache warm), with the bench's own chained inputs and bias drift."""
    import torch
    import synth
    from moe_expert_layer_sorted_gb300 import harness, route_noalloc
    from synth import workloads as W
    wl = W.WORKLOADS["cached"]
    dev = torch.device("cuda", 0)
    plan, info = harness.build_plan(wl, gpu_gen=True)
    L, H, E, k, T = wl.layers, wl.hidden, wl.experts, wl.top_k, 1
    S = args.prefetch_steps
    b0 = np.stack([info["routers"][l][1] for l in range(L)]).astype(np.float32)
    drift = np.stack([np.stack([W.bias_drift(wl, st, l) for l in range(L)]) for st in range(S)])
    bias_steps = torch.from_numpy(np.concatenate([b0[None], b0[None] + np.cumsum(drift, axis=0, dtype=np.float32)[:-1]])).to(dev)
    wr = [torch.from_numpy(info["routers"][l][0].view(np.int16).copy()).to(dev).view(torch.bfloat16) for l in range(L)]
    cs = torch.cuda.current_stream().cuda_stream
    xs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
    ys = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    noise = torch.empty(T, H, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    pidx = torch.empty(T, k, dtype=torch.int32, device=dev)
    pw = torch.empty(T, k, dtype=torch.float32, device=dev)
    acc = hits = misses = covered = pred_right = 0
    t0 = time.perf_counter()
    for st in range(S):
        plan.update_router_biases(0, bias_steps[st])
        synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, st, 0), T * H, 1.0, xs[0].data_ptr(), cs)
        pred = None
        for l in range(L):
            res = plan.residence(l)  # slot per expert at this step (-1: host only)
            plan.forward(l, xs[l], ys[l], dbg=dict(topk_idx=idx))
            if l + 1 < L:  # layer l+1's experts predicted from layer l's input
                route_noalloc(xs[l], wr[l + 1], bias_steps[st][l + 1], k, pidx, pw)
            synth.normal_f32_device(W.key(wl.seed, W.TAG_NOISE, st, l), T * H, 1.0, noise.data_ptr(), cs)
            synth.residual_bf16_device(ys[l].data_ptr(), noise.data_ptr(), T * H, xs[l + 1].data_ptr(), cs)
            torch.cuda.synchronize()
            used = set(int(e) for e in idx.cpu().numpy().ravel())
            if st >= S // 2:
                miss = {e for e in used if res[e] < 0}
                acc += len(used)
                misses += len(miss)
                hits += len(used) - len(miss)
                if pred is not None:
                    covered += len(miss & pred)
                    pred_right += len(used & pred)
            pred = set(int(e) for e in pidx.cpu().numpy().ravel()) if l + 1 < L else None
        plan.step_end()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    n_pred = (S - S // 2) * (L - 1) * k
    line = _common_line(
        args, "layer-ahead prefetch bound (cached 48-layer decode): hit rate with the predicted experts prefetched",
        (hits + covered) / max(acc, 1), "fraction", elapsed * 1e3 / S,
        {"workload": wl.desc.replace("2048 steps", f"{S} steps") + "; counted over the second half",
         "predictor": "layer l+1's router on layer l's input (bf16), top-k", "parallelism": "single GPU"},
        {"hit_rate_lfu": hits / max(acc, 1), "hit_rate_with_prefetch_bound": (hits + covered) / max(acc, 1),
         "accesses": acc, "misses": misses, "misses_covered_by_prediction": covered,
         "prediction_precision": pred_right / max(n_pred, 1), "note": "an upper bound: every predicted "
         "miss assumed fetched in time; the prefetch itself is not built", "gpu_launches": None})
    print(json.dumps(line), flush=True)
    plan.close()


def run_forwards(args):
    """A few decode-layer forwards for profiler captures: T tokens (--tokens,
    default 1), an input whose experts are all HBM-resident (so the captured
    launches show the HBM path alone), one configuration forward, then
    --steps forwards of that input.  Prints a short JSON line."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    from synth import workloads as W
    wl = W.WORKLOADS["decode"]
    T = args.tokens or 1
    dev = torch.device("cuda", 0)
    plan, info = harness.build_plan(wl)
    y = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device=dev)
    for s_ in range(256):  # the first input routed to HBM experts only
        x = torch.from_numpy(W.tokens(wl, 5000 + s_, 0, T).view(np.int16).copy()).to(dev).view(torch.bfloat16)
        plan.stats(0, reset=True)
        plan.forward(0, x, y)
        torch.cuda.synchronize()
        if plan.stats(0, reset=True)["misses"] == 0:
            break
    for _ in range(args.steps):
        plan.forward(0, x, y)
    torch.cuda.synchronize()
    print(json.dumps({"workload": f"decode layer forwards at T={T} (input {s_}, HBM experts only)",
                      "forwards": args.steps + s_ + 1}), flush=True)
    plan.close()


def run_prefill_chunked(args):
    """Chunked prefill with reserved slots (moe_prefill_forward): a long prompt
    (T tokens, chunks of 8,192) through the decode layer with its 115
    least-popular experts in pinned host memory, (a) staged once per prompt
    into 115 prefill slots, (b) read in place from host memory by every chunk,
    (c) on a plan with every expert in HBM."""
    import torch
    import synth
    from moe_expert_layer_sorted_gb300 import harness
    from synth import workloads as W
    wl = W.WORKLOADS["decode"]
    T = args.tokens or 131072  # the pages' 128K-token prompt
    dev = torch.device("cuda", 0)
    n_host = wl.host_count(0)
    plans = {"staged": harness.build_plan(wl, max_tokens=8192, prefill_slots=n_host, gpu_gen=True)[0],
             "in_place": harness.build_plan(wl, max_tokens=8192, prefill_slots=0, gpu_gen=True)[0],
             "all_hbm": harness.build_plan(wl, max_tokens=8192, all_hbm=True, gpu_gen=True)[0]}
    x = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device=dev)
    synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, 900, 0), T * wl.hidden, 1.0, x.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    y = torch.empty_like(x)
    ms, stats = {}, {}
    for name, plan in plans.items():
        for _ in range(args.warmup):
            plan.prefill_forward(0, x, y)
        torch.cuda.synchronize()
        plan.stats(0, reset=True)
        ev = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            plan.prefill_forward(0, x, y)
            b.record()
            ev.append((a, b))
        torch.cuda.synchronize()
        ms[name] = float(np.median([a.elapsed_time(b) for a, b in ev]))
        st = plan.stats(0, reset=True)
        stats[name] = {k_: st[k_] / args.steps for k_ in ("host_bytes", "fill_bytes", "hits", "misses")}
    for plan in plans.values():
        plan.close()
    line = _common_line(
        args, "chunked prefill with reserved prefill slots (ms per prompt)", ms["staged"], "ms", ms["staged"],
        {"workload": f"{T}-token prompt in chunks of 8,192 through the decode layer (H=4096, I=1024, E=384, "
                     f"top-6, int3 G128), {n_host} least-popular experts in pinned host memory",
         "parallelism": "single GPU"},
        {"higher_is_better": False, "ms_staged_slots": ms["staged"], "ms_in_place": ms["in_place"],
         "ms_all_hbm": ms["all_hbm"], "per_prompt": stats,
         "tokens_per_s_staged": T / (ms["staged"] * 1e-3), "gpu_launches": None})
    print(json.dumps(line), flush=True)


def run_prefill_staging(args):
    """Prefill with host-resident experts: the tcgen05 GEMMs reading the host
    experts' codes in place over the link (bulk-copy warp, 16-byte cp.async)
    against the same layer with every expert in HBM plus one host-to-HBM copy
    of those experts' bytes (what staging them into reserved HBM slots before
    the GEMMs would cost).  Shape of the cached decode's layer (H=2048, I=512,
    E=512, top-8, int2 G64 fp16, Zipf(1.2)), T = 8192, the 154 (30 %)
    least-popular experts in pinned host memory."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    from synth import workloads as W
    wl = W.Workload("prefill-staging", 1, 512, 2048, 512, 8, (8192,), 2, 64, W.SC_F16, "zipf", 1.2,
                    host_total=154, desc="prefill layer of the cached decode's shape: T=8192, H=2048, I=512, "
                                         "E=512, top-8, int2 G64 fp16 scales, Zipf(1.2), 154 least-popular "
                                         "experts in pinned host memory")
    T = 8192
    eb = sum(wl.codes_bytes(m) + wl.matrix_shape(m)[0] * (wl.matrix_shape(m)[1] // wl.group) * 2 for m in range(3))
    x = torch.from_numpy(W.tokens(wl, 0, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)

    def time_fwd(plan):
        for _ in range(args.warmup):
            plan.forward(0, x, y)
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            plan.forward(0, x, y)
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return float(np.median(ts))

    plan, info = harness.build_plan(wl, max_tokens=T, gpu_gen=True)
    n_host = len(info["host_sets"][0])
    t_inplace = time_fwd(plan)
    plan.close()
    plan, _ = harness.build_plan(wl, max_tokens=T, gpu_gen=True, all_hbm=True)
    t_hbm = time_fwd(plan)
    plan.close()
    nbytes = n_host * eb
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    cts = []
    for i in range(args.warmup + args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        if i >= args.warmup:
            cts.append(a.elapsed_time(b))
    t_copy = float(np.median(cts))
    line = _common_line(
        args, "prefill with host-resident experts: in-place reads vs staging into HBM (ms per forward)",
        t_inplace, "ms", t_inplace,
        {"workload": wl.desc, "tokens_per_step": T, "parallelism": "single GPU"},
        {"higher_is_better": False, "ms_in_place": t_inplace, "ms_all_hbm": t_hbm, "ms_copy_host_experts": t_copy,
         "ms_staged_serial": t_hbm + t_copy, "host_experts": n_host, "host_bytes": nbytes,
         "copy_GBps": nbytes / (t_copy * 1e-3) / 1e9, "gpu_launches": None,
         "note": "staging pays off if ms_all_hbm + ms_copy_host_experts (or the copy overlapped with the "
                 "HBM experts' work) is below ms_in_place"})
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode: leave out the prefill key")
    ap.add_argument("--no-stacks", action="store_true", help="decode: leave out the stack40 and cached keys")
    ap.add_argument("--workload", default="decode", choices=["decode", "stack40", "cached", "prefill",
                                                              "cpu-vs-uva", "prefetch-bound",
                                                              "prefill-staging", "prefill-chunked",
                                                              "forwards"])
    ap.add_argument("--prefetch-steps", type=int, default=512)
    ap.add_argument("--cpu-vs-uva-picks", type=int, default=6)
    ap.add_argument("--cached-steps", type=int, default=2048)
    ap.add_argument("--cached-layers", type=int, default=0, help="cached: layers (default 48)")
    ap.add_argument("--tokens", type=int, default=0, help="prefill: batch size (default 8192)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack40":
        run_stack(args)
    elif args.workload == "cached":
        run_cached(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "cpu-vs-uva":
        run_cpu_vs_uva(args)
    elif args.workload == "prefetch-bound":
        run_prefetch_bound(args)
    elif args.workload == "prefill-staging":
        run_prefill_staging(args)
    elif args.workload == "prefill-chunked":
        run_prefill_chunked(args)
    elif args.workload == "forwards":
        run_forwards(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
