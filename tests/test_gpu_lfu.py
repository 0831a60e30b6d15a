"""LFU expert cache on the GPU against the oracle's cache simulator.

A small cached-decode stack (the shape family of "Running a 24k-expert MoE on
a single 32 GB card", sections 2-3: every expert pinned in host memory, an
HBM cache admitted by access frequency, skewed popularity with drifting
router bias) runs step by step through the C-ABI.  The distinct experts each
forward routes to are read back and replayed through ``oracle.cache_sim``:
per-(step, layer) hits and misses, admissions, evictions and the final slot
owners must match exactly.  Layer outputs must be bit-identical to a plan
that keeps every expert in HBM (placement changes no output bit) and takes
each step's drifted router biases in one call for all layers."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

WL = W.Workload("lfu-small", 3, 24, 256, 128, 2, (2,), 2, 64, W.SC_F16, "zipf", 1.2,
                cache_frac=0.25, steps=24, drift=0.05)


def _x(step, layer, T):
    import torch
    return torch.from_numpy(W.tokens(WL, step, layer, T).view(np.int16).copy()).cuda().view(torch.bfloat16)


def test_lfu_matches_cache_simulator():
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(WL)
    ref, _ = harness.build_plan(WL, all_hbm=True)
    C = plan.desc.cache_slots
    assert C == int(np.floor(0.25 * 3 * 24))
    L, E, k, T = WL.layers, WL.experts, WL.top_k, 2
    maxd = T * k
    access = np.full((WL.steps, L, maxd), -1, np.int32)
    hits = np.zeros((WL.steps, L), np.int64)
    misses = np.zeros((WL.steps, L), np.int64)
    biases = [info["routers"][l][1].copy() for l in range(L)]
    plan.stats(-1, reset=True)
    for s in range(WL.steps):
        for l in range(L):
            x = _x(s, l, T)
            y = torch.empty_like(x)
            y_ref = torch.empty_like(x)
            idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
            plan.forward(l, x, y, dbg=dict(topk_idx=idx))
            ref.forward(l, x, y_ref)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), (s, l)
            d = np.unique(idx.cpu().numpy())
            access[s, l, : len(d)] = d
            st = plan.stats(l, reset=True)
            hits[s, l], misses[s, l] = st["hits"], st["misses"]
            assert st["accesses"] == len(d)
        plan.step_end()
        for l in range(L):  # the same drift on both plans: one layer at a time, and all layers at once
            biases[l] = biases[l] + W.bias_drift(WL, s, l)
            plan.update_router_bias(l, biases[l])
        ref.update_router_biases(0, np.ascontiguousarray(np.stack(biases), dtype=np.float32))
    torch.cuda.synchronize()
    sim = oracle.cache_sim(L, E, C, access)
    np.testing.assert_array_equal(hits, sim["hits"])
    np.testing.assert_array_equal(misses, sim["misses"])
    slot_of = np.concatenate([plan.residence(l) for l in range(L)])
    owner = np.full(C, -1, np.int64)
    for g, c in enumerate(slot_of):
        if c >= 0:
            assert owner[c] == -1
            owner[c] = g
    np.testing.assert_array_equal(owner, sim["slot_owner"])
    assert hits.sum() + misses.sum() == (access >= 0).sum()
    assert sim["admissions"] >= min(C, len(np.unique(access[access >= 0])))
    plan.close()
    ref.close()


def test_lfu_admission_counters():
    """Admission and eviction totals over a run equal the simulator's."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(WL)
    C = plan.desc.cache_slots
    L, E, k, T = WL.layers, WL.experts, WL.top_k, 2
    access = np.full((WL.steps, L, T * k), -1, np.int32)
    biases = [info["routers"][l][1].copy() for l in range(L)]
    plan.stats(-1, reset=True)
    for s in range(WL.steps):
        for l in range(L):
            x = _x(s, l, T)
            y = torch.empty_like(x)
            idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
            plan.forward(l, x, y, dbg=dict(topk_idx=idx))
            torch.cuda.synchronize()
            d = np.unique(idx.cpu().numpy())
            access[s, l, : len(d)] = d
        plan.step_end()
        for l in range(L):
            biases[l] = biases[l] + W.bias_drift(WL, s, l)
            plan.update_router_bias(l, biases[l])
    tot = plan.stats(-1)
    sim = oracle.cache_sim(L, E, C, access)
    assert tot["admissions"] == sim["admissions"]
    assert tot["evictions"] == sim["evictions"]
    assert tot["hits"] == sim["hits"].sum() and tot["misses"] == sim["misses"].sum()
    assert tot["fill_bytes"] == sim["admissions"] * plan_expert_bytes(WL)
    plan.close()


def plan_expert_bytes(wl):
    return sum(wl.codes_bytes(m) + wl.matrix_shape(m)[0] * (wl.matrix_shape(m)[1] // wl.group) * 2
               for m in range(3))


# The cached-decode cache at its full size: 48 layers x 512 experts, 17,203
# HBM slots (70 %), so the device's victim scan walks every slot in several
# rounds per thread; counts halved every 16 steps; eight tokens per step so
# that the run touches more experts than the cache holds and evicts.  The
# expert matrices keep the cached workload's shape (H=2048, I=512, int2 G64
# fp16 scales): the cache rules do not depend on it, the bytes do.  At the
# last step three layers' outputs (experts read from cache slots and in place
# from host memory) are checked against the oracle as well.
WL_FULL = W.Workload("lfu-full", 48, 512, 2048, 512, 8, (8,), 2, 64, W.SC_F16, "zipf", 1.2,
                     cache_frac=0.7, steps=320, drift=0.01)
AGING = 16


def test_lfu_full_size_with_aging_matches_cache_simulator():
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl = WL_FULL
    plan, info = harness.build_plan(wl, gpu_gen=True, aging_period=AGING)
    C = plan.desc.cache_slots
    assert C == 17_203
    L, E, k, T, S = wl.layers, wl.experts, wl.top_k, 8, wl.steps
    idx_all = torch.empty(S, L, T, k, dtype=torch.int32, device="cuda")
    xs = torch.empty(S, L, T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    import synth
    cs = torch.cuda.current_stream().cuda_stream
    for s in range(S):
        for l in range(L):
            synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, s, l), T * wl.hidden, 1.0,
                                     xs[s, l].data_ptr(), cs)
    y = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    biases = np.stack([info["routers"][l][1] for l in range(L)]).astype(np.float32)
    hits = np.zeros((S, L), np.int64)
    misses = np.zeros((S, L), np.int64)
    adm = evi = 0  # the step ends' admissions and evictions, summed over the per-layer reads
    plan.stats(-1, reset=True)
    check = (0, 29, L - 1)  # layers whose outputs at the last step go to the oracle
    y_last = {l: torch.empty(T, wl.hidden, dtype=torch.bfloat16, device="cuda") for l in check}
    bias_last = None
    for s in range(S):
        if s == S - 1:
            bias_last = biases.copy()
        for l in range(L):
            out = y_last[l] if (s == S - 1 and l in check) else y
            plan.forward(l, xs[s, l], out, dbg=dict(topk_idx=idx_all[s, l]))
        for l in range(L):
            st = plan.stats(l, reset=True)
            hits[s, l], misses[s, l] = st["hits"], st["misses"]
            adm += st["admissions"]
            evi += st["evictions"]
        plan.step_end()
        biases = biases + np.stack([W.bias_drift(wl, s, l) for l in range(L)])
        plan.update_router_biases(0, np.ascontiguousarray(biases, dtype=np.float32))
    torch.cuda.synchronize()
    idx = idx_all.cpu().numpy()
    maxd = T * k
    access = np.full((S, L, maxd), -1, np.int32)
    for s in range(S):
        for l in range(L):
            d = np.unique(idx[s, l])
            access[s, l, : len(d)] = d
    sim = oracle.cache_sim(L, E, C, access, aging_period=AGING)
    tot = plan.stats(-1)
    adm += tot["admissions"]
    evi += tot["evictions"]
    slot_of = np.concatenate([plan.residence(l) for l in range(L)])
    # outputs of the last step's checked layers (experts read from cache slots
    # and in place from host memory) against the oracle, with that step's biases
    for l in check:
        x_bits = xs[S - 1, l].view(torch.int16).cpu().numpy().view(np.uint16)
        wr = info["routers"][l][0]
        used = np.unique(idx[S - 1, l])
        experts = [None] * E
        for e in used:
            q = [oracle.quantize(W.expert_master(wl, l, int(e), m), wl.bits, wl.group, wl.scale_dtype)
                 for m in range(3)]
            experts[int(e)] = oracle.QuantExpert([c for c, _ in q], [sc for _, sc in q])
        lg = oracle.router_logits(x_bits, wr, bias_last[l])
        o_idx, _ = oracle.topk(lg, k)
        assert np.array_equal(idx[S - 1, l], o_idx), l
        ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, k, wl.bits, wl.group, wl.scale_dtype,
                                          x_bits, wr, bias_last[l], np.arange(T))
        yg = oracle.bf16_to_f32(y_last[l].view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
        err = float((np.abs(yg - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)).max())
        assert err <= 1e-2, (l, err)
    plan.close()
    assert sim["evictions"] > 1000, sim["evictions"]  # the cache filled and kept turning over
    np.testing.assert_array_equal(hits, sim["hits"])
    np.testing.assert_array_equal(misses, sim["misses"])
    assert adm == sim["admissions"] and evi == sim["evictions"]
    owner = np.full(C, -1, np.int64)
    for g, c in enumerate(slot_of):
        if c >= 0:
            assert owner[c] == -1
            owner[c] = g
    np.testing.assert_array_equal(owner, sim["slot_owner"])


def test_lfu_miss_queue_overflow_is_reported():
    """Forwarding one layer more often between step ends than the step's
    miss queue allows (here: 3 forwards of a one-layer plan with a queue of
    min(E, T*k) misses) latches the overflow; the next call that looks
    reports MOE_ERR_STATE once, and the plan then works as before."""
    import torch
    from moe_expert_layer_sorted_gb300 import MoeError, harness
    wl = W.Workload("lfu-overflow", 1, 64, 256, 128, 4, (4,), 2, 64, W.SC_F16, "plain",
                    cache_frac=0.1, steps=1)
    plan, _ = harness.build_plan(wl)
    T = 4
    y = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeError) as ei:  # a later forward or the (synchronising) stats call reports it
        for s in range(3):
            plan.forward(0, _xw(wl, s, T), y)
        plan.stats(0)
    assert ei.value.status == 5 and "miss queue" in str(ei.value)
    f0 = plan.stats(0)["forwards"]  # reported once: this call succeeds
    plan.step_end()
    plan.forward(0, _xw(wl, 9, T), y)
    st = plan.stats(0)  # one forward per step again: no overflow
    assert st["forwards"] == f0 + 1
    plan.close()


def _xw(wl, step, T):
    import torch
    return torch.from_numpy(W.tokens(wl, step, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
