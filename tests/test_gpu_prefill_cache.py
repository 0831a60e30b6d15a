"""Chunked prefill with HBM slots reserved for the prompt's experts
(moe_prefill_forward), through the C ABI.

"Running a 24k-expert MoE on a single 32 GB card", section 2: a prefill-aware
cache keeps slots for the experts a long prompt needs, and long inputs are
read in chunks of 8,192 tokens.  Staging an expert into a prefill slot changes
where it is read from, never what is computed: the outputs must equal, bit for
bit, those of the same chunks through moe_layer_forward and of a plan with
every expert in HBM, and stay within the oracle's tolerance.  Under LFU the
prefill must leave the decode cache untouched: residence, access counts and
the hit/miss sequence of later decode steps equal the oracle simulator fed
with the decode steps alone."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2

# 12 experts, the 4 least popular in pinned host memory; chunks of 128 tokens
WL = W.Workload("prefill-stage", 1, 12, 512, 256, 3, (300,), 3, 128, W.SC_BF16, "zipf", 1.0, host_total=4)


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(y):
    import torch
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def _rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float((np.abs(y - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)).max())


def _oracle_expert(wl, layer, e):
    q = [oracle.quantize(W.expert_master(wl, layer, e, m), wl.bits, wl.group, wl.scale_dtype) for m in range(3)]
    return oracle.QuantExpert([c for c, _ in q], [s for _, s in q])


@pytest.mark.parametrize("slots", [4, 2, 0])
def test_chunked_prefill_with_staged_experts(slots):
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl, T, chunk = WL, 300, 128
    plan, info = harness.build_plan(wl, max_tokens=chunk, prefill_slots=slots)
    ref, _ = harness.build_plan(wl, max_tokens=chunk, all_hbm=True)
    x_bits = W.tokens(wl, 31, 0, T)
    x = _dev(x_bits)
    y = torch.empty_like(x)
    plan.stats(0, reset=True)
    plan.prefill_forward(0, x, y)
    torch.cuda.synchronize()
    st = plan.stats(0, reset=True)
    # the same chunks through the plain forward, on this plan (host experts read in
    # place) and on the all-HBM plan: identical bits
    y_plain = torch.empty_like(x)
    y_ref = torch.empty_like(x)
    host_first = None
    for o in range(0, T, chunk):
        plan.forward(0, x[o:o + chunk], y_plain[o:o + chunk])
        ref.forward(0, x[o:o + chunk], y_ref[o:o + chunk])
        if host_first is None:  # host bytes of the first chunk read in place
            host_first = plan.stats(0, reset=True)["host_bytes"]
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), _bits(y_plain))
    assert np.array_equal(_bits(y), _bits(y_ref))
    wr, bias, _ = info["routers"][0]
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    out = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group, wl.scale_dtype,
                               x_bits, wr, bias)
    assert _rel_err(oracle.bf16_to_f32(_bits(y)), out["y"]) <= TOL
    # accounting: staged experts are read from HBM (hits); the staging copies
    # are fill bytes; with slots for every host expert nothing crosses the link
    # during the chunks, without slots each chunk reads them in place
    n_host = len(info["host_sets"][0])
    staged = min(slots, n_host)
    expert_bytes = wl.expert_bytes
    assert st["fill_bytes"] == staged * expert_bytes
    assert st["forwards"] == (T + chunk - 1) // chunk
    assert st["hits"] + st["misses"] == st["accesses"]
    if slots >= n_host:
        assert st["misses"] == 0 and st["host_bytes"] == 0
    if slots == 0:
        assert st["host_bytes"] >= host_first > 0
    plan.close()
    ref.close()


LFU_WL = W.Workload("lfu-prefill", 3, 24, 256, 128, 2, (2,), 2, 64, W.SC_F16, "zipf", 1.2,
                    cache_frac=0.25, steps=24, drift=0.05)


def test_chunked_prefill_leaves_the_decode_cache_untouched():
    """Decode steps, a chunked prefill of 40 tokens through layer 1 (chunks of
    16 with 24 prefill slots), more decode steps: residence and the decode
    steps' hits and misses are those of a plan that never ran the prefill and
    of the oracle simulator fed with the decode accesses only; the prefill's
    output is within tolerance of the oracle."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl = LFU_WL
    P, info = harness.build_plan(wl, max_tokens=16, prefill_slots=24)
    Q, _ = harness.build_plan(wl, max_tokens=16)
    C = P.desc.cache_slots
    L, E, k, T, S = wl.layers, wl.experts, wl.top_k, 2, wl.steps
    access = np.full((S, L, T * k), -1, np.int32)
    hits = np.zeros((S, L), np.int64)
    misses = np.zeros((S, L), np.int64)
    biases = [info["routers"][l][1].copy() for l in range(L)]
    P.stats(-1, reset=True)
    Q.stats(-1, reset=True)
    for s in range(S):
        if s == S // 2:
            res_before = [P.residence(l) for l in range(L)]
            xp_bits = W.tokens(wl, 777, 1, 40)
            xp = _dev(xp_bits)
            yp = torch.empty_like(xp)
            P.prefill_forward(1, xp, yp)
            torch.cuda.synchronize()
            P.stats(1, reset=True)  # the prefill's own counters are not part of the decode sequence
            for l in range(L):
                assert np.array_equal(P.residence(l), res_before[l]), l
            wr, bias, _ = info["routers"][1]
            wr = wr.copy()
            experts = [_oracle_expert(wl, 1, e) for e in range(E)]
            out = oracle.layer_forward(experts, wl.hidden, wl.inter, k, wl.bits, wl.group, wl.scale_dtype,
                                       xp_bits, wr, biases[1])
            assert _rel_err(oracle.bf16_to_f32(_bits(yp)), out["y"]) <= TOL
        for l in range(L):
            x = _dev(W.tokens(wl, s, l, T))
            y, yq = torch.empty_like(x), torch.empty_like(x)
            idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
            P.forward(l, x, y, dbg=dict(topk_idx=idx))
            Q.forward(l, x, yq)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), yq.view(torch.int16)), (s, l)
            d = np.unique(idx.cpu().numpy())
            access[s, l, : len(d)] = d
            st = P.stats(l, reset=True)
            hits[s, l], misses[s, l] = st["hits"], st["misses"]
        P.step_end()
        Q.step_end()
        for l in range(L):
            biases[l] = biases[l] + W.bias_drift(wl, s, l)
        P.update_router_biases(0, np.ascontiguousarray(np.stack(biases), dtype=np.float32))
        Q.update_router_biases(0, np.ascontiguousarray(np.stack(biases), dtype=np.float32))
    torch.cuda.synchronize()
    sim = oracle.cache_sim(L, E, C, access)
    np.testing.assert_array_equal(hits, sim["hits"])
    np.testing.assert_array_equal(misses, sim["misses"])
    for l in range(L):
        assert np.array_equal(P.residence(l), Q.residence(l)), l
    P.close()
    Q.close()


def test_chunked_prefill_needs_prefill_path_chunks():
    import torch
    from moe_expert_layer_sorted_gb300 import MoeError, harness
    plan, _ = harness.build_plan(W.WORKLOADS["tiny"])  # max_tokens 8: chunks would take the decode path
    x = torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeError) as ei:
        plan.prefill_forward(0, x, torch.empty_like(x))
    assert ei.value.status == 6
    plan.close()
