"""GPU parity through the C-ABI: the CUDA path against the oracle on the same
seeded inputs.  Routing, permutation and quantised codes bit-exact; layer
outputs within max-over-tokens ||y - y_ref||_inf / ||y_ref||_inf <= 1e-2."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _torch():
    import torch
    return torch


def _rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(y - ref).max(axis=1)
    den = np.abs(ref).max(axis=1)
    return float((num / np.maximum(den, 1e-30)).max())


def _bf16_bits_to_f64(t):
    return oracle.bf16_to_f32(t.view(_torch().int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def _oracle_expert(wl, layer, e):
    codes, scales = [], []
    for m in range(3):
        c, s = oracle.quantize(W.expert_master(wl, layer, e, m), wl.bits, wl.group, wl.scale_dtype)
        codes.append(c)
        scales.append(s)
    return oracle.QuantExpert(codes, scales)


def _run(plan, layer, x_bits, wl):
    torch = _torch()
    T = x_bits.shape[0]
    x = torch.from_numpy(x_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    E, k = wl.experts, wl.top_k
    dbg = dict(logits=torch.empty(T, E, dtype=torch.float32, device="cuda"),
               topk_idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               topk_w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    plan.forward(layer, x, y, dbg=dbg)
    torch.cuda.synchronize()
    return y, {k_: v.cpu().numpy() for k_, v in dbg.items()}


@pytest.fixture(scope="module")
def tiny():
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["tiny"]
    plan, info = harness.build_plan(wl)
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    yield wl, plan, info, experts
    plan.close()


def test_quantiser_codes_bit_exact(tiny):
    """The library's GPU quantiser and the oracle's produce the same codes and scales."""
    wl, plan, info, experts = tiny
    q = info["quantiser"]
    for e in (0, 5, 15):
        codes, scales = q.expert(0, e)
        for m in range(3):
            assert np.array_equal(codes[m].cpu().numpy(), experts[e].codes[m])
            got = scales[m].cpu().contiguous().view(-1).numpy().view(experts[e].scales[m].dtype)
            assert np.array_equal(got, experts[e].scales[m].ravel())


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_tiny_layer(tiny, T):
    wl, plan, info, experts = tiny
    wr, bias, _ = info["routers"][0]
    x = W.tokens(wl, 100 + T, 0, T)
    y, r = _run(plan, 0, x, wl)
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["logits"], ref["logits"])
    assert np.array_equal(r["topk_idx"], ref["idx"])
    np.testing.assert_allclose(r["topk_w"], ref["w"], rtol=2e-6, atol=1e-7)
    assert np.array_equal(r["counts"], ref["counts"])
    assert np.array_equal(r["offsets"], ref["offsets"])
    assert np.array_equal(r["perm"], ref["perm"])
    assert np.array_equal(r["inv"], ref["inv"])
    assert _rel_err(_bf16_bits_to_f64(y), ref["y"]) <= TOL


def test_empty_batch_is_a_noop(tiny):
    torch = _torch()
    wl, plan, _, _ = tiny
    x = torch.empty(0, wl.hidden, dtype=torch.bfloat16, device="cuda")
    plan.forward(0, x, torch.empty_like(x))


@pytest.mark.parametrize("T,mode", [(1, "pinned"), (8, "pinned"), (8, "pageable"), (5, "pinned-x-offset"),
                                    (5, "pinned-y-offset")])
def test_host_buffer_forward_matches_device_forward(tiny, T, mode):
    """Host buffers give the device forward's bits: page-locked ones through
    their device mappings (copy kernel in, direct writes out), pageable or
    misaligned ones through copy-engine copies."""
    torch = _torch()
    wl, plan, info, _ = tiny
    H = wl.hidden
    x = W.tokens(wl, 7 + T, 0, T)
    y_dev, _ = _run(plan, 0, x, wl)
    xs = torch.from_numpy(x.view(np.int16).copy())
    if mode == "pageable":
        xh, yh = xs.clone(), torch.zeros(T, H, dtype=torch.int16)
    elif mode == "pinned-x-offset":  # x 8 bytes past a 16-byte boundary
        buf = torch.zeros(T * H + 8, dtype=torch.int16).pin_memory()
        xh = buf[4:4 + T * H].view(T, H)
        xh.copy_(xs)
        yh = torch.zeros(T, H, dtype=torch.int16).pin_memory()
    elif mode == "pinned-y-offset":  # y 2 bytes past a 4-byte boundary
        xh = xs.pin_memory()
        buf = torch.zeros(T * H + 8, dtype=torch.int16).pin_memory()
        yh = buf[1:1 + T * H].view(T, H)
    else:
        xh, yh = xs.pin_memory(), torch.zeros(T, H, dtype=torch.int16).pin_memory()
    plan.forward_host(0, xh, yh)
    torch.cuda.synchronize()
    assert torch.equal(yh, y_dev.view(torch.int16).cpu())


def test_captured_forward_then_forward_on_another_stream(tiny):
    """A forward captured into a CUDA graph takes no part in the plan's
    cross-stream ordering; replays and ordinary forwards on other streams
    afterwards give the same bits."""
    torch = _torch()
    wl, plan, _, _ = tiny
    x = torch.from_numpy(W.tokens(wl, 21, 0, 8).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y_ref = torch.empty_like(x)
    plan.forward(0, x, y_ref)
    torch.cuda.synchronize()
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    y_g = torch.empty_like(x)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=a):
        plan.forward(0, x, y_g, stream=a)
    g.replay()
    torch.cuda.synchronize()
    y_b = torch.empty_like(x)
    with torch.cuda.stream(b):
        plan.forward(0, x, y_b, stream=b)
    torch.cuda.synchronize()
    assert torch.equal(y_g.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(y_b.view(torch.int16), y_ref.view(torch.int16))


def test_placement_changes_no_output_bit():
    """Same layer placed all-HBM, all-host and mixed: identical y bits."""
    torch = _torch()
    from moe_expert_layer_sorted_gb300 import RES_HBM, RES_HOST, Plan, harness
    wl = W.WORKLOADS["tiny"]
    q = harness.ExpertQuantiser(wl)
    wr, bias, _ = W.router(wl, 0)
    x = W.tokens(wl, 3, 0, 8)
    outs = []
    for mode in ("hbm", "host", "mixed"):
        res = [RES_HBM if (mode == "hbm" or (mode == "mixed" and e % 2)) else RES_HOST
               for e in range(wl.experts)]
        n_hbm = sum(r == RES_HBM for r in res)
        plan = Plan(num_layers=1, num_experts=wl.experts, hidden=wl.hidden, inter=wl.inter,
                    top_k=wl.top_k, weight_bits=wl.bits, group_size=wl.group,
                    scale_dtype=wl.scale_dtype, max_tokens=8, hbm_experts=n_hbm)
        plan.set_router(0, wr, bias)
        for e in range(wl.experts):
            codes, scales = q.expert(0, e)
            plan.place_experts(0, e, [(codes, scales)], [res[e]])
        y, _ = _run(plan, 0, x, wl)
        st = plan.stats(0)
        assert st["hits"] + st["misses"] == st["accesses"]
        if mode == "host":
            assert st["hits"] == 0 and st["misses"] == st["accesses"] > 0
        outs.append(y.view(torch.int16).cpu())
        plan.close()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_invalid_calls_return_status(tiny):
    torch = _torch()
    from moe_expert_layer_sorted_gb300 import MoeError, Plan
    wl, plan, _, _ = tiny
    x = torch.zeros(9, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeError) as ei:
        plan.forward(0, x, torch.empty_like(x))          # T > max_tokens
    assert ei.value.status == 1
    with pytest.raises(MoeError) as ei:
        plan.forward(1, x[:2], torch.empty_like(x[:2]))  # no such layer
    assert ei.value.status == 1
    p2 = Plan(num_layers=1, num_experts=16, hidden=256, inter=128, top_k=2, weight_bits=4,
              group_size=32, scale_dtype=0, max_tokens=8, hbm_experts=16)
    with pytest.raises(MoeError) as ei:
        p2.forward(0, x[:2], torch.empty_like(x[:2]))    # experts not placed
    assert ei.value.status == 5
    p2.close()
    with pytest.raises(MoeError) as ei:                  # far beyond HBM
        Plan(num_layers=1, num_experts=4096, hidden=65536, inter=65536, top_k=2, weight_bits=4,
             group_size=128, scale_dtype=1, max_tokens=8, hbm_experts=4096)
    assert ei.value.status == 2


@pytest.fixture(scope="module")
def decode_layer():
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["decode"]
    plan, info = harness.build_plan(wl)
    yield wl, plan, info
    plan.close()


@pytest.mark.parametrize("T", [1, 4, 6])
def test_decode_layer_full_size(decode_layer, T):
    """Decode layer at full size (H=4096, I=1024, E=384, int3): routing bit-exact
    and outputs of every token against the oracle, over steps until a host-resident
    expert has been read."""
    wl, plan, info = decode_layer
    wr, bias, _ = info["routers"][0]
    cache = {}
    st0 = plan.stats(0)
    saw_host = False
    for step in range(6):
        x = W.tokens(wl, 1000 * T + step, 0, T)
        y, r = _run(plan, 0, x, wl)
        lg = oracle.router_logits(x, wr, bias)
        idx, w = oracle.topk(lg, wl.top_k)
        assert np.array_equal(r["logits"], lg)
        assert np.array_equal(r["topk_idx"], idx)
        np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
        counts, offsets, perm, inv = oracle.permute(idx, wl.experts)
        assert np.array_equal(r["perm"], perm) and np.array_equal(r["offsets"], offsets)
        for e in np.unique(idx):
            if e not in cache:
                cache[e] = _oracle_expert(wl, 0, int(e))
        experts = [cache.get(e) for e in range(wl.experts)]
        ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                          wl.scale_dtype, x, wr, bias, np.arange(T))
        assert _rel_err(_bf16_bits_to_f64(y), ref) <= TOL
        saw_host |= bool(set(np.unique(idx).tolist()) & info["host_sets"][0])
        if saw_host and step >= 1:
            break
    st = plan.stats(0)
    assert st["accesses"] - st0["accesses"] == st["hits"] - st0["hits"] + st["misses"] - st0["misses"]


# more experts than one warp's 16 registers per lane hold (the list-based top-k
# of the decode prologue); T = 1, 5, 8
WIDE = W.Workload("decode-wide", 1, 600, 256, 128, 5, (8,), 3, 64, W.SC_BF16, "zipf", 1.0, host_total=150)


@pytest.mark.parametrize("T", [1, 5, 8])
def test_wide_router_layer(T):
    from moe_expert_layer_sorted_gb300 import harness
    wl = WIDE
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    x = W.tokens(wl, 300 + T, 0, T)
    y, r = _run(plan, 0, x, wl)
    routed = np.unique(r["topk_idx"])
    experts = [_oracle_expert(wl, 0, e) if e in routed else None for e in range(wl.experts)]
    ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                      wl.scale_dtype, x, wr, bias, np.arange(T))
    lg = oracle.router_logits(x, wr, bias)
    idx, w = oracle.topk(lg, wl.top_k)
    assert np.array_equal(r["logits"], lg)
    assert np.array_equal(r["topk_idx"], idx)
    np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
    counts, offsets, perm, inv = oracle.permute(idx, wl.experts)
    assert np.array_equal(r["counts"], counts) and np.array_equal(r["perm"], perm)
    assert _rel_err(_bf16_bits_to_f64(y), ref) <= TOL
    plan.close()


# H with 17 column blocks of 256: gate/up tasks split into two units (9 + 8
# blocks) whose partial sums carry across the units
LONGH = W.Workload("decode-long-h", 1, 16, 4352, 256, 2, (3,), 3, 128, W.SC_BF16, "plain")


@pytest.mark.parametrize("T", [1, 3])
def test_split_gate_up_task(T):
    from moe_expert_layer_sorted_gb300 import harness
    wl = LONGH
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    x = W.tokens(wl, 400 + T, 0, T)
    y, r = _run(plan, 0, x, wl)
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["logits"], ref["logits"])
    assert np.array_equal(r["topk_idx"], ref["idx"])
    assert _rel_err(_bf16_bits_to_f64(y), ref["y"]) <= TOL
    plan.close()


# Router rows duplicated in pairs, or all equal: equal logits must go to the
# lower expert index (the tie rule of the top-k), on both top-k paths of the
# decode kernel (E <= 512 and E > 512)
TIES = {384: W.Workload("decode-ties", 1, 384, 256, 128, 6, (8,), 3, 64, W.SC_BF16, "zipf", 1.0),
        600: WIDE}


@pytest.mark.parametrize("E", [384, 600])
@pytest.mark.parametrize("T", [1, 8])
@pytest.mark.parametrize("mode", ["pairs", "all"])
def test_router_ties_go_to_the_lower_index(E, T, mode):
    from moe_expert_layer_sorted_gb300 import harness
    wl = TIES[E]
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    wr, bias = wr.copy(), bias.copy()
    if mode == "all":
        wr[:] = wr[0]
        bias[:] = bias[0]
    else:
        src = np.random.default_rng(7 + E + T).permutation(E)
        for a_, b_ in zip(src[: E // 2], src[E // 2:]):  # expert b_ gets expert a_'s router row
            wr[b_] = wr[a_]
            bias[b_] = bias[a_]
    plan.set_router(0, wr, bias)
    x = W.tokens(wl, 500 + T, 0, T)
    y, r = _run(plan, 0, x, wl)
    lg = oracle.router_logits(x, wr, bias)
    idx, w = oracle.topk(lg, wl.top_k)
    assert np.array_equal(r["logits"], lg)
    assert np.array_equal(r["topk_idx"], idx)
    if mode == "all":
        assert (idx == np.arange(wl.top_k)).all()
    np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
    counts, offsets, perm, inv = oracle.permute(idx, wl.experts)
    assert np.array_equal(r["perm"], perm) and np.array_equal(r["inv"], inv)
    plan.close()


def test_bounded_wait_runs_out_and_the_plan_recovers():
    """The failure path without a fault: a forward whose gate/up results are
    never published runs its down units' bounded waits out and ends; the next
    call reports MOE_ERR_TIMEOUT; after it the plan gives the oracle's routing
    and outputs again, bit-identical to a forward before the failure."""
    import moe_expert_layer_sorted_gb300 as M
    from moe_expert_layer_sorted_gb300 import harness
    torch = _torch()
    wl = W.WORKLOADS["tiny"]
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    T = 4
    x = W.tokens(wl, 900, 0, T)
    y0, _ = _run(plan, 0, x, wl)
    plan.debug_fail_next_forward()
    _run(plan, 0, x, wl)  # its waits run out (bounded), the kernel ends
    with pytest.raises(M.MoeError) as ei:
        _run(plan, 0, x, wl)
    assert ei.value.status == 4  # MOE_ERR_TIMEOUT
    y1, r = _run(plan, 0, x, wl)
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["topk_idx"], ref["idx"])
    assert _rel_err(_bf16_bits_to_f64(y1), ref["y"]) <= TOL
    for _ in range(3):  # and keeps working
        y2, _ = _run(plan, 0, x, wl)
        assert torch.equal(y2.view(torch.int16), y0.view(torch.int16))
    plan.close()


def _shifted_tokens(wl, seed, T, mode):
    """Layer inputs at the method's numerical edge: a large common offset
    (c + N(0,1), c = 8 or 64), or N(0,1) with eight outlier columns of
    +-1000 (every column of a token offset or outlying, so the integer-code
    zero-point sums of every scale group carry it)."""
    x = oracle.bf16_to_f32(W.tokens(wl, seed, 0, T)).astype(np.float32)
    if mode.startswith("offset"):
        x = x + np.float32(int(mode[6:]))
    else:
        cols = np.random.default_rng(seed).choice(wl.hidden, 8, replace=False)
        x[:, cols] = np.where(np.arange(8) % 2 == 0, 1000.0, -1000.0).astype(np.float32)
    return oracle.f32_to_bf16(x)


@pytest.mark.parametrize("T", [1, 6])
@pytest.mark.parametrize("mode", ["offset8", "offset64", "outliers"])
def test_decode_activation_edge_cases(decode_layer, T, mode):
    """Decode layer at full size with offset or outlying activations: routing
    bit-exact, outputs within the per-token tolerance (the code offset folded
    into per-group sums of x must not cancel catastrophically)."""
    wl, plan, info = decode_layer
    wr, bias, _ = info["routers"][0]
    x = _shifted_tokens(wl, 7000 + T, T, mode)
    y, r = _run(plan, 0, x, wl)
    lg = oracle.router_logits(x, wr, bias)
    idx, w = oracle.topk(lg, wl.top_k)
    assert np.array_equal(r["logits"], lg)
    assert np.array_equal(r["topk_idx"], idx)
    np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
    experts = [_oracle_expert(wl, 0, e) if e in np.unique(idx) else None for e in range(wl.experts)]
    ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                      wl.scale_dtype, x, wr, bias, np.arange(T))
    assert _rel_err(_bf16_bits_to_f64(y), ref) <= TOL


@pytest.mark.parametrize("fault", ["pinned_alloc", "hbm_alloc"])
def test_injected_allocation_failure_returns_oom(fault, monkeypatch):
    """The host-side fault injection of the failure path: with MOE_FAULT set,
    the pinned host arena (or the HBM arena) allocation fails as a real one
    would, and moe_plan_create returns MOE_ERR_OOM with everything released;
    without it the same plan is created."""
    from moe_expert_layer_sorted_gb300 import MoeError, Plan
    kw = dict(num_layers=1, num_experts=16, hidden=256, inter=128, top_k=2, weight_bits=4, group_size=32,
              scale_dtype=0, max_tokens=8, hbm_experts=8)  # 8 experts in HBM, 8 in pinned host memory
    monkeypatch.setenv("MOE_FAULT", fault)
    with pytest.raises(MoeError) as ei:
        Plan(**kw)
    assert ei.value.status == 2 and "injected" in str(ei.value)
    monkeypatch.delenv("MOE_FAULT")
    Plan(**kw).close()
