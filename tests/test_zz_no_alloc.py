"""The allocation-free routing entry point (moe_route_noalloc) through the C ABI.

It is meant for callers that cannot allocate device memory when they route
(for example a serving runtime that has reserved nearly all of HBM for its own
pools, so a cudaMalloc would fail or eat into memory it manages): its work
space is a fixed array inside the library.  Its routing is checked against the
oracle (fixed-order fp32 logits with the router bias, top-k with ties to the
lower index, renormalised weights) and, bit for bit, against the routing that
moe_layer_forward reports for the same layer, on two calls in a row (the calls
share the fixed array).  This file is collected last so that a run stopping at
the first failure has run everything else."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.view(dtype)


def _route_and_compare(plan, wl, wr, bias, xs):
    """Two (or more) calls in a row: each against the oracle and, bit for
    bit, against the plan forward's routing of the same tokens."""
    import torch

    from moe_expert_layer_sorted_gb300 import route_noalloc
    E, k = wl.experts, wl.top_k
    wr_d = _dev(wr.view(np.int16))
    bias_d = None if bias is None else _dev(bias.astype(np.float32))
    for x_bits in xs:
        T = x_bits.shape[0]
        x = _dev(x_bits.view(np.int16))
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
        route_noalloc(x, wr_d, bias_d, k, idx, w)
        ref_idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        ref_w = torch.empty(T, k, dtype=torch.float32, device="cuda")
        y = torch.empty_like(x)
        plan.forward(0, x.view(torch.bfloat16), y.view(torch.bfloat16),
                     dbg=dict(topk_idx=ref_idx, topk_w=ref_w))
        torch.cuda.synchronize()
        lg = oracle.router_logits(x_bits, wr, bias)
        o_idx, o_w = oracle.topk(lg, k)
        assert np.array_equal(idx.cpu().numpy(), o_idx)
        np.testing.assert_allclose(w.cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)
        assert torch.equal(idx, ref_idx)
        assert torch.equal(w, ref_w)


def test_route_noalloc_decode_shape_twice_in_a_row():
    """The decode layer's shape (H=4096, E=384, k=6) with its router bias:
    T = 6 then T = 1 (2,304 then 384 logits through the fixed array)."""
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.Workload("decode-router", 1, 384, 4096, 128, 6, (6,), 3, 128, W.SC_BF16, "zipf", 1.0)
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    assert bias is not None and np.abs(bias).max() > 0
    _route_and_compare(plan, wl, wr, bias, [W.tokens(wl, 4242, 0, 6), W.tokens(wl, 4243, 0, 1)])
    plan.close()


def test_route_noalloc_ties_go_to_the_lower_index():
    """Router rows duplicated in pairs (equal logits): the lower expert index
    first, as in the plan forward; two calls in a row."""
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.Workload("ties-router", 1, 64, 512, 128, 4, (8,), 3, 64, W.SC_BF16, "zipf", 1.0)
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    wr, bias = wr.copy(), bias.copy()
    src = np.random.default_rng(11).permutation(wl.experts)
    for a_, b_ in zip(src[:32], src[32:]):
        wr[b_] = wr[a_]
        bias[b_] = bias[a_]
    plan.set_router(0, wr, bias)
    _route_and_compare(plan, wl, wr, bias, [W.tokens(wl, 77, 0, 8), W.tokens(wl, 78, 0, 3)])
    plan.close()


def test_route_noalloc_tiny_layer_no_bias():
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["tiny"]
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    _route_and_compare(plan, wl, wr, bias, [W.tokens(wl, 4242, 0, 8), W.tokens(wl, 4243, 0, 5)])
    plan.close()


def test_route_noalloc_t0_is_the_warm_up_and_sizes_beyond_the_array_are_rejected():
    import torch

    from moe_expert_layer_sorted_gb300 import MoeError, route_noalloc
    H, E = 256, 4096
    wr = torch.zeros(E, H, dtype=torch.int16, device="cuda")
    route_noalloc(torch.zeros(0, H, dtype=torch.int16, device="cuda"), wr, None, 2,
                  torch.empty(0, 2, dtype=torch.int32, device="cuda"),
                  torch.empty(0, 2, dtype=torch.float32, device="cuda"))
    T = 65  # 266,240 logits > 262,144
    x = torch.zeros(T, H, dtype=torch.int16, device="cuda")
    idx = torch.empty(T, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(T, 2, dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError) as ei:
        route_noalloc(x, wr, None, 2, idx, w)
    assert ei.value.status == 1
