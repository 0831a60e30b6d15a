"""The allocation-free routing entry point (moe_route_noalloc) against the
routing that moe_layer_forward reports, through the C ABI.

It is meant for callers that cannot allocate device memory when they route
(for example a runtime that has reserved nearly all HBM for its own pools):
its work space is a fixed array inside the library.  This file is collected
last so that a run stopping at the first failure has run everything else."""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu


def test_route_noalloc_matches_layer_forward_twice_in_a_row():
    import torch

    from moe_expert_layer_sorted_gb300 import harness, route_noalloc
    wl = W.WORKLOADS["tiny"]
    plan, info = harness.build_plan(wl)
    wr, bias, _ = info["routers"][0]
    wr_d = torch.from_numpy(wr.view(np.int16).copy()).cuda()
    bias_d = None if bias is None else torch.from_numpy(bias).cuda()
    E, k = wl.experts, wl.top_k
    for call, T in enumerate((8, 5)):  # two calls in a row share the fixed array
        x = torch.from_numpy(W.tokens(wl, 4242 + call, 0, T).view(np.int16).copy()).cuda()
        y = torch.empty_like(x)
        ref_idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        ref_w = torch.empty(T, k, dtype=torch.float32, device="cuda")
        plan.forward(0, x.view(torch.bfloat16), y.view(torch.bfloat16),
                     dbg=dict(topk_idx=ref_idx, topk_w=ref_w))
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
        route_noalloc(x, wr_d, bias_d, k, idx, w)
        torch.cuda.synchronize()
        assert torch.equal(idx.cpu(), ref_idx.cpu())
        np.testing.assert_allclose(w.cpu().numpy(), ref_w.cpu().numpy(), rtol=2e-6, atol=1e-7)
    plan.close()


def test_route_noalloc_rejects_sizes_beyond_its_array():
    import torch

    from moe_expert_layer_sorted_gb300 import MoeError, route_noalloc
    T, H, E = 65, 256, 4096  # 266,240 logits > 262,144
    x = torch.zeros(T, H, dtype=torch.int16, device="cuda")
    wr = torch.zeros(E, H, dtype=torch.int16, device="cuda")
    idx = torch.empty(T, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(T, 2, dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError) as ei:
        route_noalloc(x, wr, None, 2, idx, w)
    assert ei.value.status == 1
