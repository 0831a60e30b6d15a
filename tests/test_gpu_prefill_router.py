"""Prefill routing with the router logits on tensor cores, through the C ABI.

Without a request for the logits, the prefill path takes approximate logits
from a bf16 tensor-core GEMM, bounds their distance to the library's
fixed-order fp32 logits (H 2^-20 ||x|| ||w_e|| + 2^-21 |b_e| + 2^-100, four
times a worst-case accumulation model), and recomputes in the fixed order only
the experts whose upper bound reaches the k-th largest lower bound.  The
routing that results must be the top-k of the fixed-order logits, bit for bit
(the oracle's top-k of its own logits), and the whole forward bit-identical to
the forward that computes every logit exactly.  Covered: the register path
(E <= 512) and the streaming path (E = 600), near-ties and exact ties built
into the router, tokens whose bounds overflow (all E logits recomputed), more
candidates than a warp holds, and the full prefill shape."""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from test_gpu_prefill import MID, MID2, MID3, WIDEP, _run

pytestmark = pytest.mark.gpu


def _check(plan, wl, wr, bias, x):
    """Bounded routing == oracle top-k; forward == the all-exact forward."""
    T, E, k = x.shape[0], wl.experts, wl.top_k
    plan.stats(0, reset=True)
    y, r = _run(plan, x, wl, logits=False)
    st = plan.stats(0, reset=True)
    y_all, r_all = _run(plan, x, wl, logits=True)
    lg = oracle.router_logits(x, wr, bias)
    idx, w = oracle.topk(lg, k)
    assert np.array_equal(r["topk_idx"], idx)
    np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
    for key in ("topk_idx", "topk_w", "counts", "offsets", "perm", "inv"):
        assert np.array_equal(r[key], r_all[key]), key
    assert np.array_equal(y, y_all, equal_nan=True)  # rows of 1e37 overflow the FFN
    assert T * k <= st["router_exact"] <= T * E
    return st["router_exact"] / T


LONGH = W.Workload("prefill-long-h", 1, 16, 4352, 256, 2, (24,), 3, 128, W.SC_BF16, "plain")
K8 = W.Workload("prefill-k8", 1, 96, 512, 256, 8, (200,), 4, 64, W.SC_BF16, "zipf", 1.0)   # k = 8: the first
K1 = W.Workload("prefill-k1", 1, 96, 512, 256, 1, (200,), 4, 64, W.SC_BF16, "zipf", 1.0)   # round is k; k = 1


@pytest.mark.parametrize("wl,T", [(MID, 9), (MID, 300), (MID3, 700), (MID2, 600), (WIDEP, 40), (LONGH, 24),
                                  (K8, 200), (K1, 200)])
def test_bounded_router_matches_the_fixed_order(wl, T):
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(wl, max_tokens=T)
    wr, bias, _ = info["routers"][0]
    _check(plan, wl, wr, bias, W.tokens(wl, 40 + T, 0, T))
    plan.close()


NEAR = W.Workload("prefill-near-ties", 1, 128, 512, 256, 4, (96,), 4, 64, W.SC_F32, "plain")


def test_bounded_router_near_and_exact_ties():
    """Router rows in pairs one bf16 ulp apart in one element, and in exact
    duplicates; tokens of zeros (logits = bias, tied in pairs), tokens whose
    norm bound overflows (entries of 1e37: every logit recomputed), and tokens
    that put every expert inside the bound (more candidates than a warp holds)."""
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = NEAR, 96
    E, H = wl.experts, wl.hidden
    plan, info = harness.build_plan(wl, max_tokens=T)
    rng = np.random.default_rng(2024)
    wf = oracle.bf16_to_f32(info["routers"][0][0]).astype(np.float32)
    wr = oracle.f32_to_bf16(wf)
    for a in range(0, 64, 2):  # one ulp apart in element a
        wr[a + 1] = wr[a]
        wr[a + 1, a] = wr[a, a] + 1
    for a in range(64, 96):  # exact duplicates
        wr[a + 32] = wr[a]
    bias = np.repeat(rng.normal(0, 0.5, E // 2).astype(np.float32), 2)
    plan.set_router(0, wr, bias)
    x = oracle.bf16_to_f32(W.tokens(wl, 9, 0, T)).astype(np.float32)
    x[0:8] = 0.0
    x[8:16, :8] = 1e37
    # rows that make every logit (nearly) equal: one column against a router
    # whose column is constant
    x[16:24] = 0.0
    x[16:24, 5] = rng.normal(0, 1, 8)
    x = oracle.f32_to_bf16(x)
    wr2 = wr.copy()
    wr2[:, 5] = wr[0, 5]
    bias0 = np.zeros(E, np.float32)
    per_token = _check(plan, wl, wr, bias, x)
    assert per_token > wl.top_k
    plan.set_router(0, wr2, bias0)
    _check(plan, wl, wr2, bias0, x)
    plan.close()


def test_bounded_router_full_size():
    """T = 8192 at the prefill shape (H = 4096, E = 384, k = 6): the bounded
    routing equals the all-exact routing over every token, the oracle's on a
    sample, and the two forwards are bit-identical."""
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["prefill"]
    T = 8192
    plan, info = harness.build_plan(wl, gpu_gen=True)
    wr, bias, _ = info["routers"][0]
    x = W.tokens(wl, 0, 0, T)
    plan.stats(0, reset=True)
    y, r = _run(plan, x, wl, logits=False)
    st = plan.stats(0, reset=True)
    y_all, r_all = _run(plan, x, wl, logits=True)
    for key in ("topk_idx", "topk_w", "counts", "offsets", "perm", "inv"):
        assert np.array_equal(r[key], r_all[key]), key
    assert np.array_equal(y, y_all)
    samp = np.unique(np.concatenate([np.arange(3, T, 53), [T - 1]]))
    idx, w = oracle.topk(oracle.router_logits(x[samp], wr, bias), wl.top_k)
    assert np.array_equal(r["topk_idx"][samp], idx)
    np.testing.assert_allclose(r["topk_w"][samp], w, rtol=2e-6, atol=1e-7)
    per_token = st["router_exact"] / T
    print(f"fixed-order logits per token: {per_token:.2f} of {wl.experts}")
    assert wl.top_k <= per_token < 0.1 * wl.experts
    plan.close()


def test_prefill_forward_in_a_cuda_graph():
    """The prefill forward (its cuBLAS GEMM included, on the plan's own
    workspace) captured into a CUDA graph and replayed gives the eager
    forward's bits."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = MID3, 700
    plan, _ = harness.build_plan(wl, max_tokens=T)
    x = torch.from_numpy(W.tokens(wl, 99, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y_ref, y_g = torch.empty_like(x), torch.empty_like(x)
    plan.forward(0, x, y_ref)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.forward(0, x, y_g, stream=s)
    for _ in range(2):
        y_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_g.view(torch.int16), y_ref.view(torch.int16))
    plan.close()
