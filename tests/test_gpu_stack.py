"""The 40-layer stack of the decode layer at full size (15,360 experts, 4,608
of them in pinned host memory), run the way the benchmark runs it: T fresh
tokens through all 40 layers in one CUDA graph, layer l+1 taking
bf16(y_l + noise_l).  Checked against the oracle on sampled layers with
teacher forcing (each sampled layer's oracle input is the GPU's input to that
layer): routing bit-exact, outputs within max-over-tokens
||y - y_ref||_inf / ||y_ref||_inf <= 1e-2; every layer input equal, bit for
bit, to bf16(previous output + the seeded noise), so the chain itself is the
synthetic workload's; the layers' host-expert reads counted as misses."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2
STEP = 1000  # the benchmark's first step


def _oracle_expert(wl, layer, e):
    q = [oracle.quantize(W.expert_master(wl, layer, e, m), wl.bits, wl.group, wl.scale_dtype) for m in range(3)]
    return oracle.QuantExpert([c for c, _ in q], [s for _, s in q])


def _rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float((np.abs(y - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)).max())


@pytest.fixture(scope="module")
def stack():
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["stack40"]
    plan, info = harness.build_plan(wl, gpu_gen=True)
    yield wl, plan, info
    plan.close()


@pytest.mark.parametrize("T,layers", [(1, (0, 17, 39)), (4, (0, 23, 39))])
def test_stack40_full_size(stack, T, layers):
    import torch

    import synth
    wl, plan, info = stack
    L, H, k = wl.layers, wl.hidden, wl.top_k
    dev = torch.device("cuda", 0)
    cs = torch.cuda.current_stream().cuda_stream
    x0 = torch.empty(T, H, dtype=torch.int16, device=dev)
    synth.normal_bf16_device(W.key(wl.seed, W.TAG_X, STEP, 0), T * H, 1.0, x0.data_ptr(), cs)
    noise = torch.empty(L, T, H, dtype=torch.float32, device=dev)
    for l in range(L):
        synth.normal_f32_device(W.key(wl.seed, W.TAG_NOISE, STEP, l), T * H, 1.0, noise[l].data_ptr(), cs)
    xs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
    ys = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    stream = torch.cuda.Stream(dev)

    def body():
        xs[0].view(torch.int16).copy_(x0)
        for l in range(L):
            # the layer's output and the next layer's input bf16(y_l + noise_l) in one forward
            plan.forward_residual(l, xs[l], ys[l], noise[l], xs[l + 1], stream=torch.cuda.current_stream())

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        body()  # per-T launch configuration before capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    plan.stats(-1, reset=True)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    st = plan.stats(-1, reset=True)
    xb = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]
    yb = [y.view(torch.int16).cpu().numpy().view(np.uint16) for y in ys]
    nz = noise.cpu().numpy()
    # the input chain: bf16(y_l + noise_l), and the host twin of the noise and of x0
    assert np.array_equal(xb[0], W.tokens(wl, STEP, 0, T))
    for l in range(L):
        assert np.array_equal(nz[l], W.residual_noise(wl, STEP, l, T)), l
        nxt = oracle.f32_to_bf16(oracle.bf16_to_f32(yb[l]) + nz[l])
        assert np.array_equal(xb[l + 1], nxt), l
    # host-resident experts routed by these tokens were read over the link (misses)
    routed_host = 0
    for l in range(L):
        wr, bias, _ = info["routers"][l]
        idx, _ = oracle.topk(oracle.router_logits(xb[l], wr, bias), k)
        routed_host += len(set(int(e) for e in np.unique(idx)) & info["host_sets"][l])
    assert st["forwards"] == L and st["misses"] == routed_host
    # sampled layers against the oracle, each from the GPU's own input
    for l in layers:
        wr, bias, _ = info["routers"][l]
        x = xb[l]
        lg = oracle.router_logits(x, wr, bias)
        idx, w = oracle.topk(lg, k)
        ti = torch.empty(T, k, dtype=torch.int32, device=dev)
        tw = torch.empty(T, k, dtype=torch.float32, device=dev)
        yy = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        plan.forward(l, xs[l], yy, dbg=dict(topk_idx=ti, topk_w=tw))
        torch.cuda.synchronize()
        assert np.array_equal(ti.cpu().numpy(), idx), l
        np.testing.assert_allclose(tw.cpu().numpy(), w, rtol=2e-6, atol=1e-7)
        assert np.array_equal(yy.view(torch.int16).cpu().numpy().view(np.uint16), yb[l]), l  # graph == eager
        experts = [None] * wl.experts
        for e in np.unique(idx):
            experts[int(e)] = _oracle_expert(wl, l, int(e))
        ref = oracle.layer_forward_tokens(experts, H, wl.inter, k, wl.bits, wl.group, wl.scale_dtype,
                                          x, wr, bias, np.arange(T))
        assert _rel_err(oracle.bf16_to_f32(yb[l]), ref) <= TOL, l
