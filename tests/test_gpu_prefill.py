"""Prefill path (T > 8) through the C-ABI against the oracle.

Routing (logits, top-k, grouping) must match bit for bit; the layer output
within max-over-tokens ||y - y_ref||_inf / ||y_ref||_inf <= 1e-2.  Sizes span
several 128-row weight tiles and 256-token tiles with ragged tails (token
counts that are not multiples of 16 or 256, experts with a single token), and
the full prefill shape (T = 8192, H = 4096, I = 1024, E = 384, int4 G128) is
checked on every routing output and on a sample of tokens."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _rel_err(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float((np.abs(y - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)).max())


def _oracle_expert(wl, layer, e):
    q = [oracle.quantize(W.expert_master(wl, layer, e, m), wl.bits, wl.group, wl.scale_dtype) for m in range(3)]
    return oracle.QuantExpert([c for c, _ in q], [s for _, s in q])


def _run(plan, x_bits, wl, logits=True):
    """One forward with the routing outputs.  Asking for the logits makes the
    library compute every logit in its fixed order; without them the routing
    takes the bounded tensor-core pass."""
    import torch
    T = x_bits.shape[0]
    x = torch.from_numpy(x_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    E, k = wl.experts, wl.top_k
    dbg = dict(topk_idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               topk_w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    if logits:
        dbg["logits"] = torch.empty(T, E, dtype=torch.float32, device="cuda")
    plan.forward(0, x, y, dbg=dbg)
    torch.cuda.synchronize()
    yb = oracle.bf16_to_f32(y.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return yb, {k_: v.cpu().numpy() for k_, v in dbg.items()}


# a mid-sized layer: I spans 2 tiles of 128 rows, H 3 tiles, several experts
# with more than 256 tokens at the larger T
MID = W.Workload("prefill-mid", 1, 8, 512, 256, 2, (300,), 4, 64, W.SC_F32, "zipf", 1.0)
MID3 = W.Workload("prefill-mid3", 1, 12, 512, 256, 3, (700,), 3, 128, W.SC_BF16, "zipf", 1.0)
MID2 = W.Workload("prefill-mid2", 1, 16, 256, 128, 2, (600,), 2, 32, W.SC_F16, "zipf", 1.2)


@pytest.mark.parametrize("wl,T", [(MID, 9), (MID, 64), (MID, 300), (MID3, 700), (MID2, 600)])
def test_prefill_layer(wl, T):
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(wl, max_tokens=T)
    wr, bias, _ = info["routers"][0]
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    x = W.tokens(wl, 7 + T, 0, T)
    y, r = _run(plan, x, wl)
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["logits"], ref["logits"])
    assert np.array_equal(r["topk_idx"], ref["idx"])
    np.testing.assert_allclose(r["topk_w"], ref["w"], rtol=2e-6, atol=1e-7)
    assert np.array_equal(r["counts"], ref["counts"])
    assert np.array_equal(r["offsets"], ref["offsets"])
    assert np.array_equal(r["perm"], ref["perm"])
    assert np.array_equal(r["inv"], ref["inv"])
    assert _rel_err(y, ref["y"]) <= TOL
    st = plan.stats(0)
    assert st["accesses"] == int((ref["counts"] > 0).sum()) and st["pairs"] == T * wl.top_k
    plan.close()


def test_prefill_full_size_sampled():
    """T = 8192 at the prefill shape.  Logits and top-k of a sample of tokens
    bit-exact against the oracle; the grouping (counts, offsets, perm, inv)
    equal to the oracle's grouping of the GPU's top-k; outputs of sampled
    tokens, including ones routed to the busiest and the rarest experts.  A
    token's output depends only on its own row, so the oracle evaluates the
    sampled rows alone."""
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.WORKLOADS["prefill"]
    T = 8192
    plan, info = harness.build_plan(wl, gpu_gen=True)
    wr, bias, _ = info["routers"][0]
    x = W.tokens(wl, 0, 0, T)
    y, r = _run(plan, x, wl)
    samp = np.unique(np.concatenate([np.arange(0, T, 61), [T - 1]]))
    lg = oracle.router_logits(x[samp], wr, bias)
    idx, w = oracle.topk(lg, wl.top_k)
    assert np.array_equal(r["logits"][samp], lg)
    assert np.array_equal(r["topk_idx"][samp], idx)
    np.testing.assert_allclose(r["topk_w"][samp], w, rtol=2e-6, atol=1e-7)
    counts, offsets, perm, inv = oracle.permute(r["topk_idx"], wl.experts)
    assert np.array_equal(r["counts"], counts) and np.array_equal(r["offsets"], offsets)
    assert np.array_equal(r["perm"], perm) and np.array_equal(r["inv"], inv)
    gi = r["topk_idx"]
    busiest, rarest = int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    tok = np.asarray(sorted({0, T - 1, 4097, int(np.nonzero((gi == busiest).any(1))[0][0]),
                             int(np.nonzero((gi == rarest).any(1))[0][0])}))
    experts = [None] * wl.experts
    for e in np.unique(gi[tok]):
        experts[int(e)] = _oracle_expert(wl, 0, int(e))
    ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                      wl.scale_dtype, x[tok], wr, bias, np.arange(len(tok)))
    assert _rel_err(y[tok], ref) <= TOL
    plan.close()


def test_prefill_output_4byte_aligned():
    """The layer output may start on any 4-byte boundary (the ABI's rule for
    y): a y offset by 4 bytes from a 16-byte boundary gets the same bits."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = MID, 300
    plan, info = harness.build_plan(wl, max_tokens=T)
    x = torch.from_numpy(W.tokens(wl, 11, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    plan.forward(0, x, y)
    buf = torch.empty(T * wl.hidden + 8, dtype=torch.bfloat16, device="cuda")
    y2 = buf[2:2 + T * wl.hidden].view(T, wl.hidden)
    assert y2.data_ptr() % 16 == 4
    plan.forward(0, x, y2)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    plan.close()


def test_prefill_host_buffer_forward():
    """T > 8 with page-locked host buffers (copy-engine copies) gives the
    device forward's bits."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = MID, 300
    plan, info = harness.build_plan(wl, max_tokens=T)
    xs = torch.from_numpy(W.tokens(wl, 12, 0, T).view(np.int16).copy())
    x = xs.cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    plan.forward(0, x, y)
    xh, yh = xs.pin_memory(), torch.zeros(T, wl.hidden, dtype=torch.int16).pin_memory()
    plan.forward_host(0, xh, yh)
    torch.cuda.synchronize()
    assert torch.equal(yh, y.view(torch.int16).cpu())
    plan.close()


MIDH = W.Workload("prefill-mid-host", 1, 8, 512, 256, 2, (300,), 4, 64, W.SC_F32, "zipf", 1.0, host_total=4)
MID3H = W.Workload("prefill-mid3-host", 1, 12, 512, 256, 3, (700,), 3, 128, W.SC_BF16, "zipf", 1.0,
                   host_total=7)


@pytest.mark.parametrize("wl,T", [(MIDH, 300), (MID3H, 700)])
def test_prefill_host_resident(wl, T):
    """Experts in pinned host memory are read in place by the prefill GEMMs
    (16-byte cp.async of their code blocks instead of bulk copies): the layer
    output is bit-identical to a plan with every expert in HBM, within
    tolerance of the oracle, and the forward counts each routed host expert as
    a miss."""
    import torch
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(wl, max_tokens=T)
    ref_plan, _ = harness.build_plan(wl, max_tokens=T, all_hbm=True)
    wr, bias, _ = info["routers"][0]
    host = info["host_sets"][0]
    assert len(host) == wl.host_total
    x = W.tokens(wl, 3 + T, 0, T)
    y, r = _run(plan, x, wl)
    y_ref, _ = _run(ref_plan, x, wl)
    assert np.array_equal(y, y_ref)
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert _rel_err(y, ref["y"]) <= TOL
    routed = set(int(e) for e in np.nonzero(ref["counts"])[0])
    assert routed & host, "the case must route tokens to host-resident experts"
    st = plan.stats(0)
    assert st["misses"] == len(routed & host) and st["hits"] == len(routed - host)
    plan.close()
    ref_plan.close()


WIDEP = W.Workload("prefill-wide", 1, 600, 256, 128, 5, (40,), 4, 64, W.SC_F32, "zipf", 1.0)


def test_prefill_wide_router():
    """More experts than the register path of the prefill top-k holds (E > 512):
    routing bit-exact, outputs of the layer within tolerance."""
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = WIDEP, 40
    plan, info = harness.build_plan(wl, max_tokens=T)
    wr, bias, _ = info["routers"][0]
    x = W.tokens(wl, 17, 0, T)
    y, r = _run(plan, x, wl)
    lg = oracle.router_logits(x, wr, bias)
    idx, w = oracle.topk(lg, wl.top_k)
    assert np.array_equal(r["logits"], lg)
    assert np.array_equal(r["topk_idx"], idx)
    np.testing.assert_allclose(r["topk_w"], w, rtol=2e-6, atol=1e-7)
    counts, offsets, perm, inv = oracle.permute(idx, wl.experts)
    assert np.array_equal(r["counts"], counts) and np.array_equal(r["offsets"], offsets)
    assert np.array_equal(r["perm"], perm) and np.array_equal(r["inv"], inv)
    experts = [_oracle_expert(wl, 0, e) if e in np.unique(idx) else None for e in range(wl.experts)]
    ref = oracle.layer_forward_tokens(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                                      wl.scale_dtype, x, wr, bias, np.arange(T))
    assert _rel_err(y, ref) <= TOL
    plan.close()


def test_prefill_hidden_17_blocks():
    """H = 4352 (17 code blocks of 256 columns, 68 stages per gate/up unit)."""
    from moe_expert_layer_sorted_gb300 import harness
    wl = W.Workload("prefill-long-h", 1, 16, 4352, 256, 2, (24,), 3, 128, W.SC_BF16, "plain")
    T = 24
    plan, info = harness.build_plan(wl, max_tokens=T)
    wr, bias, _ = info["routers"][0]
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    x = W.tokens(wl, 5, 0, T)
    y, r = _run(plan, x, wl)
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["logits"], ref["logits"])
    assert np.array_equal(r["perm"], ref["perm"])
    assert _rel_err(y, ref["y"]) <= TOL
    plan.close()


@pytest.mark.parametrize("mode", ["offset8", "offset64", "outliers"])
def test_prefill_activation_edge_cases(mode):
    """Prefill with offset or outlying activations (c + N(0,1), or +-1000 in
    eight columns): routing bit-exact, outputs within tolerance."""
    from moe_expert_layer_sorted_gb300 import harness
    wl, T = MID3, 300
    plan, info = harness.build_plan(wl, max_tokens=T)
    wr, bias, _ = info["routers"][0]
    experts = [_oracle_expert(wl, 0, e) for e in range(wl.experts)]
    x = oracle.bf16_to_f32(W.tokens(wl, 8100, 0, T)).astype(np.float32)
    if mode.startswith("offset"):
        x = x + np.float32(int(mode[6:]))
    else:
        cols = np.random.default_rng(5).choice(wl.hidden, 8, replace=False)
        x[:, cols] = np.where(np.arange(8) % 2 == 0, 1000.0, -1000.0).astype(np.float32)
    x = oracle.f32_to_bf16(x)
    y, r = _run(plan, x, wl)
    ref = oracle.layer_forward(experts, wl.hidden, wl.inter, wl.top_k, wl.bits, wl.group,
                               wl.scale_dtype, x, wr, bias)
    assert np.array_equal(r["logits"], ref["logits"])
    assert np.array_equal(r["topk_idx"], ref["idx"])
    assert np.array_equal(r["perm"], ref["perm"])
    assert _rel_err(y, ref["y"]) <= TOL
    plan.close()
