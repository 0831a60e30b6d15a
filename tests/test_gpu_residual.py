"""The forward with the residual update fused into its combine
(moe_layer_forward_residual): y bit for bit the plain forward's, and
out = bf16(y + residual) rounded to nearest even, on both the decode (T <= 8)
and the prefill path, with host-resident experts in the layer."""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

# 8 experts, 3 of them in pinned host memory; H spans two 256-column blocks
WL = W.Workload("residual-mid", 1, 8, 512, 256, 2, (300,), 4, 64, W.SC_F32, "zipf", 1.0, host_total=3)


@pytest.fixture(scope="module")
def mid():
    from moe_expert_layer_sorted_gb300 import harness
    plan, info = harness.build_plan(WL, max_tokens=300)
    yield plan
    plan.close()


def _residual(T, H, seed):
    """fp32 residual of mixed magnitude (|r| from ~1e-3 to ~1e3)."""
    rng = np.random.default_rng(seed)
    r = rng.standard_normal((T, H)).astype(np.float32) * (10.0 ** rng.uniform(-3, 3, (T, H))).astype(np.float32)
    return r


@pytest.mark.parametrize("T", [1, 4, 8, 9, 300])
def test_residual_forward(mid, T):
    import torch
    plan = mid
    H = WL.hidden
    x = torch.from_numpy(W.tokens(WL, 40 + T, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y_ref = torch.empty_like(x)
    plan.forward(0, x, y_ref)
    torch.cuda.synchronize()
    yb = y_ref.view(torch.int16).cpu().numpy().view(np.uint16)
    r = _residual(T, H, T)
    r[:, :7] = -oracle.bf16_to_f32(yb[:, :7])  # exact cancellation: +0
    res = torch.from_numpy(r).cuda()
    y = torch.full_like(x, 7.0)
    out = torch.full_like(x, 7.0)
    plan.forward_residual(0, x, y, res, out)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    want = oracle.f32_to_bf16(oracle.bf16_to_f32(yb) + r)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), want)


def test_residual_forward_rejects_bad_buffers(mid):
    import torch
    from moe_expert_layer_sorted_gb300 import MoeError
    plan = mid
    T, H = 4, WL.hidden
    x = torch.from_numpy(W.tokens(WL, 3, 0, T).view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.empty_like(x)
    res = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError, match="MOE_ERR_INVALID"):
        plan.forward_residual(0, x, y, res, y)  # out is y
    big = torch.zeros(T * H + 8, dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError, match="MOE_ERR_INVALID"):
        plan.forward_residual(0, x, y, big[1:1 + T * H].view(T, H), torch.empty_like(x))  # 4-byte aligned
    torch.cuda.synchronize()
