"""The input generator's device twin draws exactly the host generator's values
(fp32 and bf16), so large stacks can be generated on the GPU with the same
weights the oracle would see."""
import numpy as np
import pytest

import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,start,sigma", [(1, 0, 1.0), (4099, 17, 0.02), (1 << 20, 123456, 0.05)])
def test_device_draws_match_host(n, start, sigma):
    import torch
    k = synth.key(7, synth.TAG_WEIGHT, 3, 11, 2)
    ref = synth.normal_f32(k, n, sigma, start=start)
    d = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.normal_f32_device(k, n, sigma, d.data_ptr(), torch.cuda.current_stream().cuda_stream, start=start)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    refb = synth.normal_bf16(k, n, sigma, start=start)
    db = torch.empty(n, dtype=torch.int16, device="cuda")
    synth.normal_bf16_device(k, n, sigma, db.data_ptr(), torch.cuda.current_stream().cuda_stream, start=start)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(db.cpu().numpy().view(np.uint16), refb)


def test_expert_master_on_device():
    import torch
    wl = W.WORKLOADS["decode"]
    r, c = wl.matrix_shape(2)
    d = torch.empty(r * c, dtype=torch.float32, device="cuda")
    synth.normal_f32_device(W.key(wl.seed, W.TAG_WEIGHT, 5, 17, 2), r * c, wl.w_sigma, d.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d.cpu().numpy().reshape(r, c), W.expert_master(wl, 5, 17, 2))


def test_residual_bf16_matches_torch():
    """The chained-layer input bf16(float(y) + noise), one device kernel, bit for bit
    the value of the same fp32 add rounded by torch."""
    import torch
    import synth
    n = 3 * 4096 + 7
    g = torch.Generator(device="cpu").manual_seed(3)
    y = (torch.randn(n, generator=g) * 4).to(torch.bfloat16).cuda()
    noise = torch.randn(n, generator=g).cuda()
    out = torch.empty_like(y)
    synth.residual_bf16_device(y.data_ptr(), noise.data_ptr(), n, out.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    ref = (y.float() + noise).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
