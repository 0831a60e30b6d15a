"""The host-CPU expert FFN (the comparison against reading host-resident
experts over the GPU's link) against the oracle: the same quantised expert,
the oracle's fp64 FFN on the dequantised weights, relative error of an fp32
computation.  CPU only."""
import numpy as np
import pytest

import oracle
from moe_expert_layer_sorted_gb300 import cpu_expert
from synth import workloads as W


@pytest.mark.parametrize("H,I,bits,G,sdt", [(256, 128, 4, 32, W.SC_F32), (512, 256, 3, 128, W.SC_BF16),
                                            (256, 256, 2, 64, W.SC_F16)])
@pytest.mark.parametrize("T,threads", [(1, 1), (3, 2), (8, 3)])
def test_cpu_expert_matches_oracle(H, I, bits, G, sdt, T, threads):
    rng = np.random.default_rng(H + I + bits + T)
    codes, scales, deq = [], [], []
    for rows, cols in ((I, H), (I, H), (H, I)):
        w = rng.normal(0.0, 0.02, (rows, cols)).astype(np.float32)
        c, s = oracle.quantize(w, bits, G, sdt)
        codes.append(c)
        scales.append(s)
        deq.append(oracle.dequantize(c, s, rows, cols, bits, G, sdt))
    x = oracle.f32_to_bf16(rng.normal(0.0, 1.0, (T, H)).astype(np.float32))
    got = cpu_expert.expert_ffn(codes, scales, H, I, bits, G, sdt, x, threads=threads)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    for t in range(T):
        ref = oracle.expert_ffn(deq[0], deq[1], deq[2], xf[t])
        err = np.abs(got[t].astype(np.float64) - ref).max() / np.abs(ref).max()
        assert err < 1e-5, (t, err)


def test_cpu_expert_rejects_bad_shapes():
    z = np.zeros(64, np.uint8)
    s = np.zeros(64, np.float32)
    x = np.zeros((1, 256), np.uint16)
    with pytest.raises(ValueError):
        cpu_expert.expert_ffn([z] * 3, [s] * 3, 256, 128, 5, 32, 0, x)  # 5-bit codes
    with pytest.raises(ValueError):
        cpu_expert.expert_ffn([z] * 3, [s] * 3, 256, 100, 4, 32, 0, x)  # I not a multiple of G
