"""Pins of the oracle's quantiser against hand-worked cases and the
quantisation error bound (one step; half a step when not clamped)."""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN

DT = {"f32": oracle.SC_F32, "bf16": oracle.SC_BF16, "f16": oracle.SC_F16}


def _scale_value(raw, dtype):
    if dtype == oracle.SC_F32:
        return raw.astype(np.float32)
    if dtype == oracle.SC_BF16:
        return oracle.bf16_to_f32(raw)
    return raw.view(np.float16).astype(np.float32)


def _unpack(codes, n, bits):
    bitsarr = np.unpackbits(codes, bitorder="little")
    return np.array([int(sum(int(bitsarr[i * bits + j]) << j for j in range(bits))) for i in range(n)])


CASES = json.load(open(os.path.join(GOLDEN, "quantiser_cases.json")))["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["why"][:40] for c in CASES])
def test_hand_cases(case):
    w = np.array([case["w"]], dtype=np.float32)
    dt = DT[case["dtype"]]
    codes, scales = oracle.quantize(w, case["bits"], case["group"], dt)
    s = _scale_value(scales.ravel(), dt)[0]
    assert s == pytest.approx(case["scale"], rel=1e-6, abs=0)
    off = 1 << (case["bits"] - 1)
    q = _unpack(codes, w.size, case["bits"]) - off
    assert list(q) == case["q"]
    if "codes_hex" in case:
        assert codes.tobytes().hex() == case["codes_hex"]
    if "dequant" in case:
        wh = oracle.dequantize(codes, scales, 1, w.size, case["bits"], case["group"], dt)
        np.testing.assert_allclose(wh.ravel(), case["dequant"], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("bits,group,dtype", [(4, 32, oracle.SC_F32), (3, 128, oracle.SC_BF16),
                                              (2, 64, oracle.SC_F16), (4, 128, oracle.SC_BF16)])
def test_error_within_one_step(bits, group, dtype):
    rng = np.random.default_rng(7)
    rows, cols = 16, 512
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    w[3, :group] = 0.0                                      # an all-zero group
    w[5, 7] = 0.5                                           # an outlier dominating its group
    codes, scales = oracle.quantize(w, bits, group, dtype)
    wh = oracle.dequantize(codes, scales, rows, cols, bits, group, dtype)
    s = np.repeat(_scale_value(scales.reshape(rows, -1), dtype), group, axis=1)
    qmax = (1 << (bits - 1)) - 1
    err = np.abs(wh - w)
    # every weight within one step, and within half a step where w/s is not clamped
    assert np.all(err <= s * (1 + 1e-6))
    unclamped = np.abs(w) <= qmax * s
    assert np.all(err[unclamped] <= s[unclamped] * (0.5 + 1e-6))
    assert np.all(wh[3, :group] == 0)
    # codes stay in the restricted symmetric range
    off = 1 << (bits - 1)
    u = _unpack(codes, rows * cols, bits)
    assert u.min() >= off - qmax and u.max() <= off + qmax


def test_roundtrip_of_representable_weights():
    # weights that are exact multiples of a power-of-two scale quantise exactly
    rng = np.random.default_rng(3)
    q = rng.integers(-7, 8, size=(8, 64))
    q[:, ::32] = 7                      # make amax = 7 * s in every group
    w = (q * 0.125).astype(np.float32)
    codes, scales = oracle.quantize(w, 4, 32, oracle.SC_F32)
    wh = oracle.dequantize(codes, scales, 8, 64, 4, 32, oracle.SC_F32)
    assert np.array_equal(wh, w)


def test_bad_shapes_rejected():
    w = np.zeros((2, 30), np.float32)
    with pytest.raises(ValueError):
        oracle.quantize(w, 4, 32, oracle.SC_F32)
