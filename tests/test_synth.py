"""The seeded generator: counter-based (slices regenerate identically),
thread-count independent, and of the stated mean and spread."""
import numpy as np

import synth
from synth import workloads as W


def test_counter_based_slices():
    k = synth.key(0, synth.TAG_WEIGHT, 1, 2, 0)
    full = synth.normal_f32(k, 3_000_000, 0.02)
    part = synth.normal_f32(k, 1000, 0.02, start=2_500_000)
    np.testing.assert_array_equal(full[2_500_000:2_501_000], part)


def test_moments():
    v = synth.normal_f32(synth.key(1, 2, 3, 4, 5), 2_000_000, 1.0).astype(np.float64)
    assert abs(v.mean()) < 3e-3 and abs(v.std() - 1.0) < 3e-3
    assert np.abs(v).max() <= 3.47


def test_zipf_bias_is_a_distribution():
    bias, rank = synth.zipf_bias(synth.key(0, synth.TAG_BIAS, 0), 384, 1.0)
    p = np.exp(bias.astype(np.float64))
    assert abs(p.sum() - 1.0) < 1e-5
    assert sorted(rank.tolist()) == list(range(384))
    assert np.argmax(p) == np.argmin(rank)


def test_workload_byte_counts():
    # per-expert algorithmic bytes (codes + scales of gate, up, down)
    assert W.WORKLOADS["tiny"].expert_bytes == 61_440
    assert W.WORKLOADS["decode"].expert_bytes == 4_915_200
    assert W.WORKLOADS["prefill"].expert_bytes == 6_488_064
    assert W.WORKLOADS["cached"].expert_bytes == 884_736
    assert W.WORKLOADS["cached"].cache_slots == 17_203
    s = W.WORKLOADS["stack40"]
    assert sum(s.host_count(l) for l in range(40)) == 4608
    assert {s.host_count(l) for l in range(40)} == {115, 116}
