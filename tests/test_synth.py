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


def test_plackett_luce_inclusion_closed_forms():
    """Inclusion probabilities of k draws without replacement, p_r ~ (r+1)^-s:
    they sum to k; k = 1 is the categorical law p_r itself; s = 0 is uniform k/E;
    k = E includes everyone."""
    from synth import popularity as P
    for E, k, s in ((384, 6, 1.0), (512, 8, 1.2), (40, 3, 0.7)):
        t = P.plackett_luce_inclusion(E, k, s)
        assert abs(t.sum() - k) < 1e-6
        assert np.all(np.diff(t) < 0)
    p = np.arange(1, 101, dtype=np.float64) ** -1.0
    np.testing.assert_allclose(P.plackett_luce_inclusion(100, 1, 1.0), p / p.sum(), rtol=1e-6)
    np.testing.assert_allclose(P.plackett_luce_inclusion(50, 4, 0.0), np.full(50, 4 / 50), rtol=1e-6)
    np.testing.assert_allclose(P.plackett_luce_inclusion(6, 6, 1.0), np.ones(6), rtol=1e-6)


def test_plackett_luce_inclusion_against_sequential_draws():
    """The integral equals the frequency of sequential draws without
    replacement (each draw proportional to the remaining weights)."""
    from synth import popularity as P
    E, k, s, n = 12, 3, 1.0, 200_000
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    rng = np.random.default_rng(7)
    hits = np.zeros(E)
    u = rng.random((n, k))
    for i in range(n):
        w = p.copy()
        for j in range(k):
            c = np.cumsum(w)
            r = int(np.searchsorted(c, u[i, j] * c[-1], side="right"))
            hits[r] += 1
            w[r] = 0.0
    freq = hits / n
    t = P.plackett_luce_inclusion(E, k, s)
    assert np.all(np.abs(freq - t) < 5 * np.sqrt(t * (1 - t) / n) + 1e-4)


def test_gaussian_inclusion_closed_forms():
    from synth import popularity as P
    g = P.gaussian_inclusion(np.zeros(30), 1.3, 4)
    np.testing.assert_allclose(g, np.full(30, 4 / 30), rtol=1e-6)
    # two experts, k = 1: P(l_0 > l_1) = Phi((b0 - b1) / (sd sqrt 2))
    from scipy.special import ndtr
    g2 = P.gaussian_inclusion(np.array([0.5, 0.0]), 1.0, 1)
    np.testing.assert_allclose(g2[0], ndtr(0.5 / np.sqrt(2.0)), rtol=1e-6)
    b = np.linspace(0.0, -4.0, 64)
    assert abs(P.gaussian_inclusion(b, 1.2, 5).sum() - 5) < 1e-6


def test_zipf_router_realises_the_plackett_luce_host_share():
    """The decode layer's synthetic router (seeded x ~ N(0,1) against its Wr,
    plus the calibrated bias; top-k in fp64 here) routes the 115 least popular
    experts -- the host-resident ones -- at the Plackett-Luce Zipf(1.0) share
    of the slots, and puts some host expert in the top-6 of a single token
    about as often as Plackett-Luce draws do."""
    from synth import popularity as P
    wl = W.WORKLOADS["decode"]
    wr, bias, rank = W.router(wl, 0)
    host = np.zeros(wl.experts, bool)
    host[W.host_experts(wl, 0, rank)] = True
    n = 3000
    x = synth.bf16_to_f32(W.tokens(wl, 123, 0, n)).astype(np.float64)
    lg = x @ synth.bf16_to_f32(wr).astype(np.float64).T + bias.astype(np.float64)
    top = np.argsort(-lg, axis=1, kind="stable")[:, : wl.top_k]
    share = host[top].mean()
    t = P.plackett_luce_inclusion(wl.experts, wl.top_k, wl.zipf_s)
    target = t[wl.experts - wl.host_count(0):].sum() / wl.top_k
    assert abs(share - target) < 0.15 * target, (share, target)
    # P(any host expert among a token's 6) by Gumbel-perturbed log-popularity
    rng = np.random.default_rng(3)
    p = np.arange(1, wl.experts + 1, dtype=np.float64) ** -wl.zipf_s
    g = np.log(p)[None, :] + rng.gumbel(size=(20000, wl.experts))
    pl_any = (np.argsort(-g, axis=1)[:, : wl.top_k] >= wl.experts - wl.host_count(0)).any(1).mean()
    any_host = host[top].any(1).mean()
    assert abs(any_host - pl_any) < 0.15 * pl_any, (any_host, pl_any)
    print(f"host share of slots {share:.4f} (Plackett-Luce {target:.4f}); "
          f"P(any host expert per token) {any_host:.3f} (Plackett-Luce {pl_any:.3f})")
