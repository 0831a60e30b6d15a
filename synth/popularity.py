"""Router-bias calibration for the skewed-popularity workloads (an input recipe).

The pages' cached decode relies on expert access being heavily skewed
("Running a 24k-expert MoE on a single 32 GB card", section 3: a cache of ~70 %
of the experts serves 97.8-99.7 % of reads because the hot set is obvious),
and the 384-expert layer keeps its least-used 30 % in host memory ("763B MoE in
two 96 GB cards", section "Where the VRAM gap comes from").  The workloads model
that skew as Zipf(s) popularity: a token's k experts are drawn without
replacement with probability proportional to p_r = (r+1)^-s / Z (rank r = 0 is
the most popular) -- the Plackett-Luce model.

The synthetic router produces logits bias[e] + x . Wr[e] whose noise term
x . Wr[e] is (for x ~ N(0,1) and Gaussian Wr) close to independent N(0, sd^2)
per expert.  Gaussian noise has light tails, so the plain choice bias = log p
starves the rare experts (Plackett-Luce is exact only for Gumbel noise).  This
module computes, per rank, the bias for which top-k of (bias + sd * z), z
independent standard normal, includes each expert with exactly the
Plackett-Luce inclusion probability of its rank.

Both inclusion probabilities are one-dimensional integrals over the threshold
value v: expert i is among the k largest iff its value v exceeds all but at
most k-1 of the others, so

    P(i in top-k) = integral f_i(v) * P(#{j != i : l_j > v} <= k-1) dv,

where the count is a Poisson-binomial variable, evaluated by a truncated
dynamic programme over the experts (prefix and suffix tables, so every
leave-one-out count costs O(k^2)).  Plackett-Luce is the Gumbel case of the
same integral (Gumbel-max trick): l_j = log p_j + Gumbel(0, 1).

Nothing here touches layer data: it turns (E, k, s, sd) into a bias table.
"""
from __future__ import annotations

import functools
import math

import numpy as np

_SQRT2 = math.sqrt(2.0)


def _gauss_tail(z: np.ndarray) -> np.ndarray:
    """P(Z > z) for a standard normal Z (erfc form: accurate in the far tail)."""
    from scipy.special import erfc
    return 0.5 * erfc(z / _SQRT2)


def _inclusion(tail: np.ndarray, dens: np.ndarray, dv: float, k: int, with_slope: bool = False):
    """P(i in top-k) for every i, from tail[i, g] = P(l_i > v_g) and dens[i, g]
    = the density of l_i at v_g on a uniform grid of spacing dv.  With
    with_slope, also d P(i in top-k) / d(location of l_i): the integral of
    dens[i] times the v-derivative of the leave-one-out count probability."""
    E, G = tail.shape
    pre = np.zeros((E + 1, G, k))      # pre[i][g, m] = P(m of experts < i exceed v_g), m < k
    pre[0, :, 0] = 1.0
    for i in range(E):
        q = tail[i][:, None]
        pre[i + 1] = pre[i] * (1.0 - q)
        pre[i + 1][:, 1:] += pre[i][:, :-1] * q
    suf = np.zeros((E + 1, G, k))      # suf[i][g, m] = P(m of experts >= i exceed v_g)
    suf[E, :, 0] = 1.0
    for i in range(E - 1, -1, -1):
        q = tail[i][:, None]
        suf[i] = suf[i + 1] * (1.0 - q)
        suf[i][:, 1:] += suf[i + 1][:, :-1] * q
    csuf = np.cumsum(suf, axis=2)      # P(at most m of experts >= i exceed v)
    # at most k-1 of the others: a from those below i, at most k-1-a from those above
    ok = np.einsum("igm,igm->ig", pre[:E], csuf[1:, :, ::-1])
    incl = (dens * ok).sum(axis=1) * dv
    if not with_slope:
        return incl
    slope = (dens * np.gradient(ok, dv, axis=1)).sum(axis=1) * dv
    return incl, slope


def plackett_luce_inclusion(E: int, k: int, s: float, step: float = 0.02) -> np.ndarray:
    """P(rank r among the k drawn) for k draws without replacement with
    probabilities proportional to (r+1)^-s, r = 0 .. E-1."""
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    mu = np.log(p / p.sum())
    v = np.arange(mu.min() - 5.0, mu.max() + 24.0, step)
    z = v[None, :] - mu[:, None]
    ez = np.exp(-z)
    tail = -np.expm1(-ez)              # 1 - exp(-e^-z): P(Gumbel > z)
    dens = np.exp(-z - ez)
    return _inclusion(tail, dens, step, k)


def gaussian_inclusion(bias: np.ndarray, sd: float, k: int, step: float | None = None,
                       with_slope: bool = False):
    """P(i among the k largest of bias[i] + sd * z_i), z_i independent N(0, 1)
    (and, with_slope, its derivative with respect to bias[i])."""
    b = np.asarray(bias, dtype=np.float64)
    step = step or sd / 40.0
    v = np.arange(b.min() - 9.0 * sd, b.max() + 9.0 * sd, step)
    z = (v[None, :] - b[:, None]) / sd
    tail = _gauss_tail(z)
    dens = np.exp(-0.5 * z * z) / (sd * math.sqrt(2.0 * math.pi))
    return _inclusion(tail, dens, step, k, with_slope)


@functools.lru_cache(maxsize=None)
def calibrated_rank_bias(E: int, k: int, s: float, sd: float, iters: int = 40) -> tuple:
    """Bias per popularity rank r (0 = most popular) such that top-k of
    bias + sd * N(0,1) includes rank r with its Plackett-Luce Zipf(s)
    probability.  Damped diagonal Newton steps on log inclusion (each
    expert's inclusion rises monotonically with its own bias; the coupling
    through the others is weak), shifted so that rank 0's bias is 0.
    Returns (bias tuple, max |log(achieved / target)|)."""
    target = plackett_luce_inclusion(E, k, s)
    b = sd * np.log(target / target[0])
    err = math.inf
    for _ in range(iters):
        got, slope = gaussian_inclusion(b, sd, k, with_slope=True)
        d = np.log(target) - np.log(np.maximum(got, 1e-300))
        err = float(np.abs(d).max())
        if err < 1e-4:
            break
        step = d * got / np.maximum(slope, 1e-12)
        b = b + np.clip(step, -0.5 * sd, 0.5 * sd)
        b -= b[0]
    return tuple(float(t) for t in b), err
