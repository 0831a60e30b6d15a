"""The error bound the prefill router uses to decide which router logits it
recomputes in the library's fixed order (the router of "763B MoE in two 96 GB
cards", section "Where the VRAM gap comes from": each token routed to the k of
E experts with the largest logits x . Wr[e] + b[e]).  The GPU takes
approximate logits from a bf16 tensor-core GEMM with fp32 accumulation in an
order it does not control, and treats

    d = H 2^-20 ||x|| ||w_e|| + 2^-21 |b_e| + 2^-100

as a bound on |approximate logit + bias - fixed-order logit|.  Here the bound
is checked against accumulation models written out on the CPU: blocks of n
products added to the running sum after aligning every term to the largest
exponent and truncating, with the sum truncated to fp32 (no guard bits: the
weakest tensor-core adder model the bound assumes), plain sequential fp32
sums rounded to nearest, and pairwise fp32 sums -- on Gaussian rows, rows with
a large common offset (heavy cancellation), rows with outlying columns and
rows whose products are all positive (a truncating adder's errors then add
up at every step), against the oracle's fixed-order logits.  On these rows the
weakest model reaches about 1.4 % of d at H = 4096; d itself is four times
the worst case of the analysis (every partial sum as large as sum |x_i w_i|)."""
import numpy as np
import pytest

import oracle


def _trunc_f32(v):
    """v (float64) truncated toward zero to a 24-bit significand."""
    m, e = np.frexp(v)
    ulp = np.ldexp(1.0, e - 24)
    return np.where(v == 0.0, 0.0, np.trunc(v / ulp) * ulp)


def _block_truncating(p, n):
    """Sum over the last axis of p (float64 products) in blocks of n: each block
    and the running sum aligned to the block's largest exponent and truncated,
    the sum truncated to fp32."""
    acc = np.zeros(p.shape[0])
    for c in range(0, p.shape[1], n):
        terms = np.concatenate([acc[:, None], p[:, c:c + n]], axis=1)
        big = np.max(np.abs(terms), axis=1)
        _, e = np.frexp(big)
        ulp = np.where(big > 0, np.ldexp(1.0, e - 24), 1.0)
        aligned = np.trunc(terms / ulp[:, None]) * ulp[:, None]
        acc = _trunc_f32(aligned.sum(axis=1))
    return acc


def _sequential_f32(p):
    acc = np.zeros(p.shape[0], dtype=np.float32)
    for c in range(p.shape[1]):
        acc = (acc + p[:, c].astype(np.float32)).astype(np.float32)
    return acc.astype(np.float64)


def _pairwise_f32(p):
    return np.sum(p.astype(np.float32), axis=1, dtype=np.float32).astype(np.float64)


def _rows(kind, T, H, rng):
    x = rng.standard_normal((T, H)).astype(np.float32)
    if kind == "offset":
        x += 50.0
    elif kind == "positive":  # with positive router rows: every product positive, so a
        x = np.abs(x) + 1.0   # truncating adder errs the same way at every step
    elif kind == "outliers":
        cols = rng.choice(H, 8, replace=False)
        x[:, cols] = np.where(np.arange(8) % 2 == 0, 1000.0, -1000.0)
    return oracle.f32_to_bf16(x)


@pytest.mark.parametrize("H", [256, 4096])
@pytest.mark.parametrize("kind", ["gaussian", "offset", "outliers", "positive"])
def test_router_bound_covers_the_accumulation_models(H, kind):
    rng = np.random.default_rng(H + len(kind))
    T, E = 24, 16
    x = _rows(kind, T, H, rng)
    w = rng.standard_normal((E, H)).astype(np.float32) * np.float32(np.pi / np.sqrt(6.0) / np.sqrt(H))
    if kind == "positive":
        w = np.abs(w) + np.float32(1.0 / np.sqrt(H))
    w[1] = w[0]
    w[2] = w[0] * np.float32(1.0 + 2.0 ** -7)  # near-duplicate rows
    wr = oracle.f32_to_bf16(w)
    bias = (rng.standard_normal(E) * 2.0).astype(np.float32)
    F = oracle.router_logits(x, wr, bias).astype(np.float64)  # fixed order, bias added last
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    wf = oracle.bf16_to_f32(wr).astype(np.float64)
    p = (xf[:, None, :] * wf[None, :, :]).reshape(T * E, H)  # exact products
    nx = np.sqrt((xf * xf).sum(axis=1))
    nw = np.sqrt((wf * wf).sum(axis=1))
    d = (H * 2.0 ** -20 * nx[:, None] * nw[None, :] + 2.0 ** -21 * np.abs(bias)[None, :] + 2.0 ** -100)
    models = {f"block{n}": _block_truncating(p, n) for n in (1, 4, 8, 16)}
    models["sequential"] = _sequential_f32(p)
    models["pairwise"] = _pairwise_f32(p)
    worst = 0.0
    for name, a in models.items():
        A = (a.reshape(T, E).astype(np.float32) + bias[None, :]).astype(np.float64)  # bias in fp32
        err = np.abs(A - F)
        assert np.all(err <= d), (name, float((err / d).max()))
        worst = max(worst, float((err / d).max()))
    # the bound is a bound, not a guess: the weakest model comes within a few
    # factors of it on these rows, none exceeds it
    assert worst < 1.0
