"""The precision reading for the CTA pair's score exchange, checked on the CPU.

The decode splits every score between two CTAs: CTA r holds the partial dot
product over latent columns [256r, 256r+256) and rope columns [512+32r,
512+32r+32).  Each sends its partial to the other as a 24-bit code, the
float32 value with its low 8 mantissa bits rounded to nearest (relative error
at most 2^-16).  The claim: the log-sum-exp of a row then moves by at most
2^-16 times the largest partial logit of the row (the LSE is 1-Lipschitz in
the largest score error), which keeps it inside the 2e-3 tolerance for
partial logits up to about 130 in natural-log units.

These tests restate the rounding in NumPy, apply it to one partial of each
score, and compare the row LSE with the exact float64 one, from ordinary to
very sharp attention.  They exercise the arithmetic of the reading, not the
CUDA path (the GPU parity tests cover that).
"""

import numpy as np
import pytest

SCALE = 1.0 / np.sqrt(192.0)
LATENT, ROPE = 512, 64


def to_24bit(x32, guard=True):
    """float32 -> float32 keeping the top 24 bits, rounded to nearest on the
    dropped 8 (the exchange code, restated).  Infinities and NaN (exponent all
    ones) are truncated instead of rounded, and a NaN keeps a non-zero
    mantissa (the lowest code bit is set when the payload was non-zero);
    ``guard=False`` restates the code without that exception."""
    bits = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    code = ((bits + 0x80) & 0xFFFFFFFF) >> 8
    if guard:
        special = (bits >> 8) | ((bits & 0x007FFFFF) != 0).astype(np.uint64)
        code = np.where((bits & 0x7F800000) == 0x7F800000, special, code)
    return ((code << 8) & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def partial_scores(q, kv):
    """Raw partial dot products of the two CTAs, float64: [rows, keys] each."""
    c0 = np.r_[0:256, LATENT:LATENT + 32]
    c1 = np.r_[256:512, LATENT + 32:LATENT + ROPE]
    return q[:, c0] @ kv[:, c0].T, q[:, c1] @ kv[:, c1].T


def lse(s):
    m = s.max(axis=1, keepdims=True)
    return (m[:, 0] + np.log(np.exp(s - m).sum(axis=1)))


def test_rounding_error_is_at_most_2_pow_minus_16():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * 10.0 ** rng.uniform(-3, 4, 200_000)).astype(np.float32)
    y = to_24bit(x).astype(np.float64)
    rel = np.abs(y - x) / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -16
    # rounding, not truncation: the error is symmetric
    assert abs(np.mean(np.sign(y - x))) < 0.05


@pytest.mark.parametrize("sharpness", [1.0, 4.0, 16.0, 40.0])
def test_lse_moves_by_at_most_the_largest_partial_error(sharpness):
    rng = np.random.default_rng(int(sharpness))
    rows, keys = 64, 700
    q = rng.standard_normal((rows, LATENT + ROPE)) * sharpness
    kv = rng.standard_normal((keys, LATENT + ROPE))
    s0, s1 = partial_scores(q, kv)
    exact = lse(SCALE * (s0 + s1))
    # the kernel's view: both partials in float32, the peer's through the exchange
    s0_32 = s0.astype(np.float32).astype(np.float64)
    s1_24 = to_24bit(s1.astype(np.float32)).astype(np.float64)
    got = lse(SCALE * (s0_32 + s1_24))
    # float32 rounding of each partial (2^-24) plus the exchange code (2^-16)
    bound = SCALE * (np.abs(s1).max(axis=1) * (2.0 ** -16 + 2.0 ** -24) + np.abs(s0).max(axis=1) * 2.0 ** -24)
    assert np.all(np.abs(got - exact) <= bound * (1 + 1e-6) + 1e-12)
    peak = SCALE * np.abs(s1).max()
    if peak <= 130.0:
        assert np.abs(got - exact).max() < 2e-3, peak


def test_fp16_exchange_would_break_the_bound_on_sharp_rows():
    """The rejected half-precision exchange (relative error 2^-11) leaves the
    2e-3 bound once partial logits reach the tens; the 24-bit code does not."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((64, LATENT + ROPE)) * 6.0
    kv = rng.standard_normal((700, LATENT + ROPE))
    s0, s1 = partial_scores(q, kv)
    exact = lse(SCALE * (s0 + s1))
    assert SCALE * np.abs(s1).max() > 20.0
    half = lse(SCALE * (s0 + s1.astype(np.float16).astype(np.float64)))
    code24 = lse(SCALE * (s0 + to_24bit(s1.astype(np.float32)).astype(np.float64)))
    assert np.abs(half - exact).max() > 2e-3
    assert np.abs(code24 - exact).max() <= 2.0 ** -16 * SCALE * np.abs(s1).max() * 1.01
    assert np.abs(code24 - exact).max() < 2e-3


def test_non_finite_scores_cross_unchanged():
    """An infinite partial stays that infinity and a NaN stays NaN (with its
    sign), so both CTAs of the pair see the same non-finite score.  Rounding
    them like finite values would not: the canonical NaN 0x7FFFFFFF carries
    into the sign bit and arrives as -0.0, and a negative NaN wraps to +0."""
    bits = np.array([0x7F800000, 0xFF800000, 0x7FFFFFFF, 0xFFFFFFFF, 0x7FC00000, 0x7F800001, 0xFF800080,
                     0x7F7FFFFF], dtype=np.uint32)
    x = bits.view(np.float32)
    y = to_24bit(x)
    assert y[0] == np.inf and y[1] == -np.inf
    assert np.all(np.isnan(y[2:7]))
    assert np.array_equal(np.signbit(y[2:7]), np.signbit(x[2:7]))
    # the largest finite value rounds up to infinity, as round-to-nearest does
    assert y[7] == np.inf
    bad = to_24bit(x, guard=False)
    assert bad[2] == 0.0 and np.signbit(bad[2]) and bad[3] == 0.0  # what the guard prevents
    # a NaN whose payload is only in the dropped bits would become infinite
    # if it were truncated without keeping a payload bit
    trunc = ((bits.astype(np.uint64) >> 8) << 8).astype(np.uint32).view(np.float32)
    assert np.isinf(trunc[5]) and np.isnan(y[5])
    # finite values are untouched by the guard
    rng = np.random.default_rng(3)
    f = (rng.standard_normal(10000) * 10.0 ** rng.uniform(-30, 30, 10000)).astype(np.float32)
    assert np.array_equal(to_24bit(f).view(np.uint32), to_24bit(f, guard=False).view(np.uint32))
