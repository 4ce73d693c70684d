"""The precision reading for the CTA pair's score exchange, checked on the CPU.

The decode splits every score between two CTAs: CTA r holds the partial dot
product over latent columns [256r, 256r+256) and rope columns [512+32r,
512+32r+32).  Each sends its partial to the other as a 24-bit code, the
float32 value multiplied by 1 + 85 * 2^-23 and its low 8 bits dropped
(relative error below (4/3) * 2^-16).  The claim: the log-sum-exp of a row then
moves by at most that relative error times the largest partial logit of the
row (the LSE is 1-Lipschitz in the largest score error), which keeps it
inside the 2e-3 tolerance for partial logits up to about 100 in natural-log
units.

These tests restate the rounding in NumPy, apply it to one partial of each
score, and compare the row LSE with the exact float64 one, from ordinary to
very sharp attention.  They exercise the arithmetic of the reading, not the
CUDA path (the GPU parity tests cover that).
"""

import numpy as np
import pytest

SCALE = 1.0 / np.sqrt(192.0)
LATENT, ROPE = 512, 64


CODE_ROUND = np.float32(1.0 + 85.0 * 2.0 ** -23)  # exact in float32


def to_24bit(x32, rounding="mul"):
    """float32 -> float32 keeping the top 24 bits (the exchange code,
    restated).  ``rounding="mul"``: the code's rounding, one float32
    multiply by 1 + 85 * 2^-23 and a truncation of the low 8 bits.
    ``rounding="add"``: the integer round-to-nearest add (the code this
    replaced, kept to show what it does to NaN)."""
    x32 = np.asarray(x32, dtype=np.float32)
    if rounding == "mul":
        with np.errstate(over="ignore", invalid="ignore"):
            bits = (x32 * CODE_ROUND).view(np.uint32).astype(np.uint64)
        return ((bits >> 8) << 8).astype(np.uint32).view(np.float32)
    bits = x32.view(np.uint32).astype(np.uint64)
    code = ((bits + 0x80) & 0xFFFFFFFF) >> 8
    return ((code << 8) & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def partial_scores(q, kv):
    """Raw partial dot products of the two CTAs, float64: [rows, keys] each."""
    c0 = np.r_[0:256, LATENT:LATENT + 32]
    c1 = np.r_[256:512, LATENT + 32:LATENT + ROPE]
    return q[:, c0] @ kv[:, c0].T, q[:, c1] @ kv[:, c1].T


def lse(s):
    m = s.max(axis=1, keepdims=True)
    return (m[:, 0] + np.log(np.exp(s - m).sum(axis=1)))


BOUND = (4.0 / 3.0) * 2.0 ** -16


def test_rounding_error_bound():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * 10.0 ** rng.uniform(-3, 4, 200_000)).astype(np.float32)
    y = to_24bit(x).astype(np.float64)
    rel = np.abs(y - x) / np.abs(x.astype(np.float64))
    assert rel.max() <= BOUND
    assert rel.max() > 2.0 ** -16  # the bound is the multiply's, wider than round-to-nearest
    # the error averages out: as many codes round up as down
    assert abs(np.mean(np.sign(y - x))) < 0.05
    # worst case by construction: mantissa 1.0 plus just under 0.668 of a code unit
    unit = 2.0 ** -15
    worst = np.float32(1.0 + 0.6679 * unit)
    assert abs(float(to_24bit(worst)) - float(worst)) <= 0.668 * unit


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
    # float32 rounding of each partial (2^-24) plus the exchange code
    bound = SCALE * (np.abs(s1).max(axis=1) * (BOUND + 2.0 ** -24) + np.abs(s0).max(axis=1) * 2.0 ** -24)
    assert np.all(np.abs(got - exact) <= bound * (1 + 1e-6) + 1e-12)
    peak = SCALE * np.abs(s1).max()
    if peak <= 100.0:
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
    assert np.abs(code24 - exact).max() <= BOUND * SCALE * np.abs(s1).max() * 1.01
    assert np.abs(code24 - exact).max() < 2e-3


def test_non_finite_scores_cross_unchanged():
    """An infinite partial stays that infinity and every NaN stays NaN, so
    both CTAs of the pair see the same non-finite score.  The integer rounding
    add would not: the canonical NaN 0x7FFFFFFF carries into the sign bit and
    arrives as -0.0, and a negative NaN near 0xFFFFFFFF wraps to +0."""
    bits = np.array([0x7F800000, 0xFF800000, 0x7FFFFFFF, 0xFFFFFFFF, 0x7FC00000, 0x7F800001, 0xFF800080,
                     0xFFC00000], dtype=np.uint32)
    x = bits.view(np.float32)
    y = to_24bit(x)
    assert y[0] == np.inf and y[1] == -np.inf
    assert np.all(np.isnan(y[2:]))
    bad = to_24bit(x, rounding="add")
    assert bad[2] == 0.0 and np.signbit(bad[2]) and bad[3] == 0.0  # what the multiply avoids
    # the largest finite values round up to infinity, as rounding up must
    assert to_24bit(np.array([0x7F7FFFFF], dtype=np.uint32).view(np.float32))[0] == np.inf
    # zeros and subnormals stay finite and keep their sign
    tiny = np.array([0x00000000, 0x80000000, 0x00000001, 0x807FFFFF], dtype=np.uint32).view(np.float32)
    t = to_24bit(tiny)
    assert np.all(np.isfinite(t)) and np.array_equal(np.signbit(t), np.signbit(tiny))
