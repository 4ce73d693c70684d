"""Pins of the RoPE + FP8 quantisation + cache-write oracle
(oracle/kv_write_ref.py), CPU only.

The pages show only the calls, so the pins are what the mathematics and the
formats fix: rotations worked by hand for both pairings, the rotation's norm
and relative-position properties on a RoFormer frequency table, e4m3
rounding against the format's value table, its ties and saturation, and
against torch's float8 conversion; the cache write round-trips through the
decode oracle's gather.  ``test_planted_mistake_is_caught`` plants plausible
mistakes (swapped sin sign, pairing swapped, truncation, ties away from zero,
the same four in bf16 rounding, NaN overflowing to infinity, slot split by the
wrong page size) and checks that a pin rejects each.
"""

import inspect
import math
import types

import numpy as np
import pytest

from oracle import kv_write_ref as K
from oracle import mla_ref as O


def roformer_cache(max_pos, base=10000.0, dim=64):
    """cos/sin table of RoFormer: theta_i = base^(-2i/dim), angle = p * theta_i."""
    inv = base ** (-np.arange(0, dim, 2, dtype=np.float64) / dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def pin_hand_rotation(mod):
    """Pair 0 rotated by 90 degrees, pair 1 by 180, the rest untouched
    (cos 1, sin 0), for both pairings."""
    cos = np.ones(32)
    sin = np.zeros(32)
    cos[0], sin[0] = 0.0, 1.0
    cos[1], sin[1] = -1.0, 0.0
    x = np.arange(1, 65, dtype=np.float64)
    neox = mod.rotate(x, cos, sin, True)
    want_neox = x.copy()
    want_neox[0], want_neox[32] = -x[32], x[0]      # (a, b) -> (-b, a)
    want_neox[1], want_neox[33] = -x[1], -x[33]     # (a, b) -> (-a, -b)
    inter = mod.rotate(x, cos, sin, False)
    want_inter = x.copy()
    want_inter[0], want_inter[1] = -x[1], x[0]
    want_inter[2], want_inter[3] = -x[2], -x[3]
    return np.allclose(neox, want_neox, atol=1e-15) and np.allclose(inter, want_inter, atol=1e-15)


def pin_rotation_properties(mod):
    """Norm kept; <R_m q, R_n k> depends on m - n only; position 0 is the
    identity -- for both pairings."""
    rng = np.random.default_rng(0)
    cs = roformer_cache(64)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    ok = True
    for neox in (True, False):
        r = lambda v, p: mod.rotate(v, cs[p, :32], cs[p, 32:], neox)  # noqa: E731
        ok &= abs(np.linalg.norm(r(q, 17)) - np.linalg.norm(q)) < 1e-12
        ok &= np.allclose(r(q, 0), q, atol=0)
        ok &= abs(r(q, 40) @ r(k, 33) - r(q, 7) @ r(k, 0)) < 1e-10
        ok &= abs(r(q, 40) @ r(k, 33) - q @ k) > 1e-6  # and it does rotate
    return bool(ok)


def pin_pairings_differ_by_permutation(mod):
    """Interleaved rotation = half rotation conjugated by the even/odd
    permutation."""
    rng = np.random.default_rng(1)
    cs = roformer_cache(8)
    x = rng.standard_normal(64)
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])  # interleaved -> halves
    a = mod.rotate(x, cs[5, :32], cs[5, 32:], False)
    b = mod.rotate(x[perm], cs[5, :32], cs[5, 32:], True)
    return np.allclose(a[perm], b, atol=1e-15)


def pin_e4m3_rounding(mod):
    """Every code's value maps to itself; midpoints go to the even code;
    just off a midpoint goes to the nearer; saturation at 448; sign kept."""
    vals = O.decode_e4m3fn(np.arange(0x7F, dtype=np.uint8))
    if not np.array_equal(mod.quantize_e4m3(vals), np.arange(0x7F, dtype=np.uint8)):
        return False
    mids = (vals[:-1] + vals[1:]) / 2
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    if not np.array_equal(mod.quantize_e4m3(mids), want):
        return False
    eps = 1e-9
    if not np.array_equal(mod.quantize_e4m3(mids * (1 + eps)), (lo + 1).astype(np.uint8)):
        return False
    if not np.array_equal(mod.quantize_e4m3(mids * (1 - eps)), lo.astype(np.uint8)):
        return False
    big = mod.quantize_e4m3(np.array([448.0, 449.0, 1e6, -1e6, -0.0, -1e-9]))
    return np.array_equal(big, [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x80])


def pin_against_torch(mod):
    """Values in range: the same codes as torch's float8_e4m3fn cast."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (0.01, 1.0, 30.0)])
    x = x[np.abs(x) < 440]
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # float32 first (torch's input); exact values here, as e4m3 midpoints are float32-exact
    return np.array_equal(mod.quantize_e4m3(x.astype(np.float32).astype(np.float64)), want)


def pin_cache_write_round_trip(mod):
    """Rows written at slots come back through the decode oracle's gather in
    token order; other rows are unchanged."""
    rng = np.random.default_rng(3)
    page = 32
    kv = rng.integers(0, 65535, size=(6, page, 576), dtype=np.uint16)
    bt = np.array([4, 1, 5], dtype=np.int64)
    slots = np.array([bt[j // page] * page + j % page for j in range(70)])
    rows = rng.integers(0, 65535, size=(70, 576), dtype=np.uint16)
    new = mod.kv_cache_write(kv, rows, slots, page)
    back = O.gather_rows(new, bt, 70, page)
    untouched = np.ones((6, page), dtype=bool)
    untouched[slots // page, slots % page] = False
    return np.array_equal(back, rows) and np.array_equal(new[untouched], kv[untouched])


def pin_f32_tracks_f64(mod):
    """The float32 rotation (the one codes are rounded from) follows the
    float64 one within float32 rounding, for both pairings."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 64)).astype(np.float32).astype(np.float64)
    cs = roformer_cache(40).astype(np.float32)
    ok = True
    for neox in (True, False):
        a = mod.rotate(x, cs[[5, 17, 39], :32].astype(np.float64), cs[[5, 17, 39], 32:].astype(np.float64), neox)
        b = mod.rotate_f32(x, cs[[5, 17, 39], :32], cs[[5, 17, 39], 32:], neox)
        ok &= bool(np.all(np.abs(a - b) <= 4 * np.finfo(np.float32).eps * (np.abs(x).max() + 1)))
    return ok


def _bf16_of_float32_bits(u32):
    return np.asarray(u32, dtype=np.uint32).view(np.float32)


def pin_bf16_rounding(mod):
    """round_bf16 at the places that fix round-to-nearest-even: every exact
    midpoint goes to the even neighbour (so odd kept halves round up, even
    ones down), one unit above / below a midpoint goes to the nearer value,
    signed zeros and infinities are kept, the largest finite values overflow
    to infinity exactly at the midpoint past the bf16 maximum, and NaN stays
    NaN."""
    rng = np.random.default_rng(11)
    hi = rng.integers(0, 0x7F80, size=4000).astype(np.uint32)  # finite kept halves, both parities
    hi = np.concatenate([hi, hi | 0x8000, np.array([0, 1, 0x7F7E, 0x7F7F, 0x8000, 0x8001, 0xFF7F], np.uint32)])
    even_up = hi + (hi & 1)  # ties to even: odd kept halves carry
    ok = np.array_equal(mod.round_bf16(_bf16_of_float32_bits((hi << 16) | 0x8000)), even_up.astype(np.uint16))
    ok &= np.array_equal(mod.round_bf16(_bf16_of_float32_bits((hi << 16) | 0x8001)), (hi + 1).astype(np.uint16))
    ok &= np.array_equal(mod.round_bf16(_bf16_of_float32_bits((hi << 16) | 0x7FFF)), hi.astype(np.uint16))
    ok &= np.array_equal(mod.round_bf16(_bf16_of_float32_bits(hi << 16)), hi.astype(np.uint16))
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x00008000, 0x00018000, 0x7F7F7FFF, 0x7F7F8000,
                        0xFF7F8000, 0x7F800000, 0xFF800000], dtype=np.uint32)
    want = np.array([0x0000, 0x8000, 0x0000, 0x0000, 0x0002, 0x7F7F, 0x7F80, 0xFF80, 0x7F80, 0xFF80], np.uint16)
    ok &= np.array_equal(mod.round_bf16(_bf16_of_float32_bits(special)), want)
    nan = mod.round_bf16(_bf16_of_float32_bits(np.array([0x7F800001, 0xFF800001, 0x7FC00000, 0x7FFFFFFF],
                                                         dtype=np.uint32)))
    ok &= bool(np.all((nan & 0x7F80) == 0x7F80) and np.all((nan & 0x007F) != 0))  # NaN, not infinity
    return bool(ok)


def pin_bf16_against_torch(mod):
    """Finite float32 values over the whole range, subnormals included: the
    same bf16 bits as torch's own float32 -> bfloat16 cast."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    x = rng.standard_normal(60000) * 10.0 ** rng.uniform(-44, 38.5, 60000)
    x = x[np.abs(x) < 3.0e38].astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return np.array_equal(mod.round_bf16(x), want)


def pin_rope_bf16_quarter_turns(mod):
    """rope_bf16 where the rotation is exact (quarter and half turns: a swap
    and sign changes of bf16 values), for both pairings: the output bits are
    the input's, moved and negated as worked out by hand."""
    rng = np.random.default_rng(13)
    x_bits = W_bits(rng.standard_normal(64).astype(np.float32))
    x = O.decode_bf16(x_bits)
    cs = np.zeros((3, 64), dtype=np.float32)
    cs[:, :32] = 1.0                       # position 0: identity
    cs[1, 0], cs[1, 32] = 0.0, 1.0          # position 1: pair 0 turned by 90 degrees
    cs[2, 3], cs[2, 35] = 0.0, -1.0         # position 2: pair 3 turned by -90 degrees
    cs[2, 5] = -1.0                         # ... and pair 5 by 180 degrees
    ok = True
    for neox in (True, False):
        got = mod.rope_bf16(np.stack([x_bits] * 3)[:, None, :], np.array([0, 1, 2]), cs, neox)[:, 0]
        ia = lambda i: i if neox else 2 * i  # noqa: E731  first element of pair i
        ib = lambda i: i + 32 if neox else 2 * i + 1  # noqa: E731
        want = np.stack([x.copy() for _ in range(3)])
        want[1, ia(0)], want[1, ib(0)] = -x[ib(0)], x[ia(0)]
        want[2, ia(3)], want[2, ib(3)] = x[ib(3)], -x[ia(3)]
        want[2, ia(5)], want[2, ib(5)] = -x[ia(5)], -x[ib(5)]
        ok &= np.array_equal(O.decode_bf16(got), want) and np.array_equal(got[0], x_bits)
    return bool(ok)


def pin_rope_bf16_against_torch(mod):
    """rope_bf16 on a RoFormer table against the same rotation done with
    torch float32 tensor ops (each product and sum its own rounded op) and
    torch's bf16 cast, for both pairings."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    x_bits = W_bits(rng.standard_normal((5, 2, 64)).astype(np.float32))
    cs = roformer_cache(300).astype(np.float32)
    pos = np.array([0, 3, 77, 150, 299])
    ok = True
    for neox in (True, False):
        xt = torch.from_numpy(O.decode_bf16(x_bits).astype(np.float32))
        c = torch.from_numpy(cs[pos, :32])[:, None, :]
        s_ = torch.from_numpy(cs[pos, 32:])[:, None, :]
        if neox:
            a, b = xt[..., :32], xt[..., 32:]
            r = torch.cat([torch.sub(torch.mul(a, c), torch.mul(b, s_)), torch.add(torch.mul(b, c), torch.mul(a, s_))],
                          dim=-1)
        else:
            a, b = xt[..., 0::2], xt[..., 1::2]
            r = torch.stack([torch.sub(torch.mul(a, c), torch.mul(b, s_)), torch.add(torch.mul(b, c), torch.mul(a, s_))],
                            dim=-1).reshape(xt.shape)
        want = r.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ok &= np.array_equal(mod.rope_bf16(x_bits, pos, cs, neox), want)
    return bool(ok)


def W_bits(x32):
    """float32 -> bf16 bits by torch's cast (input generation for the pins)."""
    torch = pytest.importorskip("torch")
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def all_pins(mod):
    return [pin_hand_rotation(mod), pin_rotation_properties(mod), pin_pairings_differ_by_permutation(mod),
            pin_e4m3_rounding(mod), pin_against_torch(mod), pin_cache_write_round_trip(mod),
            pin_f32_tracks_f64(mod), pin_bf16_rounding(mod), pin_bf16_against_torch(mod),
            pin_rope_bf16_quarter_turns(mod), pin_rope_bf16_against_torch(mod)]


def test_hand_rotation():
    assert pin_hand_rotation(K)


def test_rotation_properties():
    assert pin_rotation_properties(K)


def test_pairings_related_by_permutation():
    assert pin_pairings_differ_by_permutation(K)


def test_e4m3_rounding():
    assert pin_e4m3_rounding(K)


def test_e4m3_against_torch():
    assert pin_against_torch(K)


def test_cache_write_round_trip():
    assert pin_cache_write_round_trip(K)


def test_bf16_rounding():
    assert pin_bf16_rounding(K)


def test_bf16_against_torch():
    assert pin_bf16_against_torch(K)


def test_rope_bf16_quarter_turns():
    assert pin_rope_bf16_quarter_turns(K)


def test_rope_bf16_against_torch():
    assert pin_rope_bf16_against_torch(K)


def test_rope_quantize_shapes_and_values():
    """The fused oracle is the composition of its parts."""
    rng = np.random.default_rng(4)
    from paged_mla_decode_08_gb300 import workloads as W
    t, h = 3, 2
    qn = W.f32_to_bf16_bits(rng.standard_normal((t, h, 512), dtype=np.float32))
    qr = W.f32_to_bf16_bits(rng.standard_normal((t, h, 64), dtype=np.float32))
    kn = W.f32_to_bf16_bits(rng.standard_normal((t, 512), dtype=np.float32))
    kr = W.f32_to_bf16_bits(rng.standard_normal((t, 64), dtype=np.float32))
    cs = roformer_cache(100)
    pos = np.array([0, 7, 99])
    qc, kc, qv, kv = K.rope_quantize_fp8(qn, qr, kn, kr, pos, cs, False)
    assert qc.shape == (t, h, 576) and kc.shape == (t, 576)
    assert np.array_equal(qv[0, :, 512:], O.decode_bf16(qr[0]))          # position 0: identity
    assert np.array_equal(kc[:, :512], K.quantize_e4m3(O.decode_bf16(kn)))
    r = K.rotate_f32(O.decode_bf16(kr[2]), cs[99, :32], cs[99, 32:], False)
    assert np.array_equal(kc[2, 512:], K.quantize_e4m3(r.astype(np.float64)))
    assert math.isclose(np.linalg.norm(kv[1, 512:]), np.linalg.norm(O.decode_bf16(kr[1])), rel_tol=1e-6)


def test_float32_rotation_is_the_rotation():
    """rotate_f32 (the precision codes are decided in) stays within float32
    rounding of the float64 rotation, and is exact where no rounding occurs
    (cos, sin in {0, 1, -1} on bf16 inputs)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 64)).astype(np.float32).astype(np.float64)
    cs = roformer_cache(50).astype(np.float32)
    for neox in (True, False):
        a = K.rotate(x, cs[[3, 9, 27, 49], None, :32][:, 0].astype(np.float64),
                     cs[[3, 9, 27, 49], None, 32:][:, 0].astype(np.float64), neox)
        b = K.rotate_f32(x, cs[[3, 9, 27, 49], :32], cs[[3, 9, 27, 49], 32:], neox)
        assert np.all(np.abs(a - b) <= 4 * np.finfo(np.float32).eps * (np.abs(x).max() + 1))
        c = np.zeros(32, dtype=np.float32)
        c[:16] = 1
        s_ = np.zeros(32, dtype=np.float32)
        s_[16:] = -1
        assert np.array_equal(K.rotate_f32(x[0], c, s_, neox), K.rotate(x[0], c, s_, neox))


MUTATIONS = [
    ("sine sign swapped",
     "        out[..., :half] = a * cos - b * sin\n        out[..., half:] = b * cos + a * sin",
     "        out[..., :half] = a * cos + b * sin\n        out[..., half:] = b * cos - a * sin"),
    ("sine sign swapped in the float32 rotation only",
     "        out[..., 0::2] = (a * cos) - (b * sin)\n        out[..., 1::2] = (b * cos) + (a * sin)",
     "        out[..., 0::2] = (a * cos) + (b * sin)\n        out[..., 1::2] = (b * cos) - (a * sin)"),
    ("pairings swapped",
     "    if is_neox:\n        a, b = x[..., :half], x[..., half:]",
     "    if not is_neox:\n        a, b = x[..., :half], x[..., half:]"),
    ("interleaved pairs off by one",
     "        a, b = x[..., 0::2], x[..., 1::2]\n        out[..., 0::2]",
     "        a, b = x[..., 1::2], x[..., 0::2]\n        out[..., 0::2]"),
    ("truncation instead of rounding",
     "    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))",
     "    pick_hi = np.zeros(np.shape(d_hi), dtype=bool)"),
    ("ties away from zero",
     "((d_hi == d_lo) & (hi % 2 == 0))", "(d_hi == d_lo)"),
    ("sign dropped",
     "    return (code | (neg.astype(np.uint8) << 7)).astype(np.uint8)", "    return code"),
    ("bf16 ties away from zero",
     "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "    u = (u + 0x8000) >> 16"),
    ("bf16 ties to odd",
     "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "    u = (u + 0x8000 - ((u >> 16) & 1)) >> 16"),
    ("bf16 truncation",
     "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "    u = u >> 16"),
    ("bf16 wrong shift",
     "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 15"),
    ("bf16 parity bit taken from the dropped half",
     "    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "    u = (u + 0x7FFF + ((u >> 15) & 1)) >> 16"),
    ("bf16 NaN carried into infinity",
     "    u = np.where(nan, ", "    u = np.where(False, "),
    ("rope bf16 cos and sin columns swapped",
     "    cos = cs[(slice(None),) + extra + (slice(0, ROPE_DIM // 2),)]\n    sin = cs[(slice(None),) + extra + (slice(ROPE_DIM // 2, ROPE_DIM),)]",
     "    sin = cs[(slice(None),) + extra + (slice(0, ROPE_DIM // 2),)]\n    cos = cs[(slice(None),) + extra + (slice(ROPE_DIM // 2, ROPE_DIM),)]"),
    ("slot split by the wrong page size",
     "        kv[slot // page_size, slot % page_size] = rows[t]", "        kv[slot // 64, slot % 64] = rows[t]"),
]


def mutated(old, new):
    src = inspect.getsource(K).replace("from .mla_ref import", "from oracle.mla_ref import")
    assert src.count(old) >= 1, old  # a systematic mistake: every occurrence
    mod = types.ModuleType("kv_write_mutant")
    exec(compile(src.replace(old, new), "kv_write_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    try:
        results = all_pins(mutated(old, new))
    except (IndexError, ValueError):
        return
    assert not all(results), f"no pin rejects: {name}"


def test_unmutated_passes_all_pins():
    assert all(all_pins(K))
