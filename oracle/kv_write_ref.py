"""CPU oracle for the step that feeds the decode: rotary embedding of the
rope parts, FP8 quantisation, and the write of each new token's latent row
into the paged cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this file: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  It shares no code, table or helper with the CUDA path.

Source: sglang ``trtllm_mla_backend.py``, ``forward_decode`` (FP8 cache):
``mla_quantize_and_rope_for_fp8(q_nope, q_rope, k_nope, k_rope, positions,
cos_sin_cache, is_neox, kv_lora_rank, qk_rope_head_dim)`` returns the merged
FP8 query and the FP8 key parts, then ``set_mla_kv_buffer(layer,
out_cache_loc, k, k_rope)`` stores them; tokenspeed ``trtllm_mla.py``,
``forward_decode``: ``set_mla_kv_buffer(layer, out_cache_loc, k[..., :512],
k[..., 512:])``.  The pages show the calls, not their arithmetic; readings
taken (each also in the design notes):

* ``cos_sin_cache[p]`` holds the 32 cosines then the 32 sines of position
  p (one per rotated pair);
* ``is_neox`` pairs element i with element i + 32 (halves); otherwise
  element 2i with 2i + 1 (interleaved); either pair (a, b) becomes
  (a cos - b sin, b cos + a sin) -- the rotation of RoFormer (Su et al.,
  "RoFormer: Enhanced Transformer with Rotary Position Embedding", eq. 13-15);
* quantisation to float8 e4m3fn rounds to nearest (ties to even) and
  saturates at +-448, with no scale (the pages pass none);
* cache slot s is row s % page_size of page s // page_size, the layout the
  decode reads (``k_cache.view(-1, page_size, 576)``).

The rotated values that are rounded to e4m3 or bf16 are computed in float32
with each product and each sum rounded on its own (``rotate_f32``): a
quantised code is an integer decided by floating point, so both sides decide
it in the same precision (the kernel's; the pages fix none).  ``rotate`` is
the same rotation in float64, which the pins check against the mathematics
and ``rotate_f32`` against within float32 rounding.

parity pinned: tests/test_kv_write_oracle.py (hand-computed rotations, norm
and relative-position properties of the rotation built from a RoFormer
frequency table, both pairings, e4m3 rounding against the format table and
torch, bf16 rounding against exact midpoints, signed zeros, the overflow
boundary and torch's own cast, the bf16 rope output against exact quarter
and half turns and against a float32 rotation done in torch, slot round trip
through the decode's gather).
"""

from __future__ import annotations

import numpy as np

from .mla_ref import decode_bf16, decode_e4m3fn

KV_LORA_RANK = 512
ROPE_DIM = 64


def rotate(x: np.ndarray, cos: np.ndarray, sin: np.ndarray, is_neox: bool) -> np.ndarray:
    """Rotary embedding of the last axis (64 wide) of float64 ``x`` with
    per-pair ``cos``/``sin`` (32 wide, broadcast over leading axes)."""
    half = ROPE_DIM // 2
    out = np.empty_like(x)
    if is_neox:
        a, b = x[..., :half], x[..., half:]
        out[..., :half] = a * cos - b * sin
        out[..., half:] = b * cos + a * sin
    else:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * cos - b * sin
        out[..., 1::2] = b * cos + a * sin
    return out


def rotate_f32(x, cos, sin, is_neox: bool) -> np.ndarray:
    """``rotate`` in float32: a*cos, b*sin, b*cos, a*sin each rounded to
    float32, then the difference / sum rounded (no fused multiply-add).
    Returns float32."""
    x = np.asarray(x, dtype=np.float32)
    cos = np.asarray(cos, dtype=np.float32)
    sin = np.asarray(sin, dtype=np.float32)
    half = ROPE_DIM // 2
    out = np.empty_like(x)
    if is_neox:
        a, b = x[..., :half], x[..., half:]
        out[..., :half] = (a * cos) - (b * sin)
        out[..., half:] = (b * cos) + (a * sin)
    else:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = (a * cos) - (b * sin)
        out[..., 1::2] = (b * cos) + (a * sin)
    return out


def _e4m3_values() -> np.ndarray:
    """The 126 finite non-negative e4m3fn values, ascending (from the
    format: 4-bit exponent, bias 7, 3-bit mantissa, no infinities, 0x7F NaN)."""
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00..0x7E
    return decode_e4m3fn(codes)


def quantize_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> e4m3fn codes: the nearest finite value (ties to the even
    code), magnitudes past 448 saturated to 448, the sign kept."""
    vals = _e4m3_values()  # code i has value vals[i], increasing
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(vals, a, side="left").clip(0, len(vals) - 1)  # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == vals[hi], hi, code).astype(np.uint8)
    neg = np.signbit(x)  # the sign survives rounding to zero (-0 is 0x80)
    return (code | (neg.astype(np.uint8) << 7)).astype(np.uint8)


def rope_quantize_fp8(q_nope_bits, q_rope_bits, k_nope_bits, k_rope_bits, positions, cos_sin_cache,
                      is_neox: bool):
    """Returns (q codes uint8 [T, H, 576] = [q_nope | rope(q_rope)],
    k codes uint8 [T, 576] = [k_nope | rope(k_rope)]) and the float64
    pre-rounding values (q_val, k_val) the codes were rounded from."""
    t = q_nope_bits.shape[0]
    cs = np.asarray(cos_sin_cache, dtype=np.float32)[np.asarray(positions, dtype=np.int64)]
    cos, sin = cs[:, : ROPE_DIM // 2], cs[:, ROPE_DIM // 2:]
    q_rot = rotate_f32(decode_bf16(q_rope_bits), cos[:, None, :], sin[:, None, :], is_neox)
    k_rot = rotate_f32(decode_bf16(k_rope_bits).reshape(t, ROPE_DIM), cos, sin, is_neox)
    q_val = np.concatenate([decode_bf16(q_nope_bits), q_rot.astype(np.float64)], axis=-1)
    k_val = np.concatenate([decode_bf16(k_nope_bits).reshape(t, KV_LORA_RANK), k_rot.astype(np.float64)], axis=-1)
    return quantize_e4m3(q_val), quantize_e4m3(k_val), q_val, k_val


def round_bf16(x) -> np.ndarray:
    """float32 values -> bf16 bit patterns, round to nearest, ties to even
    (the IEEE 754 default, which bf16 -- float32's top 16 bits -- inherits).

    On the bit pattern u: the kept half is u >> 16; the dropped half is
    compared with 0x8000 by adding 0x7FFF plus the kept half's lowest bit, so
    a carry happens above the midpoint, and at the midpoint only when the kept
    half is odd.  A carry out of the mantissa moves the exponent up, which is
    also how the largest finite values overflow to infinity.  Infinities are
    unchanged by this; NaN is handled apart (a quiet NaN of the same sign), as
    the carry could turn a NaN into an infinity."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    u = np.where(nan, ((np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16) | 0x0040), u)
    return u.astype(np.uint16)


def rope_bf16(rope_bits, positions, cos_sin_cache, is_neox: bool) -> np.ndarray:
    """bf16 bits of rope(x) for rows [T, ..., 64] of bf16 ``rope_bits``
    (rotation in float32 as above, then nearest-even to bf16)."""
    cs = np.asarray(cos_sin_cache, dtype=np.float32)[np.asarray(positions, dtype=np.int64)]
    x = decode_bf16(rope_bits)
    extra = (None,) * (x.ndim - 2)
    cos = cs[(slice(None),) + extra + (slice(0, ROPE_DIM // 2),)]
    sin = cs[(slice(None),) + extra + (slice(ROPE_DIM // 2, ROPE_DIM),)]
    return round_bf16(rotate_f32(x, cos, sin, is_neox))


def kv_cache_write(kv_bits: np.ndarray, rows: np.ndarray, out_cache_loc, page_size: int) -> np.ndarray:
    """A copy of the cache ``kv_bits [P, page, 576]`` with token t's stored
    row ``rows[t]`` (576 wide, cache element type) at slot out_cache_loc[t]."""
    kv = np.array(kv_bits, copy=True)
    for t, slot in enumerate(np.asarray(out_cache_loc, dtype=np.int64)):
        kv[slot // page_size, slot % page_size] = rows[t]
    return kv
