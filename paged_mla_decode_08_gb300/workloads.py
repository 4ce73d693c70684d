"""Seeded synthetic inputs for paged MLA decode.

This module only *makes data*: request lengths, shuffled block tables and the
stored bit patterns of the query and of the paged latent KV cache.  It holds
none of the decode arithmetic, so both the float64 oracle and the CUDA path
can consume the very same inputs without sharing any code of the method.

Shapes follow the serving pages (sglang ``trtllm_mla_backend.py``,
``forward_decode``; tokenspeed ``flashmla.py``, ``forward_decode``):

* query is split into the absorbed no-PE part ``q_nope [T, H, 512]`` and the
  rotary part ``q_pe [T, H, 64]`` with ``T = batch * q_len`` (request-major,
  then query position);
* the cache is ``kv_pages [P, page_size, 576]``: 512 latent columns (c_kv)
  followed by 64 rotary-key columns (k_pe); one latent head shared by all
  query heads;
* ``block_table [batch, bt_stride]`` int32 holds physical page ids, padded
  with -1 past ``ceil(seq_len / page_size)`` entries (those entries are never
  read);
* ``seq_lens [batch]`` int32 counts KV tokens *including* the q_len new ones.

Values are drawn with ``numpy.random.default_rng(seed)`` and rounded to the
stored type with round-to-nearest-even (bf16) or round-to-nearest-even with
saturation at +-448 (float8 e4m3fn).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

KV_LORA_RANK = 512
ROPE_DIM = 64
KV_DIM = KV_LORA_RANK + ROPE_DIM
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

# The five synthetic workloads.  Sizes are the ones the decode benchmark uses.
CONFIGS = {
    "tiny": dict(
        batch=2, q_len=1, num_heads=16, page_size=64, kv_dtype="bf16",
        seq_lens=[64, 100], pool_pages=4, k_scale=1.0,
        desc="B=2, q_len=1, H=16, seq_lens {64,100}, page 64, 4-page pool",
    ),
    "dsv3": dict(
        batch=64, q_len=1, num_heads=128, page_size=64, kv_dtype="bf16",
        seq_len_uniform=(1024, 4096), pool_pages=16384, k_scale=1.0,
        desc="DeepSeek-V3-shaped: B=64, q_len=1, H=128, L~U[1024,4096], page 64, 16384-page pool",
    ),
    "long_skewed": dict(
        batch=8, q_len=1, num_heads=128, page_size=32, kv_dtype="bf16",
        seq_lens=[131072, 65536, 32768, 16384, 4096, 1024, 256, 17],
        pool_pages=16384, k_scale=1.0,
        desc="B=8, q_len=1, H=128, L={128k,64k,32k,16k,4k,1k,256,17}, page 32",
    ),
    "spec_q4": dict(
        batch=128, q_len=4, num_heads=16, page_size=64, kv_dtype="bf16",
        seq_len_uniform=(2048, 8192), pool_pages=16384, k_scale=1.0,
        desc="B=128, q_len=4 causal, H=16, L~U[2048,8192], page 64",
    ),
    "fp8_kv": dict(
        batch=256, q_len=1, num_heads=128, page_size=64, kv_dtype="e4m3",
        seq_len_lognormal=(7.5, 1.0, 0, 16384), zero_frac=0.05,
        pool_pages=16384, k_scale=0.5,
        desc="B=256, q_len=1, H=128, e4m3 KV (k_scale 0.5), L~lognormal(7.5,1) in [0,16384], 5% empty, page 64",
    ),
}


# Ragged query lengths: draft extend after speculative decoding, where each
# request keeps a different number of accepted draft tokens (1..4 here, the
# usual MTP draft width), 16 heads per GPU as in the q_len=4 verify case.
RAGGED_CONFIGS = {
    "draft_extend": dict(
        batch=128, q_len_range=(1, 4), num_heads=16, page_size=64, kv_dtype="bf16",
        seq_len_uniform=(2048, 8192), pool_pages=16384, k_scale=1.0,
        desc="B=128, ragged q_len~U{1..4} causal (cu_seqlens_q), H=16, L~U[2048,8192], page 64",
    ),
}


@dataclass
class Workload:
    """One batch of decode inputs, as stored bit patterns on the host."""

    name: str
    batch: int
    q_len: int
    num_heads: int
    page_size: int
    kv_dtype: str  # "bf16" or "e4m3"
    scale: float
    k_scale: float
    seq_lens: np.ndarray  # int32 [B]
    block_table: np.ndarray  # int32 [B, bt_stride]
    q_nope_bits: np.ndarray  # uint16 [T, H, 512] (bf16 bits)
    q_pe_bits: np.ndarray  # uint16 [T, H, 64] (bf16 bits)
    kv_bits: np.ndarray  # uint16 (bf16) or uint8 (e4m3) [P, page, 576]
    meta: dict = field(default_factory=dict)
    # ragged query lengths (draft extend): tokens of request b are rows
    # cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1; q_len is then their maximum
    cu_seqlens_q: np.ndarray | None = None  # int32 [B + 1]

    @property
    def num_tokens(self) -> int:
        if self.cu_seqlens_q is not None:
            return int(self.cu_seqlens_q[-1])
        return self.batch * self.q_len

    def q_lens(self) -> np.ndarray:
        """Query tokens of each request."""
        if self.cu_seqlens_q is not None:
            return np.diff(self.cu_seqlens_q).astype(np.int32)
        return np.full(self.batch, self.q_len, dtype=np.int32)

    @property
    def num_pages(self) -> int:
        return int(self.kv_bits.shape[0])

    @property
    def kv_elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1


# ---------------------------------------------------------------- rounding


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def f32_to_e4m3fn_bits(x: np.ndarray) -> np.ndarray:
    """Round finite values to float8 e4m3fn (nearest, ties to even, saturating
    at +-448); return the byte patterns.

    e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (step 2^-9); the all-ones pattern is NaN, so the
    largest finite magnitude is 448.
    """
    a = np.abs(np.asarray(x, dtype=np.float64))
    neg = np.signbit(np.asarray(x, dtype=np.float64))
    a = np.minimum(a, 448.0)
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))  # a = m * 2^ex, m in [0.5,1)
    e = ex.astype(np.int64) - 1  # floor(log2(a)) for normals, -6 below
    step = np.ldexp(1.0, (e - 3).astype(np.int32))
    q = np.rint(a / step) * step  # ties to even
    q = np.minimum(q, 448.0)
    bits = np.zeros(q.shape, dtype=np.int64)
    sub = q < 2.0 ** -6
    bits[sub] = np.rint(q[sub] / 2.0 ** -9).astype(np.int64)
    nrm = ~sub
    _, qex = np.frexp(q[nrm])
    qe = qex.astype(np.int64) - 1
    mant = np.rint((q[nrm] / np.ldexp(1.0, qe.astype(np.int32)) - 1.0) * 8.0).astype(np.int64)
    bits[nrm] = ((qe + 7) << 3) | mant
    bits = bits | (neg.astype(np.int64) << 7)
    return bits.astype(np.uint8)


BF16_NAN_BITS = np.uint16(0x7FC0)
E4M3_NAN_BITS = np.uint8(0x7F)


# ---------------------------------------------------------------- lengths


def draw_seq_lens(cfg: dict, rng: np.random.Generator) -> np.ndarray:
    b = cfg["batch"]
    if "seq_lens" in cfg:
        lens = np.asarray(cfg["seq_lens"], dtype=np.int64)
        assert lens.shape == (b,)
    elif "seq_len_uniform" in cfg:
        lo, hi = cfg["seq_len_uniform"]
        lens = rng.integers(lo, hi + 1, size=b, dtype=np.int64)
    elif "seq_len_lognormal" in cfg:
        mu, sigma, lo, hi = cfg["seq_len_lognormal"]
        lens = np.rint(rng.lognormal(mu, sigma, size=b)).astype(np.int64)
        lens = np.clip(lens, lo, hi)
        nz = int(round(cfg.get("zero_frac", 0.0) * b))
        if nz:
            lens[rng.choice(b, size=nz, replace=False)] = 0
    else:
        raise ValueError("config has no sequence-length rule")
    return lens.astype(np.int32)


# ---------------------------------------------------------------- builder


def build_workload(
    name: str,
    cfg: dict,
    seed: int = 0,
    fill: str = "zero",
    bt_pad_value: int = -1,
    bt_extra_cols: int = 0,
) -> Workload:
    """Draw one workload.

    fill: what goes into cache rows that no request may read (rows past
      seq_len in a request's last page and pages no request owns):
      "zero", "nan" (NaN bit patterns, to prove they are never used) or
      "random" (same distribution as live rows).
    bt_pad_value: value stored in block-table padding entries.
    bt_extra_cols: extra padding columns appended to every block-table row.
    """
    rng = np.random.default_rng(seed)
    b, q_len, h = cfg["batch"], cfg["q_len"], cfg["num_heads"]
    page = cfg["page_size"]
    kv_dtype = cfg["kv_dtype"]
    k_scale = float(cfg.get("k_scale", 1.0))
    seq_lens = draw_seq_lens(cfg, rng)
    pages_per_req = (seq_lens.astype(np.int64) + page - 1) // page
    need = int(pages_per_req.sum())
    pool = max(int(cfg.get("pool_pages", need)), need, 1)
    bt_stride = max(int(pages_per_req.max(initial=0)), 1) + bt_extra_cols
    perm = rng.permutation(pool).astype(np.int32)
    block_table = np.full((b, bt_stride), bt_pad_value, dtype=np.int32)
    cur = 0
    for r in range(b):
        n = int(pages_per_req[r])
        block_table[r, :n] = perm[cur : cur + n]
        cur += n

    t = b * q_len
    q_nope_bits = f32_to_bf16_bits(rng.standard_normal((t, h, KV_LORA_RANK), dtype=np.float32))
    q_pe_bits = f32_to_bf16_bits(rng.standard_normal((t, h, ROPE_DIM), dtype=np.float32))

    if kv_dtype == "bf16":
        kv = np.empty((pool, page, KV_DIM), dtype=np.uint16)
        dead = BF16_NAN_BITS
        encode = f32_to_bf16_bits
    elif kv_dtype == "e4m3":
        kv = np.empty((pool, page, KV_DIM), dtype=np.uint8)
        dead = E4M3_NAN_BITS
        encode = lambda v: f32_to_e4m3fn_bits(v / k_scale)  # noqa: E731
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype}")

    if fill == "random":
        kv[...] = encode(rng.standard_normal(kv.shape, dtype=np.float32))
    else:
        kv[...] = dead if fill == "nan" else 0
        # live rows, request-major, in block-table order
        for r in range(b):
            n_tok = int(seq_lens[r])
            for p in range(int(pages_per_req[r])):
                rows = min(page, n_tok - p * page)
                kv[block_table[r, p], :rows] = encode(
                    rng.standard_normal((rows, KV_DIM), dtype=np.float32)
                )
    return Workload(
        name=name, batch=b, q_len=q_len, num_heads=h, page_size=page,
        kv_dtype=kv_dtype, scale=DEFAULT_SCALE, k_scale=k_scale,
        seq_lens=seq_lens, block_table=block_table,
        q_nope_bits=q_nope_bits, q_pe_bits=q_pe_bits, kv_bits=kv,
        meta=dict(seed=seed, fill=fill, pool_pages=pool, desc=cfg.get("desc", "")),
    )


def make_workload(name: str, seed: int = 0, fill: str = "zero", **overrides) -> Workload:
    """Build one of the named workloads; ``overrides`` replace config keys."""
    cfg = dict(CONFIGS[name])
    bt_pad_value = overrides.pop("bt_pad_value", -1)
    bt_extra_cols = overrides.pop("bt_extra_cols", 0)
    if "seq_lens" in overrides:
        for k in ("seq_len_uniform", "seq_len_lognormal", "zero_frac"):
            cfg.pop(k, None)
    cfg.update(overrides)
    if "seq_lens" in cfg:
        cfg["batch"] = len(cfg["seq_lens"])
    return build_workload(name, cfg, seed=seed, fill=fill,
                          bt_pad_value=bt_pad_value, bt_extra_cols=bt_extra_cols)


def make_ragged_workload(name: str = "draft_extend", seed: int = 0, q_lens=None, fill: str = "zero",
                         **overrides) -> Workload:
    """A workload whose requests carry different numbers of query tokens
    (``q_lens``, drawn from the config's ``q_len_range`` when not given),
    packed back to back; ``overrides`` replace config keys as in
    ``make_workload``."""
    cfg = dict(RAGGED_CONFIGS[name])
    bt_pad_value = overrides.pop("bt_pad_value", -1)
    bt_extra_cols = overrides.pop("bt_extra_cols", 0)
    if "seq_lens" in overrides:
        cfg.pop("seq_len_uniform", None)
    cfg.update(overrides)
    if "seq_lens" in cfg:
        cfg["batch"] = len(cfg["seq_lens"])
    b = cfg["batch"]
    if q_lens is None:
        lo, hi = cfg["q_len_range"]
        q_lens = np.random.default_rng(seed + 7919).integers(lo, hi + 1, size=b)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    assert q_lens.shape == (b,) and q_lens.min(initial=0) >= 0
    cfg["q_len"] = max(int(q_lens.max(initial=1)), 1)
    w = build_workload(name, cfg, seed=seed, fill=fill, bt_pad_value=bt_pad_value, bt_extra_cols=bt_extra_cols)
    cu = np.zeros(b + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    t = int(cu[-1])
    w.q_nope_bits = w.q_nope_bits[:t]
    w.q_pe_bits = w.q_pe_bits[:t]
    w.cu_seqlens_q = cu
    return w


def workload_stats(w: Workload) -> dict:
    """Algorithmic work of one decode step over ``w`` (per-unit figures:
    per visible KV token of a request, 576 stored elements are read once and
    2*H*q_len*(576+512) flops are done; per query row, the 576-wide query is
    read and the 512-wide output plus one lse are written)."""
    lens = w.seq_lens.astype(np.int64)
    kv_tokens = int(lens.sum())
    # causal q_len>1: query i of a request sees L - q_len + 1 + i keys
    vis = 0
    ql = w.q_lens().astype(np.int64)
    for i in range(w.q_len):
        vis += int(np.where(i < ql, np.maximum(lens - ql + 1 + i, 0), 0).sum())
    h = w.num_heads
    t = w.num_tokens
    kv_bytes = kv_tokens * KV_DIM * w.kv_elem_bytes
    q_bytes = t * h * KV_DIM * 2
    out_bytes = t * h * KV_LORA_RANK * 2
    lse_bytes = t * h * 4
    bt_bytes = int(((lens + w.page_size - 1) // w.page_size).sum()) * 4 + w.batch * 4
    flops = 2 * h * vis * (KV_DIM + KV_LORA_RANK)
    return dict(
        kv_tokens=kv_tokens, visible_rows=vis, kv_bytes=kv_bytes, q_bytes=q_bytes,
        out_bytes=out_bytes, lse_bytes=lse_bytes, bt_bytes=bt_bytes,
        alg_bytes=kv_bytes + q_bytes + out_bytes + lse_bytes + bt_bytes,
        flops=flops, tokens=t,
    )


# ---------------------------------------------------------------- request pools


@dataclass
class RequestPool:
    """A serving-side request pool holding the pages of a batch.

    ``req_to_token [pool_rows, token_cols]`` int32: cache slot of each token
    of a pool row, slot = page id * page_size + offset in the page (the cache
    is ``[num_pages, page_size, 576]``, one slot per row); slots of tokens a
    request does not have are ``unused_slot``.  ``req_to_page [pool_rows,
    page_cols]`` int32: the same pages as a page list, 0 past a request's
    pages.  ``req_pool_indices [batch]`` int32: the pool row of each request
    of the batch.  Rows no request of the batch owns hold random values.
    """

    req_to_token: np.ndarray
    req_to_page: np.ndarray
    req_pool_indices: np.ndarray
    page_size: int


def make_request_pool(block_table: np.ndarray, seq_lens: np.ndarray, page_size: int, pool_rows: int,
                      seed: int = 0, token_cols: int | None = None, page_cols: int | None = None,
                      unused_slot: int = 2 ** 31 - 1) -> RequestPool:
    """Lay the pages of ``block_table`` (first ceil(L/page) entries of each
    row) into a request pool whose rows are a seeded random choice of
    ``pool_rows`` rows."""
    rng = np.random.default_rng(seed)
    batch = len(seq_lens)
    assert pool_rows >= batch
    lens = np.asarray(seq_lens, dtype=np.int64)
    pages = (lens + page_size - 1) // page_size
    need_pages = int(pages.max(initial=0))
    if page_cols is None:
        page_cols = max(need_pages, 1)
    if token_cols is None:
        token_cols = page_cols * page_size
    assert page_cols >= need_pages and token_cols >= need_pages * page_size
    rows = rng.choice(pool_rows, size=batch, replace=False).astype(np.int32)
    r2t = rng.integers(0, 2 ** 31 - 1, size=(pool_rows, token_cols), dtype=np.int64).astype(np.int32)
    r2p = rng.integers(0, 2 ** 31 - 1, size=(pool_rows, page_cols), dtype=np.int64).astype(np.int32)
    for b in range(batch):
        r = rows[b]
        n = int(pages[b])
        r2t[r, :] = unused_slot
        r2p[r, :] = 0
        r2p[r, :n] = block_table[b, :n]
        j = np.arange(int(lens[b]), dtype=np.int64)
        r2t[r, : len(j)] = (block_table[b, j // page_size].astype(np.int64) * page_size + j % page_size).astype(np.int32)
    return RequestPool(req_to_token=r2t, req_to_page=r2p, req_pool_indices=rows, page_size=page_size)
