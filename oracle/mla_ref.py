"""Float64 CPU oracle for weight-absorbed MLA decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this file: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  It shares no code, table or helper with the CUDA path.

What it computes is the plain definition of the decode the serving pages call
into (no blocking, no split-KV, no online softmax).  For request ``b`` with
``L = seq_lens[b]`` cache tokens and query position ``i`` of ``q_len``:

1. visible keys ``V = L - q_len + 1 + i`` (bottom-right causal alignment: the
   last query token sees all L keys).  Sources: tokenspeed ``flashmla.py``,
   ``FlashMLABackend.forward_extend`` (``flash_mla_with_kvcache(...,
   cache_seqlens=seq_lens + draft_token_num, causal=True)``); tokenspeed
   ``trtllm_mla.py``, ``forward_decode`` (draft catch-up: per-token seq_lens
   advance by one so each token sees its own KV write); sglang
   ``trtllm_mla_backend.py``, ``init_forward_metadata`` (target verify uses
   ``seq_lens + num_draft_tokens``).
2. ``V <= 0``: output 0 and lse = -inf (sglang ``trtllm_mla_backend.py``,
   ``forward_extend``: zero-KV rows are forced to out=0, lse=-inf so that a
   later merge ignores them).
3. cache row ``j < V`` is ``kv_pages[block_table[b][j // page], j % page]``
   (sglang ``forward_decode``: ``k_cache.view(-1, page_size,
   kv_cache_dim)``; tokenspeed ``trtllm_mla.py``, ``_create_block_kv_indices``:
   entries past the request's pages are never read).  FP8 rows are
   dequantised as ``k_scale * stored`` (tokenspeed ``forward_decode``:
   ``bmm1_scale = k_scale * layer.scaling``; sglang
   ``_compute_decode_bmm1_scale``: k_scale applies only to an FP8 cache).
4. score ``s_j = scale * (q_nope . row[:512] + q_pe . row[512:])`` with
   ``scale = 1/sqrt(head_dim)`` (``layer.scaling``), row width 576 =
   kv_lora_rank 512 + qk_rope_head_dim 64.
5. ``out = sum_j softmax(s)_j * row_j[:512]`` (``head_dim_v = kv_lora_rank``
   in ``flash_mla_with_kvcache``) and ``lse = ln sum_j exp(s_j)``.

``mla_decode_ragged`` is the same decode with a different number of query
tokens per request (packed by ``cu_seqlens_q``); token i of a request with
q_b tokens sees ``L - q_b + 1 + i`` keys, the result of the pages' pad /
uniform decode / unpad route (pinned against that route in
tests/test_oracle_ragged.py).

Readings taken where the pages are silent: lse uses the natural log and
includes the scale; the FP8 value scale equals k_scale (the latent row is both
key and value); the stored query stays bf16.
"""

from __future__ import annotations

import numpy as np

KV_LORA_RANK = 512
ROPE_DIM = 64
KV_DIM = KV_LORA_RANK + ROPE_DIM


# ------------------------------------------------------------------ decoding


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _e4m3fn_table() -> np.ndarray:
    """All 256 float8 e4m3fn values, from the format definition: sign bit,
    4-bit exponent with bias 7, 3-bit mantissa; exponent 0 encodes
    subnormals mant/8 * 2^-6; exponent 15 with mantissa 7 is NaN (no inf)."""
    t = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            t[code] = np.nan
        elif e == 0:
            t[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            t[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


E4M3FN_VALUES = _e4m3fn_table()


def decode_e4m3fn(bits: np.ndarray) -> np.ndarray:
    return E4M3FN_VALUES[np.asarray(bits, dtype=np.uint8)]


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return decode_bf16(bits)
    if dtype == "e4m3":
        return decode_e4m3fn(bits)
    raise ValueError(dtype)


# ------------------------------------------------------------------ decode


def gather_rows(kv_bits: np.ndarray, bt_row: np.ndarray, n: int, page_size: int) -> np.ndarray:
    """Stored rows 0..n-1 of one request, in token order, via its block table."""
    j = np.arange(n, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[j // page_size]
    return kv_bits[pages, j % page_size]


def request_rows(kv_bits: np.ndarray, kv_dtype: str, bt_row: np.ndarray, n: int, page_size: int,
                 k_scale: float) -> np.ndarray:
    """Dequantised float64 cache rows 0..n-1 of one request: an FP8 cache
    scales by k_scale, a bf16 cache is taken as stored."""
    dq = k_scale if kv_dtype == "e4m3" else 1.0
    return decode(gather_rows(kv_bits, bt_row, n, page_size), kv_dtype) * dq


def attend(qn: np.ndarray, qp: np.ndarray, rows: np.ndarray, scale: float):
    """Softmax attention of query heads ``qn [H,512]``, ``qp [H,64]`` over
    cache rows ``rows [V,576]`` (float64).  Returns (out [H,512], lse [H])."""
    h = qn.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((h, KV_LORA_RANK)), np.full(h, -np.inf)
    s = scale * (qn @ rows[:, :KV_LORA_RANK].T + qp @ rows[:, KV_LORA_RANK:].T)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1)
    out = (p @ rows[:, :KV_LORA_RANK]) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return out, lse


def mla_decode(
    q_nope_bits: np.ndarray,
    q_pe_bits: np.ndarray,
    kv_bits: np.ndarray,
    kv_dtype: str,
    block_table: np.ndarray,
    seq_lens: np.ndarray,
    q_len: int,
    page_size: int,
    scale: float,
    k_scale: float = 1.0,
    requests=None,
    q_dtype: str = "bf16",
):
    """Reference decode over stored inputs.

    q_nope_bits [T,H,512], q_pe_bits [T,H,64]: uint16 bf16 bits, or with
    q_dtype="e4m3" uint8 e4m3fn codes (the merged FP8 query of the pages'
    FP8 path, split at column 512; decoded exactly, no query scale: sglang
    trtllm_mla_backend.py, _compute_decode_bmm1_scale takes q_scale = 1);
    kv_bits [P,page,576] (uint16 bf16 bits or uint8 e4m3fn codes).
    Returns float64 (out [T,H,512], lse [T,H]); with ``requests`` given, only
    those requests' rows are filled (the rest stay NaN).
    """
    t, h, _ = q_nope_bits.shape
    out = np.full((t, h, KV_LORA_RANK), np.nan)
    lse = np.full((t, h), np.nan)
    reqs = range(len(seq_lens)) if requests is None else requests
    for b in reqs:
        n = int(seq_lens[b])
        rows = request_rows(kv_bits, kv_dtype, block_table[b], n, page_size, k_scale)
        for i in range(q_len):
            tok = b * q_len + i
            v = max(n - q_len + 1 + i, 0)
            out[tok], lse[tok] = attend(
                decode(q_nope_bits[tok], q_dtype), decode(q_pe_bits[tok], q_dtype), rows[:v], scale
            )
    return out, lse


def mla_decode_ragged(
    q_nope_bits: np.ndarray,
    q_pe_bits: np.ndarray,
    kv_bits: np.ndarray,
    kv_dtype: str,
    block_table: np.ndarray,
    seq_lens: np.ndarray,
    cu_seqlens_q: np.ndarray,
    page_size: int,
    scale: float,
    k_scale: float = 1.0,
):
    """Reference decode with a different number of query tokens per request
    (draft extend with a varying count of accepted drafts).

    Query tokens of request b are rows ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1``
    of ``q_*_bits [T,H,*]`` (sglang ``trtllm_mla_backend.py``,
    ``init_forward_metadata``, draft-extend branch: ``cu_seqlens_q`` is the
    zero-prefixed cumulative sum of ``extend_seq_lens``).  With ``q_b`` tokens
    and ``L = seq_lens[b]`` cache tokens (its own new tokens included), token
    i < q_b sees ``V = L - q_b + 1 + i`` keys: the pages pad every request's
    queries to ``max_q`` rows, run the uniform decode with ``seq_lens_k = L -
    q_b + max_q`` (same file, draft-extend branch and ``forward_extend``:
    ``pad_draft_extend_query`` / ``unpad_draft_extend_output``), and keep
    the first ``q_b`` rows, whose bottom-right causal rule gives that count.
    Returns float64 (out [T,H,512], lse [T,H]); rows no request owns stay NaN.
    """
    t, h, _ = q_nope_bits.shape
    out = np.full((t, h, KV_LORA_RANK), np.nan)
    lse = np.full((t, h), np.nan)
    for b in range(len(seq_lens)):
        n = int(seq_lens[b])
        t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        q_b = t1 - t0
        rows = request_rows(kv_bits, kv_dtype, block_table[b], n, page_size, k_scale)
        for i in range(q_b):
            v = max(n - q_b + 1 + i, 0)
            out[t0 + i], lse[t0 + i] = attend(
                decode_bf16(q_nope_bits[t0 + i]), decode_bf16(q_pe_bits[t0 + i]), rows[:v], scale
            )
    return out, lse


def merge_splits(outs, lses):
    """Merge attention results over disjoint key sets by their log-sum-exp:
    ``lse = ln sum_k exp(lse_k)``, ``out = sum_k exp(lse_k - lse) out_k``;
    parts with lse=-inf weigh nothing, all -inf gives 0 and -inf."""
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in lses])
    outs = np.stack([np.asarray(x, dtype=np.float64) for x in outs])
    m = lses.max(axis=0)
    safe_m = np.where(np.isneginf(m), 0.0, m)
    w = np.exp(lses - safe_m)
    tot = w.sum(axis=0)
    lse = np.where(tot > 0, safe_m + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wn = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)
    out = (wn[..., None] * outs).sum(axis=0)
    return out, lse
