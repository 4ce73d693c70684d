"""Pins for the float64 oracle, against facts other than the oracle itself:
closed forms, invariants, a brute-force non-absorbed MLA, a library special
case (torch SDPA in float64 on the CPU) and the float formats' definitions.
A plausible slip in the oracle (dropped rope term, wrong value slice, causal
off-by-one, wrong log base, swapped page/slot index, k_scale on one side only)
fails at least one of these; ``test_oracle_mutations.py`` plants such slips
and checks that they are caught.
"""

import math

import numpy as np
import torch

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import workloads as W

SCALE = 1.0 / math.sqrt(192.0)


def tiny_bf16_workload(seq_lens, q_len=1, h=4, page=32, seed=1, dtype="bf16", k_scale=1.0, fill="nan"):
    cfg = dict(batch=len(seq_lens), q_len=q_len, num_heads=h, page_size=page,
               kv_dtype=dtype, seq_lens=list(seq_lens), k_scale=k_scale,
               pool_pages=sum((l + page - 1) // page for l in seq_lens) + 3)
    return W.build_workload("t", cfg, seed=seed, fill=fill)


def run(w, decode=None, **kw):
    fn = decode or O.mla_decode
    return fn(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
              w.q_len, w.page_size, w.scale, w.k_scale, **kw)


# ------------------------------------------------------------ pin helpers
# Each helper returns the largest deviation it sees; the mutation test calls
# them with a deliberately broken oracle and expects a large deviation.


def pin_sdpa(decode=O.mla_decode, seed=3):
    """Library special case: per request, F.scaled_dot_product_attention in
    float64 on the CPU with an explicit bottom-right causal mask (q_len=3,
    every query row sees at least one key), keys = full 576-wide rows,
    values = first 512 columns; lse via torch.logsumexp of the masked,
    scaled logits."""
    w = tiny_bf16_workload([40, 7, 65], q_len=3, h=5, page=32, seed=seed)
    out, lse = run(w, decode)
    worst = 0.0
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        j = np.arange(L)
        rows = torch.from_numpy(
            w.kv_bits[w.block_table[b][j // w.page_size], j % w.page_size].astype(np.int16)
        ).view(torch.bfloat16).double()
        qn = torch.from_numpy(w.q_nope_bits[b * 3:(b + 1) * 3].astype(np.int16)).view(torch.bfloat16).double()
        qp = torch.from_numpy(w.q_pe_bits[b * 3:(b + 1) * 3].astype(np.int16)).view(torch.bfloat16).double()
        q = torch.cat([qn, qp], dim=-1).reshape(3 * w.num_heads, 576)  # row = i*H + h
        i = torch.arange(3).repeat_interleave(w.num_heads)
        mask = torch.arange(L)[None, :] < (L - 3 + 1 + i)[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], rows[None], rows[None, :, :512], attn_mask=mask[None], scale=SCALE)[0]
        logits = (q @ rows.T) * SCALE
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
        got = out[b * 3:(b + 1) * 3].reshape(3 * w.num_heads, 512)
        got_lse = lse[b * 3:(b + 1) * 3].reshape(-1)
        worst = max(worst, float(np.abs(got - ref.numpy()).max()),
                    float(np.abs(got_lse - ref_lse.numpy()).max()))
    return worst


def pin_absorption(attend=O.attend, seed=4):
    """Brute-force non-absorbed MLA on tiny inputs: per head, expand the
    latent rows through random W_UK (128x512) and W_UV (128x512) into full keys
    and values, attend with (q_h, q_pe), and compare with absorbed attention
    (q_nope = W_UK^T q_h over the latent rows) mapped through W_UV."""
    rng = np.random.default_rng(seed)
    h, n, dn = 3, 9, 128
    c = rng.standard_normal((n, 512))
    kpe = rng.standard_normal((n, 64))
    rows = np.concatenate([c, kpe], axis=1)
    wuk = rng.standard_normal((h, dn, 512)) / 16
    wuv = rng.standard_normal((h, dn, 512)) / 16
    qh = rng.standard_normal((h, dn))
    qpe = rng.standard_normal((h, 64))
    worst = 0.0
    # brute force, explicit loops over heads and keys
    brute_o = np.zeros((h, dn))
    brute_lse = np.zeros(h)
    for hh in range(h):
        k_nope = np.array([wuk[hh] @ c[j] for j in range(n)])  # [n,128]
        v = np.array([wuv[hh] @ c[j] for j in range(n)])  # [n,128]
        s = np.array([SCALE * (qh[hh] @ k_nope[j] + qpe[hh] @ kpe[j]) for j in range(n)])
        e = np.exp(s - s.max())
        brute_o[hh] = (e[:, None] * v).sum(0) / e.sum()
        brute_lse[hh] = s.max() + math.log(e.sum())
    q_abs = np.einsum("hdk,hd->hk", wuk, qh)
    lat, lse = attend(q_abs, qpe, rows, SCALE)
    absorbed_o = np.einsum("hdk,hk->hd", wuv, lat)
    worst = max(float(np.abs(absorbed_o - brute_o).max()), float(np.abs(lse - brute_lse).max()))
    return worst


def pin_page_permutation(decode=O.mla_decode, seed=5):
    """Moving physical pages and rewriting the block table changes nothing
    (bit-identical)."""
    w = tiny_bf16_workload([70, 33, 128, 5], q_len=2, h=3, page=32, seed=seed)
    out0, lse0 = run(w, decode)
    rng = np.random.default_rng(seed + 100)
    perm = rng.permutation(w.num_pages)  # new slot of old page p is perm[p]
    kv2 = np.empty_like(w.kv_bits)
    kv2[perm] = w.kv_bits
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out1, lse1 = decode(w.q_nope_bits, w.q_pe_bits, kv2, w.kv_dtype, bt2, w.seq_lens,
                        w.q_len, w.page_size, w.scale, w.k_scale)
    if not (np.array_equal(out0, out1) and np.array_equal(lse0, lse1)):
        return float(max(np.nanmax(np.abs(out0 - out1)), np.nanmax(np.abs(lse0 - lse1)), 1.0))
    return 0.0


def pin_single_key(decode=O.mla_decode, seed=6):
    """seq_len = 1: the output is that row's 512 latent columns exactly and
    lse is the single scaled score (the fill value padded CUDA-graph rows
    run with)."""
    w = tiny_bf16_workload([1, 1], q_len=1, h=4, page=64, seed=seed)
    out, lse = run(w, decode)
    worst = 0.0
    for b in range(2):
        row = O.decode_bf16(w.kv_bits[w.block_table[b, 0], 0])
        qn = O.decode_bf16(w.q_nope_bits[b])
        qp = O.decode_bf16(w.q_pe_bits[b])
        s0 = SCALE * (qn @ row[:512] + qp @ row[512:])
        worst = max(worst, float(np.abs(out[b] - row[None, :512]).max()), float(np.abs(lse[b] - s0).max()))
    return worst


def pin_equal_scores(decode=O.mla_decode, seed=7):
    """q = 0: every score is 0, so the output is the mean of the latent rows
    and lse = ln L."""
    w = tiny_bf16_workload([50, 97], q_len=1, h=2, page=32, seed=seed)
    w.q_nope_bits[...] = 0
    w.q_pe_bits[...] = 0
    out, lse = run(w, decode)
    worst = 0.0
    for b in range(2):
        L = int(w.seq_lens[b])
        j = np.arange(L)
        rows = O.decode_bf16(w.kv_bits[w.block_table[b][j // 32], j % 32])
        worst = max(worst, float(np.abs(out[b] - rows[:, :512].mean(0)).max()),
                    float(np.abs(lse[b] - math.log(L)).max()))
    return worst


def pin_zero_length(decode=O.mla_decode, seed=8):
    """Rows with no visible key give exactly 0 and -inf, also the early
    causal rows of a q_len=3 request holding only 2 keys."""
    w = tiny_bf16_workload([0, 2, 9], q_len=3, h=2, page=32, seed=seed)
    out, lse = run(w, decode)
    bad = 0.0
    for tok in (0, 1, 2, 3):  # request 0: all; request 1, i=0: V=2-3+1+0=0
        if not (np.all(out[tok] == 0) and np.all(np.isneginf(lse[tok]))):
            bad = 1.0
    for tok in (4, 5, 6, 7, 8):
        if not np.all(np.isfinite(lse[tok])):
            bad = 1.0
    return bad


def pin_draft_expansion(decode=O.mla_decode, seed=9):
    """q_len>1 causal decode equals the draft catch-up expansion: q_len
    separate q_len=1 rows whose seq_lens advance by one per token."""
    q_len = 4
    w = tiny_bf16_workload([11, 64, 100], q_len=q_len, h=3, page=32, seed=seed)
    out, lse = run(w, decode)
    bt = np.repeat(w.block_table, q_len, axis=0)
    lens = (np.repeat(w.seq_lens, q_len) - q_len + 1 + np.tile(np.arange(q_len), w.batch)).astype(np.int32)
    out1, lse1 = decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, bt, lens,
                        1, w.page_size, w.scale, w.k_scale)
    return float(max(np.abs(out - out1).max(), np.abs(lse - lse1).max()))


def pin_split_merge(attend=O.attend, merge=O.merge_splits, seed=10):
    """Attention over contiguous key chunks, merged by lse, equals attention
    over all keys (including an empty chunk)."""
    rng = np.random.default_rng(seed)
    rows = rng.standard_normal((77, 576))
    qn = rng.standard_normal((5, 512))
    qp = rng.standard_normal((5, 64))
    full_o, full_l = attend(qn, qp, rows, SCALE)
    cuts = [0, 10, 10, 41, 77]
    parts = [attend(qn, qp, rows[a:b], SCALE) for a, b in zip(cuts[:-1], cuts[1:])]
    o, l = merge([p[0] for p in parts], [p[1] for p in parts])
    return float(max(np.abs(o - full_o).max(), np.abs(l - full_l).max()))


def pin_fp8_scale(decode=O.mla_decode, seed=11):
    """e4m3 cache with k_scale: equals the bf16 decode of the dequantised
    values when those are bf16-exact (k_scale a power of two, e4m3 values
    are bf16-exact), i.e. k_scale multiplies both score and value."""
    w = tiny_bf16_workload([45, 64], q_len=1, h=3, page=32, seed=seed, dtype="e4m3", k_scale=0.5)
    out, lse = run(w, decode)
    vals = O.decode_e4m3fn(w.kv_bits) * 0.5
    vals = np.where(np.isnan(vals), 0.0, vals)
    kv16 = W.f32_to_bf16_bits(vals.astype(np.float32))
    out2, lse2 = decode(w.q_nope_bits, w.q_pe_bits, kv16, "bf16", w.block_table, w.seq_lens,
                        1, w.page_size, w.scale, 1.0)
    return float(max(np.abs(out - out2).max(), np.abs(lse - lse2).max()))


# ------------------------------------------------------------ tests


def test_sdpa_special_case():
    assert pin_sdpa() < 1e-12


def test_absorption_identity():
    assert pin_absorption() < 1e-10


def test_page_permutation_invariance():
    assert pin_page_permutation() == 0.0


def test_single_key():
    assert pin_single_key() < 1e-13


def test_equal_scores_mean():
    assert pin_equal_scores() < 1e-13


def test_zero_length_rows():
    assert pin_zero_length() == 0.0


def test_draft_expansion():
    assert pin_draft_expansion() == 0.0


def test_split_merge():
    assert pin_split_merge() < 1e-12


def test_fp8_scale_reading():
    assert pin_fp8_scale() < 1e-12


def test_merge_all_empty():
    o, l = O.merge_splits([np.ones((2, 3)), np.ones((2, 3))], [np.full(2, -np.inf), np.full(2, -np.inf)])
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_closed_form_two_keys():
    """Worked by hand: one head, two keys whose scaled scores are 0 and ln 3
    (weights 1/4, 3/4); output = (r0 + 3 r1)/4, lse = ln 4."""
    r = np.zeros((2, 576))
    r[0, :512] = 1.0
    r[1, :512] = 5.0
    qn = np.zeros((1, 512))
    qp = np.zeros((1, 64))
    # put the score on the rope column: s1 = SCALE * qp[0]*r[1,512] = ln 3
    r[1, 512] = 1.0
    qp[0, 0] = math.log(3.0) / SCALE
    out, lse = O.attend(qn, qp, r, SCALE)
    assert np.allclose(out[0], (1.0 + 3 * 5.0) / 4.0, rtol=0, atol=1e-14)
    assert abs(lse[0] - math.log(4.0)) < 1e-14


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    with np.errstate(invalid="ignore"):  # the NaN bit patterns are part of the sweep
        got = O.decode_bf16(bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])


def test_e4m3_decode_matches_format_and_torch():
    # values fixed by the e4m3fn definition
    assert O.decode_e4m3fn(np.uint8(0x38)) == 1.0
    assert O.decode_e4m3fn(np.uint8(0xB8)) == -1.0
    assert O.decode_e4m3fn(np.uint8(0x7E)) == 448.0
    assert O.decode_e4m3fn(np.uint8(0x08)) == 2.0 ** -6
    assert O.decode_e4m3fn(np.uint8(0x01)) == 2.0 ** -9
    assert O.decode_e4m3fn(np.uint8(0x07)) == 7 * 2.0 ** -9
    assert np.isnan(O.decode_e4m3fn(np.uint8(0x7F))) and np.isnan(O.decode_e4m3fn(np.uint8(0xFF)))
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = O.decode_e4m3fn(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])


def test_generator_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 4,
                        np.float32([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 300.0, 1000.0, -1000.0, 2 ** -10])])
    bf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), bf)
    x8 = np.clip(x, -448, 448)
    f8 = torch.from_numpy(x8).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(W.f32_to_e4m3fn_bits(x8), f8)
    # saturation
    assert W.f32_to_e4m3fn_bits(np.float32([1000.0]))[0] == 0x7E


def test_tail_rows_never_read():
    """NaN in every cache slot no request owns (tails and spare pages) and -1
    or garbage in padding block-table entries leave the result unchanged."""
    a = tiny_bf16_workload([70, 33], q_len=1, h=3, page=32, seed=12, fill="nan")
    out, lse = run(a)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    a.block_table[a.block_table < 0] = 10 ** 6
    out2, lse2 = run(a)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_golden_tiny():
    """Regression pin: the oracle's output on the seeded tiny workload equals
    the values written by tests/golden/make_golden.py."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.txt")
    stored = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split("=", 1)
            stored[k.strip()] = np.array([float(x) for x in v.split()])
    w = W.make_workload("tiny", seed=0)
    out, lse = run(w)
    assert np.allclose(lse.reshape(-1), stored["lse"], rtol=0, atol=1e-12)
    assert np.allclose(out.reshape(-1)[:: 97], stored["out_every_97th"], rtol=0, atol=1e-12)
    assert np.allclose(out.sum(axis=-1).reshape(-1), stored["out_row_sums"], rtol=0, atol=1e-10)


def test_e4m3_query_is_its_exact_value():
    """An e4m3 query decodes to the same numbers as its exact bf16 form
    (every e4m3 value is a bf16 value): the two decodes agree bit for bit."""
    from paged_mla_decode_08_gb300 import workloads as W
    rng = np.random.default_rng(31)
    w = W.make_workload("tiny", seed=31, kv_dtype="e4m3", k_scale=0.5, seq_lens=[70, 1, 0], num_heads=4)
    qn8 = W.f32_to_e4m3fn_bits(rng.standard_normal(w.q_nope_bits.shape).astype(np.float32))
    qp8 = W.f32_to_e4m3fn_bits(rng.standard_normal(w.q_pe_bits.shape).astype(np.float32))
    qn16 = W.f32_to_bf16_bits(O.decode_e4m3fn(qn8).astype(np.float32))
    qp16 = W.f32_to_bf16_bits(O.decode_e4m3fn(qp8).astype(np.float32))
    assert np.array_equal(O.decode_bf16(qn16), O.decode_e4m3fn(qn8))  # exact
    a = O.mla_decode(qn8, qp8, w.kv_bits, "e4m3", w.block_table, w.seq_lens, 1, w.page_size, w.scale, 0.5,
                     q_dtype="e4m3")
    b = O.mla_decode(qn16, qp16, w.kv_bits, "e4m3", w.block_table, w.seq_lens, 1, w.page_size, w.scale, 0.5)
    assert np.array_equal(a[0], b[0], equal_nan=True) and np.array_equal(a[1], b[1])
