"""GPU parity of the decode that takes the merged e4m3 query (the pages' FP8
path) against the float64 oracle, and the whole FP8 decode step: RoPE +
quantisation + cache write, then the decode over the written cache."""

import numpy as np
import pytest
import torch

from oracle import kv_write_ref as K
from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

from test_kv_write_oracle import roformer_cache
from test_parity import check

pytestmark = pytest.mark.gpu


def merged_e4m3_query(w, seed):
    rng = np.random.default_rng(seed)
    t, h = w.num_tokens, w.num_heads
    return W.f32_to_e4m3fn_bits(rng.standard_normal((t, h, 576)).astype(np.float32))


def run_fp8q(db, q8, cu=None):
    q = torch.from_numpy(q8).cuda()
    B.mla_decode_fp8q(db.plan, q, db.kv, db.block_table, db.seq_lens, db.w.scale, db.w.k_scale, db.out, db.lse,
                      db.workspace, cu_seqlens_q=cu)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    return db.out, db.lse


@pytest.mark.parametrize("name,kw", [("fp8_kv", {}), ("tiny", dict(kv_dtype="e4m3", k_scale=0.5, num_heads=16,
                                                                    seq_lens=[1, 65, 700, 0], page_size=32))])
def test_fp8_query_against_oracle(name, kw):
    w = W.make_workload(name, seed=1, **kw)
    q8 = merged_e4m3_query(w, 2)
    out, lse = run_fp8q(R.upload(w), q8)
    ref = O.mla_decode(q8[..., :512], q8[..., 512:], w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens, w.q_len,
                       w.page_size, w.scale, w.k_scale, q_dtype="e4m3")
    check(w, out, lse, *ref)


def test_fp8_query_equals_its_bf16_form_bitwise():
    """Every e4m3 value is exact in bf16 and fp16: decoding the e4m3 query
    and decoding its bf16 form feed the same fp16 MMAs, bit for bit."""
    w = W.make_workload("fp8_kv", seed=3, batch=32)
    q8 = merged_e4m3_query(w, 4)
    db = R.upload(w)
    o8, l8 = (t.clone() for t in run_fp8q(db, q8))
    vals = O.decode_e4m3fn(q8).astype(np.float32)
    db.q_nope = torch.from_numpy(W.f32_to_bf16_bits(vals[..., :512]).view(np.int16)).cuda().view(torch.bfloat16)
    db.q_pe = torch.from_numpy(W.f32_to_bf16_bits(vals[..., 512:]).view(np.int16)).cuda().view(torch.bfloat16)
    o16, l16 = R.decode(db)
    torch.cuda.synchronize()
    assert torch.equal(o8.view(torch.int16), o16.view(torch.int16)) and torch.equal(l8, l16)


def test_fp8_query_ragged():
    w = W.make_ragged_workload("draft_extend", seed=5, kv_dtype="e4m3", k_scale=0.5, batch=40)
    q8 = merged_e4m3_query(w, 6)
    db = R.upload(w)
    out, lse = run_fp8q(db, q8, cu=db.cu_seqlens_q)
    # the ragged oracle takes bf16 bits: give it the exact bf16 form of the e4m3 query
    vals = O.decode_e4m3fn(q8).astype(np.float32)
    ref = O.mla_decode_ragged(W.f32_to_bf16_bits(vals[..., :512]), W.f32_to_bf16_bits(vals[..., 512:]), w.kv_bits,
                              w.kv_dtype, w.block_table, w.seq_lens, w.cu_seqlens_q, w.page_size, w.scale, w.k_scale)
    check(w, out, lse, *ref)


def test_fp8_decode_step_end_to_end():
    """The pages' FP8 step: new tokens' keys roped + quantised into the e4m3
    cache, the query roped + quantised to the merged e4m3 form, then the
    decode over that cache with that query."""
    rng = np.random.default_rng(7)
    lens_before = np.array([100, 63, 2000, 0, 640, 4096], dtype=np.int32)
    w = W.make_workload("fp8_kv", seed=7, seq_lens=list(lens_before + 1), num_heads=32, k_scale=1.0,
                        pool_pages=300)
    t, h, page = w.batch, w.num_heads, w.page_size
    cs = roformer_cache(8192).astype(np.float32)
    pos = lens_before.astype(np.int64)
    slots = np.array([w.block_table[b, lens_before[b] // page] * page + lens_before[b] % page for b in range(t)],
                     dtype=np.int64)
    bf = lambda shape: W.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))  # noqa: E731
    q_nope, q_rope, k_nope, k_rope = bf((t, h, 512)), bf((t, h, 64)), bf((t, 512)), bf((t, 64))
    db = R.upload(w)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()  # noqa: E731
    q_out = torch.empty((t, h, 576), dtype=torch.uint8, device="cuda")
    B.mla_rope_quantize_cache_write(dev16(q_nope), dev16(q_rope), q_out, B.MLA_Q_E4M3, dev16(k_nope), dev16(k_rope),
                                    torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(), False, db.kv,
                                    B.MLA_KV_E4M3, torch.from_numpy(slots).cuda())
    B.mla_decode_fp8q(db.plan, q_out, db.kv, db.block_table, db.seq_lens, w.scale, w.k_scale, db.out, db.lse,
                      db.workspace)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    qc, kc, _, _ = K.rope_quantize_fp8(q_nope, q_rope, k_nope, k_rope, pos, cs, False)
    assert np.array_equal(q_out.cpu().numpy(), qc)
    kv_new = K.kv_cache_write(w.kv_bits, kc, slots, page)
    ref = O.mla_decode(qc[..., :512], qc[..., 512:], kv_new, "e4m3", w.block_table, w.seq_lens, 1, page, w.scale,
                       w.k_scale, q_dtype="e4m3")
    check(w, db.out, db.lse, *ref)
