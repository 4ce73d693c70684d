"""GPU parity of the ragged-query decode (per-request query counts packed by
cu_seqlens_q) against the float64 oracle, through the C ABI, with the same
tolerances as the uniform decode."""

import numpy as np
import pytest
import torch

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

from test_parity import check, run_gpu

pytestmark = pytest.mark.gpu


def oracle_ragged(w, seq_lens=None, cu=None):
    return O.mla_decode_ragged(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table,
                               w.seq_lens if seq_lens is None else seq_lens,
                               w.cu_seqlens_q if cu is None else cu, w.page_size, w.scale, w.k_scale)


@pytest.mark.parametrize("seed", [0, 1])
def test_draft_extend_full(seed):
    """The draft-extend workload at full size (B=128, q_len~U{1..4}, H=16)."""
    w = W.make_ragged_workload("draft_extend", seed=seed)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle_ragged(w))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("page", [32, 64])
def test_edges(kv_dtype, page):
    """Zero-query requests, requests shorter than their query count, splits
    of long requests (combine over ragged rows), both page sizes, NaN in
    every unread cache slot."""
    q_lens = [3, 0, 1, 4, 2, 4, 0, 1]
    lens = [2, 50, 0, 30000, 129, 1, 7, 9000]
    w = W.make_ragged_workload("draft_extend", seed=2, q_lens=q_lens, seq_lens=lens, page_size=page,
                               kv_dtype=kv_dtype, k_scale=0.5 if kv_dtype == "e4m3" else 1.0, fill="nan",
                               pool_pages=2048)
    db, out, lse = run_gpu(w)
    assert db.plan.num_partial_slots > 0
    check(w, out, lse, *oracle_ragged(w))


@pytest.mark.parametrize("heads,q_lens", [(16, [8, 1, 5, 8]), (128, [1, 0, 1, 1]), (3, [7, 2, 40, 1])])
def test_row_counts(heads, q_lens):
    """Up to 128 query rows per request (heads x the largest count)."""
    lens = [3000, 64, 5000, 700]
    w = W.make_ragged_workload("draft_extend", seed=3, q_lens=q_lens, seq_lens=lens, num_heads=heads)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle_ragged(w))


def test_equal_counts_match_uniform_bitwise():
    """A ragged batch whose requests all carry q tokens is the uniform decode,
    bit for bit."""
    w = W.make_ragged_workload("draft_extend", seed=4, q_lens=[3] * 16, batch=16)
    _, out_r, lse_r = run_gpu(w)
    out_r, lse_r = out_r.clone(), lse_r.clone()
    u = W.make_ragged_workload("draft_extend", seed=4, q_lens=[3] * 16, batch=16)
    u.cu_seqlens_q = None
    _, out_u, lse_u = run_gpu(u)
    assert torch.equal(out_r.view(torch.int16), out_u.view(torch.int16)) and torch.equal(lse_r, lse_u)


def test_malformed_offsets_are_reported_not_followed():
    """Device offsets that break the planned bounds: that request gets no row
    (nothing read or written), the others are exact, the error word is 0x501.
    Planned counts [2, 3, 1]: at most 3 tokens per request, 6 rows."""
    w = W.make_ragged_workload("draft_extend", seed=5, q_lens=[2, 3, 1], seq_lens=[900, 5000, 40])
    db = R.upload(w)
    ref_out, ref_lse = oracle_ragged(w)
    sentinel = 1024.0  # exact in bf16 and fp32
    cases = [
        ([0, 2, 6, 6], [0, 1]),           # request 1: 4 tokens > 3 planned; request 2: none
        ([0, 2, 5, 9], [0, 1, 2, 3, 4]),  # request 2 ends past the 6 rows
        ([3, 2, 5, 6], [2, 3, 4, 5]),     # request 0 ends before it starts
    ]
    for cu, good_rows in cases:
        db.cu_seqlens_q.copy_(torch.tensor(cu, dtype=torch.int32))
        db.out.fill_(sentinel)
        db.lse.fill_(sentinel)
        R.decode(db)
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0x501
        rows = np.array(good_rows)
        check(w, db.out, db.lse, ref_out, ref_lse, rows=rows)
        untouched = np.setdiff1d(np.arange(w.num_tokens), rows)
        assert np.all(db.lse.cpu().numpy()[untouched] == sentinel), "a dropped request wrote lse"
        assert torch.all(db.out[torch.from_numpy(untouched)].float() == sentinel), "a dropped request wrote out"
    db.cu_seqlens_q.copy_(torch.from_numpy(w.cu_seqlens_q))
    R.decode(db)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    check(w, db.out, db.lse, ref_out, ref_lse)


def test_graph_replay_with_new_counts():
    """Planned once for at most 4 tokens per request, captured into a CUDA
    graph, replayed with other device query counts and lengths."""
    q_lens = np.array([4, 4, 4, 4, 4, 4])
    lens = np.array([2000, 1000, 300, 5, 64, 1500], dtype=np.int32)
    w = W.make_ragged_workload("draft_extend", seed=6, q_lens=q_lens, seq_lens=list(lens))
    db = R.upload(w)
    R.decode(db)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            R.decode(db, s)
    for new_q, new_l in (([4, 4, 4, 4, 4, 4], lens), ([1, 3, 0, 2, 4, 1], [1999, 640, 300, 1, 64, 1]),
                         ([0, 0, 1, 0, 0, 0], [0, 0, 7, 0, 0, 0])):
        cu = np.zeros(7, dtype=np.int32)
        cu[1:] = np.cumsum(new_q)
        new_l = np.asarray(new_l, dtype=np.int32)
        db.cu_seqlens_q.copy_(torch.from_numpy(cu))
        db.seq_lens.copy_(torch.from_numpy(new_l))
        db.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0
        ref_out, ref_lse = oracle_ragged(w, seq_lens=new_l, cu=cu)
        rows = np.arange(int(cu[-1]))
        if len(rows):
            check(w, db.out, db.lse, ref_out, ref_lse, rows=rows)
