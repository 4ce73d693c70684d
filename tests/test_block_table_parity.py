"""GPU parity of the block-table builders against the CPU oracle, bit-exact
(integer work), through the C ABI; then the built table driving the decode.

Every case prefills the output table with a garbage pattern, so an entry the
kernel failed to write shows up as a mismatch.
"""

import numpy as np
import pytest
import torch

from oracle import block_table_ref as BT
from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GARBAGE = 0x5A5A5A5A


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def build_tokens(pool, lens, page, max_blocks, batch=None):
    batch = len(lens) if batch is None else batch
    bt = torch.full((batch, max_blocks), GARBAGE, dtype=torch.int32, device="cuda")
    B.mla_block_table_from_tokens(dev(pool.req_to_token), dev(pool.req_pool_indices), dev(lens), page, bt)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    return bt.cpu().numpy()


def build_pages(pool, max_blocks):
    bt = torch.full((len(pool.req_pool_indices), max_blocks), GARBAGE, dtype=torch.int32, device="cuda")
    B.mla_block_table_from_pages(dev(pool.req_to_page), dev(pool.req_pool_indices), bt)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    return bt.cpu().numpy()


def case(name, seed, **kw):
    w = W.make_workload(name, seed=seed, **kw)
    pool = W.make_request_pool(w.block_table, w.seq_lens, w.page_size, pool_rows=w.batch + 37, seed=seed)
    return w, pool


CASES = [
    ("tiny", dict(seq_lens=[0, 1, 31, 32, 33, 63, 64, 65, 200], page_size=32, pool_pages=64)),
    ("tiny", dict(seq_lens=[0, 1, 31, 32, 33, 63, 64, 65, 200], page_size=64, pool_pages=64)),
    ("dsv3", dict()),
    ("spec_q4", dict(batch=64)),
    ("long_skewed", dict(seq_lens=[131072, 17, 0, 40000])),   # 4096 entries: 16 chunks
    ("tiny", dict(seq_lens=list(np.random.default_rng(3).integers(0, 300, size=700)), pool_pages=8192)),
]


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("extra", [0, 5, -1])
def test_from_tokens_matches_oracle(name, kw, extra):
    w, pool = case(name, 1, **kw)
    need = max(int(w.block_table.shape[1]), 1)
    mb = max(need + extra, 1)   # extra < 0: a table narrower than the longest request
    got = build_tokens(pool, w.seq_lens, w.page_size, mb)
    want = BT.block_table_from_tokens(pool.req_to_token, pool.req_pool_indices, w.seq_lens, w.page_size, mb)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("extra", [0, 7, -1])
def test_from_pages_matches_oracle(name, kw, extra):
    w, pool = case(name, 2, **kw)
    mb = max(pool.req_to_page.shape[1] + extra, 1)
    got = build_pages(pool, mb)
    want = BT.block_table_from_pages(pool.req_to_page, pool.req_pool_indices, mb)
    assert np.array_equal(got, want)


def test_out_of_range_lookups_are_reported_not_read():
    """Pool row -1 and past the pool, a lookup past the pool's columns, a
    negative slot and a negative length: each entry gets the padding value
    and the error word names the first event; nothing is read out of
    bounds."""
    page = 64
    r2t = np.zeros((4, 128), dtype=np.int32)
    r2t[0, :] = np.arange(128) + 5 * page
    r2t[1, 64] = -7
    pool = W.RequestPool(req_to_token=r2t, req_to_page=np.zeros((4, 3), np.int32),
                         req_pool_indices=np.array([0], np.int32), page_size=page)
    base = build_tokens(pool, np.array([128], np.int32), page, 4)
    assert np.array_equal(base, [[5, 6, -1, -1]])
    for idx, L, code in [(-1, 10, 0x301), (4, 10, 0x301), (0, 129, 0x302), (1, 100, 0x304), (0, -3, 0x303)]:
        pool.req_pool_indices = np.array([idx], np.int32)
        bt = torch.full((1, 4), GARBAGE, dtype=torch.int32, device="cuda")
        B.mla_block_table_from_tokens(dev(r2t), dev(pool.req_pool_indices), dev([L]), page, bt)
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == code
        row = bt.cpu().numpy()[0]
        if code == 0x302:   # the third page's first token lies past the pool's 128 columns
            assert np.array_equal(row, [5, 6, -1, -1])
        elif code == 0x304:
            assert row[0] == 0 and np.all(row[1:] == -1)
        else:
            assert np.all(row == -1)
    r2p = np.arange(12, dtype=np.int32).reshape(4, 3)
    bt = torch.full((2, 4), GARBAGE, dtype=torch.int32, device="cuda")
    B.mla_block_table_from_pages(dev(r2p), dev([3, 9]), bt)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0x301
    assert np.array_equal(bt.cpu().numpy(), [[9, 10, 11, 0], [0, 0, 0, 0]])


@pytest.mark.parametrize("name", ["dsv3", "fp8_kv"])
def test_built_table_drives_decode(name):
    """Token pool -> GPU block table -> GPU decode equals the oracle decode
    over the table the pool was laid out from, and the decode over the
    workload's own table bit for bit."""
    w, pool = case(name, 3)
    mb = w.block_table.shape[1] + 3
    db = R.upload(w)
    out0, lse0 = (t.clone() for t in R.decode(db))
    bt = torch.full((w.batch, mb), GARBAGE, dtype=torch.int32, device="cuda")
    B.mla_block_table_from_tokens(dev(pool.req_to_token), dev(pool.req_pool_indices), db.seq_lens,
                                  w.page_size, bt)
    db.block_table = bt
    out, lse = R.decode(db)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16)) and torch.equal(lse, lse0)
    from test_parity import check
    check(w, out, lse, *O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table,
                                     w.seq_lens, w.q_len, w.page_size, w.scale, w.k_scale))


def test_graph_captured_build_and_decode():
    """Block-table build and decode captured together in one CUDA graph, then
    replayed after the pool row indices and lengths change on the device."""
    lens = np.array([2000, 1000, 300, 5, 64, 1500], dtype=np.int32)
    upper = np.array([2600, 1600, 900, 700, 700, 2100], dtype=np.int32)
    w = W.make_workload("dsv3", seed=4, seq_lens=list(lens), bt_extra_cols=12)
    pool = W.make_request_pool(w.block_table, w.seq_lens, w.page_size, pool_rows=40, seed=4,
                               token_cols=w.block_table.shape[1] * w.page_size)
    db = R.upload(w, plan_seq_lens=upper)
    r2t, idx = dev(pool.req_to_token), dev(pool.req_pool_indices)
    bt = torch.full_like(db.block_table, GARBAGE)
    B.mla_block_table_from_tokens(r2t, idx, db.seq_lens, w.page_size, bt)
    B.mla_decode(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, bt, db.seq_lens, w.scale, w.k_scale,
                 db.out, db.lse, db.workspace)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.mla_block_table_from_tokens(r2t, idx, db.seq_lens, w.page_size, bt, stream=s)
            B.mla_decode(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, bt, db.seq_lens, w.scale,
                         w.k_scale, db.out, db.lse, db.workspace, None, s)
    # second replay: the batch's requests in another order, some shorter
    # (each new length within both the planned upper bound of its batch slot
    # and the tokens its pool row holds)
    perm = np.array([5, 0, 3, 1, 4, 2])
    new_lens = np.minimum(lens[perm], np.array([1500, 1600, 1, 700, 0, 300]))
    assert np.all(new_lens <= upper)
    from test_parity import check
    for ln, order in ((lens, np.arange(6)), (new_lens, perm)):
        bt.fill_(GARBAGE)
        db.seq_lens.copy_(torch.from_numpy(ln.astype(np.int32)))
        idx.copy_(torch.from_numpy(pool.req_pool_indices[order]))
        g.replay()
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0
        want_bt = BT.block_table_from_tokens(pool.req_to_token, pool.req_pool_indices[order], ln, w.page_size,
                                             bt.shape[1])
        assert np.array_equal(bt.cpu().numpy(), want_bt)
        ref_out, ref_lse = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, want_bt, ln,
                                        w.q_len, w.page_size, w.scale, w.k_scale)
        check(w, db.out, db.lse, ref_out, ref_lse)
