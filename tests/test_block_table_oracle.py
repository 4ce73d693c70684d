"""Pins of the block-table oracle (oracle/block_table_ref.py), CPU only.

The pages print no worked example of this step, so the pins are tables
written out by hand from the pool layout (slot = page * page_size + offset in
the page), the agreement of the token-pool and page-pool constructions on one
pool, a brute-force check over every live token, and the decode's
indifference to which padding a table holds.  A plausible mistake in the
oracle (pages counted with a floor, the pool read at token i instead of
i * page_size, the batch row used in place of its pool row, wrong padding)
fails at least one of them; ``test_planted_mistake_is_caught`` plants each.
"""

import inspect
import types

import numpy as np
import pytest

from oracle import block_table_ref as BT
from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import workloads as W

U = 2 ** 31 - 1  # a slot no request has


def hand_pool():
    """Three requests in a 4-row token pool, page size 32, written out slot by
    slot.  Pool row 2: 40 tokens on pages 7 then 3.  Row 0: empty.  Row 3:
    exactly 32 tokens on page 5.  Row 1 belongs to no request."""
    r2t = np.full((4, 96), U, dtype=np.int64)
    r2t[2, :32] = np.arange(7 * 32, 8 * 32)
    r2t[2, 32:40] = np.arange(3 * 32, 3 * 32 + 8)
    r2t[3, :32] = np.arange(5 * 32, 6 * 32)
    r2t[1, :] = 12345
    pool = np.array([2, 0, 3], dtype=np.int32)
    lens = np.array([40, 0, 32], dtype=np.int32)
    return r2t.astype(np.int32), pool, lens


def pin_hand_tokens(fn):
    r2t, pool, lens = hand_pool()
    want = np.array([[7, 3, -1, -1], [-1, -1, -1, -1], [5, -1, -1, -1]], dtype=np.int32)
    got = fn(r2t, pool, lens, 32, 4)
    short = fn(r2t, pool, lens, 32, 1)
    return np.array_equal(got, want) and np.array_equal(short, want[:, :1])


def pin_hand_tokens_page64(fn):
    """Page size 64: 65 tokens need two pages, 64 need one, 1 needs one."""
    r2t = np.full((3, 192), U, dtype=np.int64)
    r2t[0, :64] = np.arange(9 * 64, 10 * 64)
    r2t[0, 64] = 2 * 64
    r2t[1, :64] = np.arange(4 * 64, 5 * 64)
    r2t[2, 0] = 11 * 64
    pool = np.array([1, 0, 2], dtype=np.int32)
    lens = np.array([64, 65, 1], dtype=np.int32)
    want = np.array([[4, -1, -1], [9, 2, -1], [11, -1, -1]], dtype=np.int32)
    return np.array_equal(fn(r2t.astype(np.int32), pool, lens, 64, 3), want)


def pin_hand_pages(fn):
    r2p = np.array([[0, 0, 0], [8, 8, 8], [7, 3, 0], [5, 0, 0]], dtype=np.int32)
    pool = np.array([2, 0, 3], dtype=np.int32)
    wide = fn(r2p, pool, 5)
    narrow = fn(r2p, pool, 2)
    return (np.array_equal(wide, [[7, 3, 0, 0, 0], [0, 0, 0, 0, 0], [5, 0, 0, 0, 0]])
            and np.array_equal(narrow, [[7, 3], [0, 0], [5, 0]]))


def random_case(seed):
    w = W.make_workload("tiny", seed=seed, seq_lens=[0, 1, 31, 32, 33, 64, 65, 200, 127, 128],
                        page_size=32 if seed % 2 else 64, pool_pages=64)
    p = W.make_request_pool(w.block_table, w.seq_lens, w.page_size, pool_rows=23, seed=seed)
    return w, p


def pin_round_trip(tok_fn, page_fn, seed):
    """On a pool laid out from a known table, both constructions give that
    table's live entries; padding is -1 (tokens) and 0 (pages)."""
    w, p = random_case(seed)
    mb = w.block_table.shape[1] + 2
    t = tok_fn(p.req_to_token, p.req_pool_indices, w.seq_lens, w.page_size, mb)
    g = page_fn(p.req_to_page, p.req_pool_indices, mb)
    n = (w.seq_lens.astype(np.int64) + w.page_size - 1) // w.page_size
    ok = True
    for b in range(w.batch):
        ok &= np.array_equal(t[b, : n[b]], w.block_table[b, : n[b]]) and np.all(t[b, n[b]:] == -1)
        ok &= np.array_equal(g[b, : n[b]], w.block_table[b, : n[b]]) and np.all(g[b, n[b]:] == 0)
    return bool(ok)


def pin_every_live_token(tok_fn, seed):
    """Brute force: every live token's slot lies in the page the table names
    for it, at its offset in the page."""
    w, p = random_case(seed)
    t = tok_fn(p.req_to_token, p.req_pool_indices, w.seq_lens, w.page_size, w.block_table.shape[1])
    for b in range(w.batch):
        for j in range(int(w.seq_lens[b])):
            slot = int(p.req_to_token[p.req_pool_indices[b], j])
            if slot != int(t[b, j // w.page_size]) * w.page_size + j % w.page_size:
                return False
    return True


def pin_decode_unchanged(tok_fn, seed):
    """The float64 decode over the constructed table equals the decode over
    the table the pool was laid out from, bit for bit."""
    w, p = random_case(seed)
    t = tok_fn(p.req_to_token, p.req_pool_indices, w.seq_lens, w.page_size, w.block_table.shape[1])
    a = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
                     w.q_len, w.page_size, w.scale, w.k_scale)
    b = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, t, w.seq_lens,
                     w.q_len, w.page_size, w.scale, w.k_scale)
    return np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def all_pins(mod):
    tok, pg = mod.block_table_from_tokens, mod.block_table_from_pages
    return [
        pin_hand_tokens(tok), pin_hand_tokens_page64(tok), pin_hand_pages(pg),
        pin_round_trip(tok, pg, 1), pin_round_trip(tok, pg, 2),
        pin_every_live_token(tok, 3), pin_every_live_token(tok, 4), pin_decode_unchanged(tok, 5),
    ]


def test_hand_written_token_pool():
    assert pin_hand_tokens(BT.block_table_from_tokens)
    assert pin_hand_tokens_page64(BT.block_table_from_tokens)


def test_hand_written_page_pool():
    assert pin_hand_pages(BT.block_table_from_pages)


@pytest.mark.parametrize("seed", [1, 2, 6, 7])
def test_round_trip_both_constructions(seed):
    assert pin_round_trip(BT.block_table_from_tokens, BT.block_table_from_pages, seed)


@pytest.mark.parametrize("seed", [3, 4])
def test_every_live_token(seed):
    assert pin_every_live_token(BT.block_table_from_tokens, seed)


def test_decode_over_constructed_table():
    assert pin_decode_unchanged(BT.block_table_from_tokens, 5)


# (name, text in the oracle, planted replacement)
MUTATIONS = [
    ("pages counted with a floor",
     "pages = (length + page_size - 1) // page_size", "pages = length // page_size"),
    ("pool read at token i",
     "req_to_token[row, i * page_size]", "req_to_token[row, i]"),
    ("pool read one token into the page",
     "req_to_token[row, i * page_size]", "req_to_token[row, i * page_size + 1]"),
    ("batch row instead of pool row (tokens)",
     "row = int(req_pool_indices[b])\n        length", "row = b\n        length"),
    ("token padding 0",
     "table = np.full((batch, max_blocks), -1, dtype=np.int64)",
     "table = np.full((batch, max_blocks), 0, dtype=np.int64)"),
    ("slot not divided by the page size",
     "table[b, i] = first_token_slot // page_size", "table[b, i] = first_token_slot"),
    ("batch row instead of pool row (pages)",
     "row = int(req_pool_indices[b])\n        for i in range(copy_len)", "row = b\n        for i in range(copy_len)"),
    ("page copy one column short",
     "copy_len = min(max_blocks, req_to_page.shape[1])", "copy_len = min(max_blocks, req_to_page.shape[1]) - 1"),
    ("page padding -1",
     "table = np.zeros((batch, max_blocks), dtype=np.int64)",
     "table = np.full((batch, max_blocks), -1, dtype=np.int64)"),
]


def mutated(old, new):
    src = inspect.getsource(BT)
    assert src.count(old) == 1, old
    mod = types.ModuleType("block_table_mutant")
    exec(compile(src.replace(old, new), "block_table_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    try:
        results = all_pins(mutated(old, new))
    except (IndexError, ValueError):
        return  # the mutant cannot even run the pins
    assert not all(results), f"no pin rejects: {name}"


def test_unmutated_passes_all_pins():
    assert all(all_pins(BT))
