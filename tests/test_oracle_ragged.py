"""Pins of the oracle's ragged-query decode (``mla_decode_ragged``), CPU only.

The serving pages reach a ragged batch by padding every request's queries to
the longest, running the uniform decode with shifted lengths, and dropping
the padding rows.  That route, written out here with the oracle's uniform
decode (itself pinned in test_oracle.py) as a step, must give the ragged
result exactly; so must the uniform case and each request decoded alone.
Planted mistakes (causal rule from the longest query, packed rows read at
request * max_q, an off-by-one in the visible count) must fail a pin.
"""

import inspect
import types

import numpy as np
import pytest

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import workloads as W


def ragged_case(seed, q_lens, lens, page=32):
    # the cache covers each request's padded length (L - q_b + max_q), as the
    # pages' block table does for the padded route
    q_lens = np.asarray(q_lens)
    lens = np.asarray(lens)
    pad_lens = lens - q_lens + q_lens.max()
    w = W.make_ragged_workload("draft_extend", seed=seed, q_lens=q_lens, seq_lens=list(pad_lens),
                               num_heads=4, page_size=page, pool_pages=64)
    return w, lens.astype(np.int32)


def ragged(mod, w, lens):
    return mod.mla_decode_ragged(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, lens,
                                 w.cu_seqlens_q, w.page_size, w.scale, w.k_scale)


def pin_pad_route(mod, seed):
    """Pad to max_q (zero queries), decode uniformly with seq_lens_k =
    L - q_b + max_q, keep each request's first q_b rows."""
    q_lens = [1, 3, 2, 4, 1, 4]
    lens = [40, 3, 100, 70, 1, 2]   # includes requests shorter than their query count
    w, L = ragged_case(seed, q_lens, lens)
    b, mq, h = len(q_lens), max(q_lens), w.num_heads
    cu = w.cu_seqlens_q
    pn = np.zeros((b * mq, h, 512), dtype=np.uint16)
    pp = np.zeros((b * mq, h, 64), dtype=np.uint16)
    for r in range(b):
        pn[r * mq: r * mq + q_lens[r]] = w.q_nope_bits[cu[r]: cu[r + 1]]
        pp[r * mq: r * mq + q_lens[r]] = w.q_pe_bits[cu[r]: cu[r + 1]]
    seq_k = L - np.asarray(q_lens) + mq
    po, pl = O.mla_decode(pn, pp, w.kv_bits, w.kv_dtype, w.block_table, seq_k, mq, w.page_size, w.scale)
    ro, rl = ragged(mod, w, L)
    for r in range(b):
        for i in range(q_lens[r]):
            if not (np.array_equal(ro[cu[r] + i], po[r * mq + i]) and np.array_equal(rl[cu[r] + i], pl[r * mq + i])):
                return False
    return True


def pin_uniform(mod, seed):
    """Equal query counts: the uniform decode, row for row."""
    q = 3
    w, L = ragged_case(seed, [q] * 4, [90, 2, 64, 33])
    uo, ul = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, L, q, w.page_size,
                          w.scale)
    ro, rl = ragged(mod, w, L)
    return np.array_equal(ro, uo) and np.array_equal(rl, ul)


def pin_alone(mod, seed):
    """Each request decoded alone (batch of one, q_len = q_b) gives its rows;
    a request with no query token owns no row."""
    q_lens = [2, 0, 4, 1]
    w, L = ragged_case(seed, q_lens, [50, 10, 129, 7])
    ro, rl = ragged(mod, w, L)
    cu = w.cu_seqlens_q
    if ro.shape[0] != sum(q_lens) or np.isnan(ro).any():
        return False
    for r in range(len(q_lens)):
        if q_lens[r] == 0:
            continue
        ao, al = O.mla_decode(w.q_nope_bits[cu[r]: cu[r + 1]], w.q_pe_bits[cu[r]: cu[r + 1]], w.kv_bits,
                              w.kv_dtype, w.block_table[r: r + 1], L[r: r + 1], q_lens[r], w.page_size, w.scale)
        if not (np.array_equal(ro[cu[r]: cu[r + 1]], ao) and np.array_equal(rl[cu[r]: cu[r + 1]], al)):
            return False
    return True


def pin_empty_rows(mod, seed):
    """Token i of a request with L < q_b - i sees no key: 0 and -inf."""
    w, L = ragged_case(seed, [4, 1], [2, 0])
    ro, rl = ragged(mod, w, L)
    # request 0: tokens 0, 1 see 2-4+1+i <= 0 keys; request 1 sees none
    return (np.all(ro[[0, 1, 4]] == 0) and np.all(np.isneginf(rl[[0, 1, 4]]))
            and np.all(np.isfinite(rl[[2, 3]])))


def all_pins(mod):
    return [pin_pad_route(mod, 1), pin_pad_route(mod, 2), pin_uniform(mod, 3), pin_alone(mod, 4),
            pin_empty_rows(mod, 5)]


def test_pad_route():
    assert pin_pad_route(O, 1) and pin_pad_route(O, 2)


def test_uniform_special_case():
    assert pin_uniform(O, 3)


def test_requests_alone():
    assert pin_alone(O, 4)


def test_empty_rows():
    assert pin_empty_rows(O, 5)


MUTATIONS = [
    ("causal rule from the longest query",
     "v = max(n - q_b + 1 + i, 0)\n            out[t0 + i]",
     "v = max(n - int(np.diff(cu_seqlens_q).max()) + 1 + i, 0)\n            out[t0 + i]"),
    ("packed rows read at request * max_q",
     "t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])",
     "t0, t1 = b * int(np.diff(cu_seqlens_q).max()), b * int(np.diff(cu_seqlens_q).max()) + int(cu_seqlens_q[b + 1] - cu_seqlens_q[b])"),
    ("visible count one short",
     "v = max(n - q_b + 1 + i, 0)\n            out[t0 + i]", "v = max(n - q_b + i, 0)\n            out[t0 + i]"),
    ("top-left causal alignment",
     "v = max(n - q_b + 1 + i, 0)\n            out[t0 + i]", "v = min(i + 1, n)\n            out[t0 + i]"),
]


def mutated(old, new):
    src = inspect.getsource(O)
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_ragged_mutant")
    exec(compile(src.replace(old, new), "oracle_ragged_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    try:
        results = all_pins(mutated(old, new))
    except (IndexError, ValueError):
        return
    assert not all(results), f"no pin rejects: {name}"


def test_unmutated_passes_all_pins():
    assert all(all_pins(O))
