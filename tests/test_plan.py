"""Host split-KV planner: bit-exact against a plain restatement of its
documented rule, plus the coverage invariants any valid schedule must meet
(each (request, tile) in exactly one segment, a request's segments contiguous
and in order, one direct segment or consecutive partial slots)."""

import numpy as np
import pytest

from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import workloads as W


def plan_rule(lens, workers, tile, ovh, min_split):
    """The planner's rule, restated: a capacity-bounded greedy fill of the
    workers in request order (tiles + ovh per segment, pieces of at least
    min_split tiles), at the smallest capacity whose fill keeps the last
    worker within it."""
    tiles = [-(-int(L) // tile) for L in lens]
    W = workers

    def fill(cap, emit):
        segs = []
        w, used, cum = 0, False, 0
        for b, n_b in enumerate(tiles):
            if n_b == 0:
                if used and w < W - 1 and cum + ovh > cap:
                    w, used, cum = w + 1, False, 0
                segs.append([w, b, 0, 0])
                used = True
                cum += ovh
                continue
            t = 0
            while t < n_b:
                left = n_b - t
                room = cap - cum - ovh
                if w == W - 1 or left <= room:
                    n = left
                elif room >= min_split and left - min_split >= min_split:
                    n = min(room, left - min_split)
                elif used:
                    w, used, cum = w + 1, False, 0
                    continue
                else:
                    n = min(left, min_split)
                    if left - n < min_split:
                        n = left
                segs.append([w, b, t, t + n])
                used = True
                cum += n + ovh
                t += n
        return segs, (cum if w == W - 1 else 0)

    total = sum(n + ovh for n in tiles)
    lo, hi = max(1, -(-total // W)), total + ovh * W + min_split
    while lo < hi:
        mid = (lo + hi) // 2
        if fill(mid, False)[1] <= mid:
            hi = mid
        else:
            lo = mid + 1
    segs, _ = fill(lo, True)
    cap = lo
    counts = {}
    for s in segs:
        counts[s[1]] = counts.get(s[1], 0) + 1
    slot, base = 0, {}
    for b in range(len(lens)):
        if counts.get(b, 0) >= 2:
            base[b] = slot
            slot += counts[b]
    seen = {}
    for s in segs:
        b = s[1]
        if b in base:
            s.append(base[b] + seen.get(b, 0))
            seen[b] = seen.get(b, 0) + 1
        else:
            s.append(-1)
    return np.array(segs, dtype=np.int32).reshape(-1, 5), slot, cap


def check_invariants(segs, lens, workers, tile, slots):
    tiles = [-(-int(L) // tile) for L in lens]
    assert np.all(np.diff(segs[:, 0]) >= 0), "segments not in worker order"
    assert segs[:, 0].min() >= 0 and segs[:, 0].max() < workers
    used_slots = []
    for b, n_b in enumerate(tiles):
        mine = segs[segs[:, 1] == b]
        assert len(mine) >= 1
        if n_b == 0:
            assert len(mine) == 1 and mine[0, 2] == 0 and mine[0, 3] == 0
        else:
            assert mine[0, 2] == 0 and mine[-1, 3] == n_b
            assert np.all(mine[1:, 2] == mine[:-1, 3]), "gap or overlap"
            assert np.all(mine[:, 3] > mine[:, 2]), "empty piece of a live request"
        if len(mine) == 1:
            assert mine[0, 4] == -1
        else:
            assert np.all(np.diff(mine[:, 4]) == 1) and mine[0, 4] >= 0
            used_slots.extend(mine[:, 4].tolist())
    assert sorted(used_slots) == list(range(slots))


def lens_of(name, seed=0):
    cfg = dict(W.CONFIGS[name])
    return W.draw_seq_lens(cfg, np.random.default_rng(seed))


CASES = [(n, s) for n in W.CONFIGS for s in (148, 152)] + [("dsv3", 2), ("fp8_kv", 16), ("tiny", 160)]


@pytest.mark.parametrize("name,sms", CASES)
def test_plan_matches_rule(name, sms):
    tile, ovh, mn = B.mla_planner_constants()
    assert (tile, ovh, mn) == (64, 3, 4)
    cfg = W.CONFIGS[name]
    lens = lens_of(name)
    p = B.mla_decode_plan(lens, cfg["page_size"], cfg["num_heads"], cfg["q_len"], num_sms=sms)
    segs = p.segments()
    want, slots, cap = plan_rule(lens, sms // 2, tile, ovh, mn)
    assert np.array_equal(segs, want)
    assert p.num_partial_slots == slots
    check_invariants(segs, lens, sms // 2, tile, slots)
    rows = cfg["num_heads"] * cfg["q_len"]
    if slots:
        o = slots * rows * 512 * 2
        want_ws = -(-o // 256) * 256 + -(-(slots * rows * 4) // 256) * 256
    else:
        want_ws = 0
    assert p.workspace_bytes == want_ws
    # balance: no worker exceeds the capacity (an empty worker's minimum
    # piece aside), and the capacity is within a couple of pieces of the mean
    loads = np.zeros(sms // 2, dtype=np.int64)
    for w_, b, t0, t1, _ in segs:
        loads[w_] += (t1 - t0) + ovh
    assert loads.max(initial=0) <= cap + mn, (loads.max(), cap)
    mean = -(-sum(-(-int(L) // tile) + ovh for L in lens) // (sms // 2))
    assert cap <= mean + 2 * (mn + ovh) or len(lens) < sms // 2, (cap, mean)


def test_plan_fuzz():
    rng = np.random.default_rng(123)
    tile, ovh, mn = B.mla_planner_constants()
    for it in range(300):
        bsz = int(rng.integers(1, 300))
        kind = it % 3
        if kind == 0:
            lens = rng.integers(0, 5000, size=bsz)
        elif kind == 1:
            lens = np.where(rng.random(bsz) < 0.3, 0, rng.integers(1, 200, size=bsz))
        else:
            lens = (rng.lognormal(8, 1.5, size=bsz)).astype(np.int64).clip(0, 200000)
        sms = int(rng.integers(2, 257))
        p = B.mla_decode_plan(lens.astype(np.int32), 64, 16, 1, num_sms=sms)
        segs = p.segments()
        want, slots, _ = plan_rule(lens, min(sms // 2, 128), tile, ovh, mn)
        assert np.array_equal(segs, want), (it, bsz, sms)
        check_invariants(segs, lens, min(sms // 2, 128), tile, slots)


@pytest.mark.parametrize("bad", [
    dict(page_size=16), dict(page_size=128), dict(num_heads=0), dict(q_len=0),
    dict(num_heads=128, q_len=2), dict(num_heads=129), dict(num_sms=1), dict(num_sms=-1),
])
def test_plan_rejects(bad):
    kw = dict(page_size=64, num_heads=16, q_len=1, num_sms=148)
    kw.update(bad)
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan([10, 20], **kw)
    assert ei.value.code == B.MLA_ERR_ARG


def test_plan_rejects_negative_length():
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan([10, -1], 64, 16, 1, num_sms=148)
    assert ei.value.code == B.MLA_ERR_ARG


def test_plan_single_worker_takes_everything():
    p = B.mla_decode_plan([100, 0, 5000], 64, 16, 1, num_sms=2)
    segs = p.segments()
    assert np.all(segs[:, 0] == 0) and np.all(segs[:, 4] == -1)
    assert p.workspace_bytes == 0
