"""Device-side planner: its rule restated in Python (used bit for bit by the
GPU tests, which read back the schedule the planner kernel built), the
invariants any valid schedule meets checked on the restatement over many
length sets, and the host side of device plans (arguments, workspace size)."""

import numpy as np
import pytest

from paged_mla_decode_08_gb300 import binding as B

from test_plan import check_invariants

TILE, OVH, MIN = 64, 3, 4  # the library's planner constants (checked in test_abi_host)


def device_plan_rule(lens, workers, cap_tokens=1 << 30):
    """The planner kernel's rule: tiles n_b (lengths clamped to cap_tokens),
    cost n_b + OVH, exclusive prefix P_b, cap = max(ceil(total / W), MIN); request b's
    tiles occupy cost [P_b, P_b + n_b) and are cut at multiples of cap,
    pieces of any length; a request without tiles is one empty segment on
    the worker holding P_b.
    Returns (segments [n, 5], slots, jobs [(req, slot_begin, nsplit)])."""
    n = [(-(-min(max(int(L), 0), cap_tokens) // TILE)) for L in lens]
    total = sum(x + OVH for x in n)
    cap = max(-(-total // workers), MIN)
    segs, jobs = [], []
    p, slot = 0, 0
    for b, nb in enumerate(n):
        if nb == 0:
            segs.append([min(p // cap, workers - 1), b, 0, 0, -1])
        else:
            w0, w1 = p // cap, min((p + nb - 1) // cap, workers - 1)
            w0 = min(w0, w1)
            ns = w1 - w0 + 1
            for i in range(ns):
                w = w0 + i
                t0 = 0 if i == 0 else w * cap - p
                t1 = nb if i == ns - 1 else (w + 1) * cap - p
                segs.append([w, b, t0, t1, slot + i if ns > 1 else -1])
            if ns > 1:
                jobs.append((b, slot, ns))
                slot += ns
        p += nb + OVH
    return np.array(segs, dtype=np.int32).reshape(-1, 5), slot, jobs


def test_rule_constants_are_the_librarys():
    assert B.mla_planner_constants() == (TILE, OVH, MIN)


def random_lens(rng, kind, bsz):
    if kind == 0:
        return rng.integers(0, 5000, size=bsz)
    if kind == 1:
        return np.where(rng.random(bsz) < 0.3, 0, rng.integers(1, 200, size=bsz))
    if kind == 2:
        return rng.lognormal(8, 1.5, size=bsz).astype(np.int64).clip(0, 200000)
    return np.ones(bsz, dtype=np.int64)  # padded graph rows: the seq_len fill value 1


def test_rule_invariants_fuzz():
    rng = np.random.default_rng(7)
    for it in range(400):
        bsz = int(rng.integers(1, 1794 if it % 20 == 0 else 300))
        lens = random_lens(rng, it % 4, bsz)
        W = int(rng.integers(1, 129))
        segs, slots, jobs = device_plan_rule(lens, W)
        check_invariants(segs, lens, W, TILE, slots)
        assert len(segs) <= bsz + W - 1
        assert len(jobs) <= max(W - 1, 0) and slots <= 2 * max(W - 1, 0)
        for b, nsplit in [(j[0], j[2]) for j in jobs]:
            mine = segs[segs[:, 1] == b]
            assert len(mine) == nsplit and np.all(mine[:, 3] > mine[:, 2])


def test_rule_balance():
    """Each worker's load stays within the capacity plus the overhead of the
    two split pieces it may hold beyond what the cost stream charged."""
    rng = np.random.default_rng(8)
    for it in range(100):
        lens = random_lens(rng, it % 3, int(rng.integers(1, 400)))
        W = int(rng.integers(2, 129))
        segs, _, _ = device_plan_rule(lens, W)
        n = [-(-int(L) // TILE) for L in lens]
        cap = max(-(-sum(x + OVH for x in n) // W), MIN)
        load = np.zeros(W, dtype=np.int64)
        for w, b, t0, t1, _ in segs:
            load[w] += t1 - t0 + OVH
        assert load.max() <= cap + 2 * OVH, (load.max(), cap)


def test_rule_clamps_like_the_decode():
    segs, _, _ = device_plan_rule([10 ** 6, 100], 4, cap_tokens=64 * 10)
    assert segs[segs[:, 1] == 0][:, 3].max() == 10


@pytest.mark.parametrize("bad", [dict(batch=0), dict(batch=1794), dict(page_size=16), dict(num_heads=0),
                                 dict(num_heads=64, q_len=3), dict(num_sms=1)])
def test_device_plan_rejects(bad):
    kw = dict(batch=8, page_size=64, num_heads=16, q_len=1, num_sms=148)
    kw.update(bad)
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan_device(**kw)
    assert ei.value.code == B.MLA_ERR_ARG


@pytest.mark.parametrize("sms,heads,q", [(148, 128, 1), (152, 16, 4), (2, 128, 1), (256, 8, 2)])
def test_device_plan_workspace(sms, heads, q):
    p = B.mla_decode_plan_device(64, 64, heads, q, num_sms=sms)
    assert p.is_device and p.num_workers == min(sms // 2, 128)
    W = p.num_workers
    slots = 2 * (W - 1)
    rows = heads * q
    sched = -(-(8 + 129 * 4 + 1920 * 16) // 256) * 256
    part = -(-(sched + 16 + 128 * 16) // 256) * 256
    o = -(-(slots * rows * 512 * 2) // 256) * 256
    lse = -(-(slots * rows * 4) // 256) * 256
    assert p.workspace_bytes == part + o + lse
    assert p.num_partial_slots == slots
    assert len(p.segments()) == 0
    assert not B.mla_decode_plan([10], 64, 16, 1, num_sms=148).is_device
