"""GPU: decodes planned on the device (mla_decode_plan_device).  The schedule
the planner kernel built is read back and compared bit for bit with the
rule's Python restatement; the decode is compared with the float64 oracle;
one CUDA graph is replayed for unrelated lengths."""

import numpy as np
import pytest
import torch

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

from test_parity import check, oracle
from test_plan_device import device_plan_rule, random_lens

pytestmark = pytest.mark.gpu


def upload_device_planned(w, num_sms=0):
    """runner.upload with the host plan swapped for a device plan."""
    db = R.upload(w, num_sms=num_sms)
    db.plan = B.mla_decode_plan_device(w.batch, w.page_size, w.num_heads, w.q_len, num_sms)
    db.workspace = torch.empty(db.plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    db.workspace.random_(0, 256)  # no initial contents needed
    return db


def run(db):
    out, lse = R.decode(db)
    torch.cuda.synchronize()
    err = B.mla_decode_device_error()
    if err:
        # say whether the schedule the planner left behind is the rule's
        got = db.plan.device_segments(db.workspace)
        lens = db.seq_lens.cpu().numpy()
        want, _, _ = device_plan_rule(lens, db.plan.num_workers,
                                      cap_tokens=db.block_table.shape[1] * db.w.page_size)
        same = got.shape == want.shape and np.array_equal(got, want)
        raise AssertionError(f"kernel error word {err:#x}; device schedule matches the rule: {same}")
    return out, lse


def expect_schedule(db, lens):
    w = db.w
    got = db.plan.device_segments(db.workspace)
    want, _, _ = device_plan_rule(lens, db.plan.num_workers, cap_tokens=db.block_table.shape[1] * w.page_size)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_configs_against_oracle(name):
    w = W.make_workload(name, seed=0)
    db = upload_device_planned(w)
    out, lse = run(db)
    expect_schedule(db, w.seq_lens)
    check(w, out, lse, *oracle(w))


def test_repeatable_with_garbage_workspace():
    """Repeated device-planned decodes are bit-identical (the rule is fixed)."""
    w = W.make_workload("long_skewed", seed=1)
    db = upload_device_planned(w)
    o1, l1 = (t.clone() for t in run(db))
    db.workspace.fill_(255)
    o2, l2 = run(db)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    check(w, o2, l2, *oracle(w))


def test_schedule_fuzz_matches_rule():
    """Many length sets (zero, short, skewed, all-ones graph padding) on one
    plan: the device-built schedule equals the restated rule each time."""
    rng = np.random.default_rng(21)
    w = W.make_workload("tiny", seed=2, seq_lens=[1] * 300, pool_pages=64, bt_extra_cols=200)
    db = upload_device_planned(w)
    for it in range(24):
        lens = random_lens(rng, it % 4, 300).clip(0, 64 * 201).astype(np.int32)
        db.seq_lens.copy_(torch.from_numpy(lens))
        R.decode(db)
        torch.cuda.synchronize()
        expect_schedule(db, lens)


def test_ragged_with_device_plan():
    w = W.make_ragged_workload("draft_extend", seed=3)
    db = R.upload(w)
    db.plan = B.mla_decode_plan_device(w.batch, w.page_size, w.num_heads, w.q_len)
    db.workspace = torch.empty(db.plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out, lse = run(db)
    check(w, out, lse, *O.mla_decode_ragged(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table,
                                             w.seq_lens, w.cu_seqlens_q, w.page_size, w.scale, w.k_scale))


def test_one_graph_any_lengths():
    """Captured once; replayed with lengths the capture never saw, longer and
    shorter, including the padded-row fill value 1 and empty requests."""
    b, page = 12, 64
    stride = 200  # pages per block-table row: up to 12800 keys
    w = W.make_workload("dsv3", seed=4, seq_lens=[stride * page] * b, pool_pages=b * stride)
    db = upload_device_planned(w)
    run(db)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            R.decode(db, s)
    rng = np.random.default_rng(5)
    cases = [np.full(b, 1), rng.integers(0, stride * page + 1, size=b), np.array([12800, 0, 1, 1, 1, 1, 5000, 0,
                                                                                   64, 65, 3000, 12799])]
    for lens in cases:
        lens = lens.astype(np.int32)
        db.seq_lens.copy_(torch.from_numpy(lens))
        db.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0
        expect_schedule(db, lens)
        ref_out, ref_lse = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, lens,
                                        w.q_len, w.page_size, w.scale, w.k_scale)
        check(w, db.out, db.lse, ref_out, ref_lse)


def test_noalloc_with_device_plan():
    """Small rows fit the built-in scratch: the device plan needs no caller
    workspace there either."""
    w = W.make_workload("spec_q4", seed=6, batch=16, num_heads=4)
    db = R.upload(w)
    plan = B.mla_decode_plan_device(w.batch, w.page_size, w.num_heads, w.q_len)
    assert plan.workspace_bytes <= B.MLA_NOALLOC_SCRATCH_BYTES
    B.mla_decode_noalloc(plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens, w.scale,
                         w.k_scale, db.out, db.lse)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    check(w, db.out, db.lse, *oracle(w))


@pytest.mark.parametrize("name", ["spec_q4", "draft_extend"])
def test_padding_rows_never_stall_the_pair(name):
    """64 live query rows of 128: the warps owning only padding rows must not
    wait on the pair's exchange barriers (they could fall two phases behind
    and hang on an aliased parity).  Before the fix these device-planned
    decodes timed out in 40-70 % of runs; 20 in a row must all be clean."""
    w = W.make_ragged_workload(name, seed=3) if name == "draft_extend" else W.make_workload(name, seed=0)
    db = R.upload(w)
    db.plan = B.mla_decode_plan_device(w.batch, w.page_size, w.num_heads, w.q_len)
    db.workspace = torch.empty(db.plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    for _ in range(20):
        R.decode(db)
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0
    if db.cu_seqlens_q is None:
        check(w, db.out, db.lse, *oracle(w))
