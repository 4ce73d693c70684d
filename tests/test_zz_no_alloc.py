"""mla_decode_noalloc, the entry point for callers that cannot allocate device
memory (it keeps the split partials in the library's built-in scratch array
instead of a caller workspace).  Checked through the C ABI against mla_decode
with a caller workspace, within the parity tolerances, on two calls in a row
(the second one reusing the scratch left by the first).  The file name makes
pytest collect it last."""

import numpy as np
import pytest
import torch

from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def close(a_out, a_lse, b_out, b_lse):
    a = a_out.float().cpu().numpy().astype(np.float64)
    b = b_out.float().cpu().numpy().astype(np.float64)
    la = a_lse.cpu().numpy().astype(np.float64)
    lb = b_lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(la)
    assert np.array_equal(empty, np.isneginf(lb))
    assert np.all(b[empty] == 0)
    live = ~empty
    ref_max = np.abs(a[live]).max()
    assert np.abs(a[live] - b[live]).max() <= 1e-2 * ref_max + 1e-3
    assert np.abs(la[live] - lb[live]).max() <= 2e-3


def noalloc(db):
    out = torch.full_like(db.out, float("nan"))
    lse = torch.full_like(db.lse, float("nan"))
    B.mla_decode_noalloc(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                         db.w.scale, db.w.k_scale, out, lse)
    return out, lse


def test_noalloc_matches_workspace_decode_twice():
    # two different split batches, one after the other
    wa = W.make_workload("dsv3", seed=31, batch=16)
    wb = W.make_workload("fp8_kv", seed=32, batch=24)
    dba, dbb = R.upload(wa), R.upload(wb)
    for db in (dba, dbb):
        assert 0 < db.plan.workspace_bytes <= B.MLA_NOALLOC_SCRATCH_BYTES
        assert db.plan.num_partial_slots > 0  # the scratch really is used
    ref_a = tuple(t.clone() for t in R.decode(dba))
    ref_b = tuple(t.clone() for t in R.decode(dbb))
    got_a = noalloc(dba)
    got_b = noalloc(dbb)
    torch.cuda.synchronize()
    close(*ref_a, *got_a)
    close(*ref_b, *got_b)


def test_noalloc_rejects_plan_larger_than_scratch():
    lens = np.full(256, 8192, dtype=np.int32)
    plan = B.mla_decode_plan(lens, 64, 128, 1, num_sms=152)
    assert plan.workspace_bytes > B.MLA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((256, 128, 512), dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros((256, 128, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((4, 64, 576), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((256, 128), dtype=torch.int32, device="cuda")
    sl = torch.from_numpy(lens).cuda()
    out = torch.empty_like(q)
    lse = torch.empty((256, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_noalloc(plan, q, qp, kv, B.MLA_KV_BF16, bt, sl, 0.07, 1.0, out, lse)
    assert ei.value.code == B.MLA_ERR_WORKSPACE
