"""mla_decode_noalloc, the decode for callers that cannot allocate device
memory -- code that is handed only its inputs and outputs, such as a plugin
running under a host framework's own memory manager, or an allocation-free
serving loop.  It keeps the split partials in the library's built-in scratch
array instead of a caller workspace.

Checked through the C ABI, after the scratch has been filled with NaN
partials (a no-allocation decode of an all-NaN query over a batch with many
split requests): three calls in a row -- batch A, batch B, then batch A
again -- must each give exactly the bits of mla_decode with a caller
workspace (the same plan runs the same kernels), and stay within the parity
tolerances of the float64 oracle.  The third call shows that the slots batch
B left behind are rewritten before they are read.  The file name makes
pytest collect it last."""

import numpy as np
import pytest
import torch

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def same_bits(a, b):
    (ao, al), (bo, bl) = a, b
    return torch.equal(ao.view(torch.int16), bo.view(torch.int16)) and torch.equal(al.view(torch.int32),
                                                                                  bl.view(torch.int32))


def check_oracle(w, out, lse):
    ref_out, ref_lse = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
                                    w.q_len, w.page_size, w.scale, w.k_scale)
    got = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(ref_lse)
    assert np.all(np.isneginf(got_lse[empty])) and np.all(got[empty] == 0)
    live = ~empty
    ref_max = np.abs(ref_out[live]).max()
    err = np.abs(got[live] - ref_out[live]).max()
    if w.kv_dtype == "bf16":
        assert err <= 1e-2 * ref_max + 1e-3, (err, ref_max)
    else:
        assert err <= 5e-2 * ref_max, (err, ref_max)
    assert np.abs(got_lse[live] - ref_lse[live]).max() <= 2e-3


def noalloc(db):
    out = torch.full_like(db.out, float("nan"))
    lse = torch.full_like(db.lse, float("nan"))
    B.mla_decode_noalloc(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                         db.w.scale, db.w.k_scale, out, lse)
    return out, lse


def test_noalloc_matches_workspace_decode_after_nan_scratch():
    # NaN partials in every slot a split-heavy batch uses
    wn = W.make_workload("long_skewed", seed=30)
    wn.q_nope_bits[:] = 0x7FC0
    wn.q_pe_bits[:] = 0x7FC0
    dbn = R.upload(wn)
    wa = W.make_workload("dsv3", seed=31, batch=16)
    wb = W.make_workload("fp8_kv", seed=32, batch=24)
    dba, dbb = R.upload(wa), R.upload(wb)
    for db in (dba, dbb):
        assert 0 < db.plan.workspace_bytes <= B.MLA_NOALLOC_SCRATCH_BYTES
        assert 0 < db.plan.num_partial_slots <= dbn.plan.num_partial_slots  # the NaN slots cover them
    assert dbn.plan.workspace_bytes <= B.MLA_NOALLOC_SCRATCH_BYTES
    nan_out, _ = noalloc(dbn)
    torch.cuda.synchronize()
    assert torch.isnan(nan_out).all()

    ref_a = tuple(t.clone() for t in R.decode(dba))
    ref_b = tuple(t.clone() for t in R.decode(dbb))
    got_a = tuple(t.clone() for t in noalloc(dba))
    got_b = noalloc(dbb)
    again_a = noalloc(dba)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    assert same_bits(ref_a, got_a)
    assert same_bits(ref_b, got_b)
    assert same_bits(ref_a, again_a)
    check_oracle(wa, *got_a)
    check_oracle(wb, *got_b)


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
