"""GPU: mla_decode_host_io, the decode whose per-step inputs come from and
whose results go to host memory.  Its device input buffers are filled with
NaN first, so only the inputs it copies in can make the output right; the
host results must be exactly the bits of mla_decode on the same inputs
(the same plan runs the same kernels), and within the oracle's tolerance."""

import numpy as np
import pytest
import torch

from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

from test_zz_no_alloc import check_oracle, same_bits

pytestmark = pytest.mark.gpu


def host_copies(db, pinned):
    def h(t):
        x = t.cpu()
        return x.pin_memory() if pinned else x
    ins = [h(db.q_nope), h(db.q_pe), h(db.block_table), h(db.seq_lens)]
    outs = [torch.full(db.out.shape, float("nan"), dtype=db.out.dtype),
            torch.full(db.lse.shape, float("nan"), dtype=db.lse.dtype)]
    if pinned:
        outs = [o.pin_memory() for o in outs]
    return ins, outs


def spoil_inputs(db):
    db.q_nope.fill_(float("nan"))
    db.q_pe.fill_(float("nan"))
    db.block_table.fill_(-1)
    db.seq_lens.fill_(0)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_io_matches_device_decode(pinned):
    w = W.make_workload("dsv3", seed=41, batch=16)
    db = R.upload(w)
    ref = tuple(t.clone() for t in R.decode(db))
    (hq, hp, hbt, hsl), (ho, hl) = host_copies(db, pinned)
    spoil_inputs(db)
    stream = torch.cuda.current_stream()
    B.mla_decode_host_io(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                         w.scale, w.k_scale, db.out, db.lse, db.workspace, hq, hp, hbt, hsl, ho, hl, stream)
    stream.synchronize()
    assert B.mla_decode_device_error() == 0
    assert same_bits(ref, (ho.cuda(), hl.cuda()))
    check_oracle(w, ho, hl)


def test_host_io_two_streams_overlapped():
    """Two buffer sets on two streams, alternating, several steps in flight:
    each step's host results are its own decode's bits."""
    ws = [W.make_workload("fp8_kv", seed=50 + i, batch=24) for i in range(2)]
    dbs = [R.upload(w) for w in ws]
    refs = [tuple(t.clone() for t in R.decode(db)) for db in dbs]
    host = [host_copies(db, True) for db in dbs]
    for db in dbs:
        spoil_inputs(db)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for k in range(6):
        i = k & 1
        if k >= 2:
            streams[i].synchronize()
            assert same_bits(refs[i], (host[i][1][0].cuda(), host[i][1][1].cuda()))
            host[i][1][0].fill_(float("nan"))
            host[i][1][1].fill_(float("nan"))
        db, w = dbs[i], ws[i]
        (hq, hp, hbt, hsl), (ho, hl) = host[i]
        B.mla_decode_host_io(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                             w.scale, w.k_scale, db.out, db.lse, db.workspace, hq, hp, hbt, hsl, ho, hl, streams[i])
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    for i in range(2):
        assert same_bits(refs[i], (host[i][1][0].cuda(), host[i][1][1].cuda()))
