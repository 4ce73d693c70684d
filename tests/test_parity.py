"""GPU parity: the CUDA path through the C ABI against the float64 oracle,
element by element, on seeded inputs.

Tolerances (fixed for this decode): bf16 cache
``max|out - ref| <= 1e-2 * max|ref| + 1e-3`` and ``|lse - ref| <= 2e-3``;
e4m3 cache ``max|out - ref| <= 5e-2 * max|ref|`` (lse: 2e-3, the dequantised
values are exact in bf16); rows with no
visible key exactly 0 and -inf.
"""

import numpy as np
import pytest
import torch

from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from paged_mla_decode_08_gb300 import binding as B


def oracle(w, requests=None):
    return O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
                        w.q_len, w.page_size, w.scale, w.k_scale, requests=requests)


def check(w, out, lse, ref_out, ref_lse, rows=None):
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        out, lse, ref_out, ref_lse = out[rows], lse[rows], ref_out[rows], ref_lse[rows]
    empty = np.isneginf(ref_lse)
    assert np.all(np.isneginf(lse[empty])), "empty rows must give lse = -inf"
    assert np.all(out[empty] == 0.0), "empty rows must give out = 0"
    live = ~empty
    assert np.all(np.isfinite(lse[live])) and np.all(np.isfinite(out[live]))
    if not live.any():
        return 0.0, 0.0
    err = np.abs(out[live] - ref_out[live]).max()
    lerr = np.abs(lse[live] - ref_lse[live]).max()
    ref_max = np.abs(ref_out[live]).max()
    if w.kv_dtype == "bf16":
        assert err <= 1e-2 * ref_max + 1e-3, (err, ref_max)
        assert lerr <= 2e-3, lerr
    else:
        assert err <= 5e-2 * ref_max, (err, ref_max)
        assert lerr <= 2e-3, lerr
    return err, lerr


def run_gpu(w, **kw):
    db = R.upload(w, **kw)
    out, lse = R.decode(db)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0, "a bounded wait timed out inside the kernel"
    return db, out, lse


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_config_full(name):
    """Every benchmark workload at full size, in the benchmark's launch
    configuration (plan for the device's SM count), against the oracle."""
    w = W.make_workload(name, seed=0)
    _, out, lse = run_gpu(w)
    ref_out, ref_lse = oracle(w)
    check(w, out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("name", ["tiny", "spec_q4"])
def test_config_other_seeds(name, seed):
    w = W.make_workload(name, seed=seed, batch=8) if name == "spec_q4" else W.make_workload(name, seed=seed)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


@pytest.mark.parametrize("page", [32, 64])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_nan_in_unread_slots(page, kv_dtype):
    """Cache rows past seq_len and pages nobody owns hold NaN; block-table
    padding holds garbage ids; neither may reach the result."""
    lens = [1, 17, 63, 64, 65, 100, 127, 128, 129, 700, 1000, 0]
    w = W.make_workload("tiny", seed=3, fill="nan", seq_lens=lens, page_size=page, num_heads=16,
                        kv_dtype=kv_dtype, k_scale=0.5 if kv_dtype == "e4m3" else 1.0,
                        pool_pages=80, bt_pad_value=2 ** 30, bt_extra_cols=3)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


@pytest.mark.parametrize("pad", [-1, 0])
def test_padding_values(pad):
    w = W.make_workload("dsv3", seed=4, seq_lens=[1024, 77, 3000, 5], bt_pad_value=pad, bt_extra_cols=2)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


def test_single_key_rows_equal_cache_row():
    """seq_len = 1 (the fill value of padded CUDA-graph rows): out is the row's
    latent columns, rounded to bf16, lse the single score."""
    w = W.make_workload("dsv3", seed=5, seq_lens=[1, 1, 1])
    _, out, lse = run_gpu(w)
    ref_out, ref_lse = oracle(w)
    check(w, out, lse, ref_out, ref_lse)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    for b in range(3):
        row = w.kv_bits[w.block_table[b, 0], 0, :512]
        assert np.array_equal(got[b], np.broadcast_to(row, got[b].shape))


def test_all_empty_batch():
    w = W.make_workload("tiny", seed=6, seq_lens=[0, 0, 0])
    _, out, lse = run_gpu(w)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("q_len", [2, 3, 4])
def test_causal_short_requests(q_len):
    """q_len > 1 with requests shorter than q_len: early query rows see no key."""
    lens = [0, 1, 2, 3, 4, 5, 64, 65, 300]
    w = W.make_workload("spec_q4", seed=7, seq_lens=lens, q_len=q_len, num_heads=8)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


def test_heads_times_qlen_128():
    w = W.make_workload("spec_q4", seed=8, seq_lens=[3000, 1500, 20, 4100], q_len=2, num_heads=64)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


@pytest.mark.parametrize("heads", [1, 3, 100])
def test_odd_head_counts(heads):
    w = W.make_workload("dsv3", seed=9, seq_lens=[2000, 640, 33], num_heads=heads)
    _, out, lse = run_gpu(w)
    check(w, out, lse, *oracle(w))


def test_plan_from_upper_bounds():
    """Planned with longer lengths than the device seq_lens: the decode masks
    with the device lengths and only skips work."""
    w = W.make_workload("dsv3", seed=10, seq_lens=[2000, 1000, 300, 0, 64])
    upper = np.array([4096, 1500, 2000, 200, 64], dtype=np.int32)
    w2 = W.make_workload("dsv3", seed=10, seq_lens=[2000, 1000, 300, 0, 64], bt_extra_cols=40)
    _, out, lse = run_gpu(w2, plan_seq_lens=upper)
    check(w2, out, lse, *oracle(w))


def test_garbage_workspace_and_repeat_determinism():
    """The workspace needs no initial contents, and repeated calls give
    bit-identical results."""
    w = W.make_workload("long_skewed", seed=11, seq_lens=[40000, 9000, 17, 0])
    db = R.upload(w)
    assert db.workspace is not None
    db.workspace.random_(0, 256)
    out1, lse1 = (t.clone() for t in R.decode(db))
    db.workspace.fill_(255)  # NaN patterns everywhere
    out2, lse2 = R.decode(db)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    check(w, out2, lse2, *oracle(w))


def test_main_then_combine_equals_decode():
    w = W.make_workload("dsv3", seed=12, seq_lens=[4096, 4000, 3000, 100])
    db = R.upload(w)
    R.decode(db)
    o1, l1 = db.out.clone(), db.lse.clone()
    db.out.zero_()
    db.lse.zero_()
    R.decode_main(db)
    R.decode_combine(db)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), db.out.view(torch.int16)) and torch.equal(l1, db.lse)


def test_side_stream():
    w = W.make_workload("tiny", seed=13)
    db = R.upload(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.decode(db)
    s.synchronize()
    check(w, db.out, db.lse, *oracle(w))


def test_cuda_graph_replay_with_new_lengths():
    """Graph-captured decode: planned once from upper-bound lengths, captured
    (main kernel + combine, with its programmatic-dependent edge) into a CUDA
    graph, then replayed after the device lengths change; each replay must
    match the oracle for the lengths it ran with."""
    lens = np.array([2000, 1000, 300, 5, 64, 1500], dtype=np.int32)
    upper = np.array([2600, 1600, 900, 700, 700, 2100], dtype=np.int32)
    w = W.make_workload("dsv3", seed=14, seq_lens=list(lens), bt_extra_cols=12)
    db = R.upload(w, plan_seq_lens=upper)
    R.decode(db)  # warm: one-time host work (tensor-map encoder lookup) outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.mla_decode(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                         w.scale, w.k_scale, db.out, db.lse, db.workspace, None, s)
    for new_lens in (lens, np.array([1999, 63, 1, 0, 64, 2100], dtype=np.int32)):
        db.seq_lens.copy_(torch.from_numpy(new_lens))
        db.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert B.mla_decode_device_error() == 0
        ref_out, ref_lse = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table,
                                        new_lens, w.q_len, w.page_size, w.scale, w.k_scale)
        check(w, db.out, db.lse, ref_out, ref_lse)


def test_wide_batch_large_schedule():
    """700 short requests: more segments than the small schedule capacity,
    so the launch takes the large-capacity kernel instantiation."""
    lens = np.random.default_rng(15).integers(0, 200, size=700)
    w = W.make_workload("tiny", seed=15, seq_lens=list(lens), num_heads=16, pool_pages=4096)
    db, out, lse = run_gpu(w)
    assert len(db.plan.segments()) > 448
    check(w, out, lse, *oracle(w))


# ---------------------------------------------------------------- non-finite and large scores

def check_nan_rows(w, out, lse, ref_out, ref_lse):
    """Rows the definition makes NaN are NaN everywhere (out and lse); every
    other row is checked with the usual tolerances."""
    got = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    nan_rows = np.isnan(ref_lse)
    assert nan_rows.any()
    assert np.all(np.isnan(got_lse[nan_rows])), "a NaN score must make the row's lse NaN"
    assert np.all(np.isnan(got[nan_rows])), "a NaN score must make the row's output NaN"
    keep = ~nan_rows.any(axis=1)  # tokens with no NaN row
    check(w, out, lse, ref_out, ref_lse, rows=keep)


# NaN bit patterns: quiet, negative quiet, and a payload in the lowest bit
BF16_NANS = {"qnan": 0x7FC0, "neg_qnan": 0xFFC0, "low_payload": 0x7F81}
E4M3_NANS = {"qnan": 0x7F, "neg_qnan": 0xFF, "low_payload": 0x7F}  # e4m3fn has one NaN code per sign


@pytest.mark.parametrize("pattern", list(BF16_NANS))
@pytest.mark.parametrize("where", ["latent", "rope", "query"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_nan_in_visible_row(pattern, where, kv_dtype):
    """One NaN in a visible cache row (latent or rope column) of a request
    split over many workers, or in one head's query: the rows that read it
    are NaN, as the float64 definition gives, on both CTAs of the pair (the
    24-bit score code keeps the tensor core's NaN results NaN) and through the
    LSE combine; every other row matches the oracle.  NaN of either sign and
    with its payload in the lowest bit all behave the same."""
    lens = [3000, 9000, 500, 0]
    w = W.make_workload("dsv3", seed=21, seq_lens=lens, num_heads=128, kv_dtype=kv_dtype,
                        k_scale=0.5 if kv_dtype == "e4m3" else 1.0)
    nan = BF16_NANS[pattern] if kv_dtype == "bf16" else E4M3_NANS[pattern]
    key = 7000  # request 1: in a later split of the request
    page, off = w.block_table[1, key // w.page_size], key % w.page_size
    if where == "latent":
        w.kv_bits[page, off, 100] = nan
    elif where == "rope":
        w.kv_bits[page, off, 530] = nan
    else:
        w.q_nope_bits[2, 17, 5] = BF16_NANS[pattern]  # request 2, head 17 only
    db, out, lse = run_gpu(w)
    assert db.plan.num_partial_slots > 0
    ref_out, ref_lse = oracle(w)
    check_nan_rows(w, out, lse, ref_out, ref_lse)
    if where == "query":
        assert np.isnan(lse.cpu().numpy()).sum() == 1
    else:
        assert np.all(np.isnan(lse.cpu().numpy()[1]))


def _scaled_query(w, factor, seed):
    """Replace the query with bf16 of N(0, factor^2): sharp attention with
    partial logits in the tens to about a hundred (natural-log units)."""
    rng = np.random.default_rng(seed)
    w.q_nope_bits = W.f32_to_bf16_bits(rng.standard_normal(w.q_nope_bits.shape).astype(np.float32) * factor)
    w.q_pe_bits = W.f32_to_bf16_bits(rng.standard_normal(w.q_pe_bits.shape).astype(np.float32) * factor)
    return w


@pytest.mark.parametrize("factor", [8.0, 16.0])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_large_logits_scaled_query(factor, kv_dtype):
    """Queries 8x and 16x the benchmark's: logits reach ~100, the lazy
    rescale fires and the pair's 24-bit partial scores carry large values;
    requests are split, so the combine merges lse values far apart."""
    lens = [4096, 20000, 700, 64, 1, 3000, 12000, 2500]
    w = W.make_workload("dsv3", seed=22, seq_lens=lens, kv_dtype=kv_dtype,
                        k_scale=0.5 if kv_dtype == "e4m3" else 1.0)
    _scaled_query(w, factor, seed=23)
    ref_out, ref_lse = oracle(w)
    # the case really is sharp: scores far beyond the unit-variance data
    assert np.nanmax(ref_lse) > 40.0
    db, out, lse = run_gpu(w)
    assert db.plan.num_partial_slots > 0
    check(w, out, lse, ref_out, ref_lse)


def _query_direction(w, b):
    """Unit 576-vector along the sum of request b's query heads (float64): a
    cache row along it scores high for nearly every head."""
    t = b * w.q_len
    u = np.concatenate([O.decode_bf16(w.q_nope_bits[t]).sum(axis=0), O.decode_bf16(w.q_pe_bits[t]).sum(axis=0)])
    return u / np.linalg.norm(u)


def _set_row(w, b, key, values):
    page, off = w.block_table[b, key // w.page_size], key % w.page_size
    if w.kv_dtype == "bf16":
        w.kv_bits[page, off] = W.f32_to_bf16_bits(values.astype(np.float32))
    else:
        w.kv_bits[page, off] = W.f32_to_e4m3fn_bits((values / w.k_scale).astype(np.float32))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_spike_keys_force_rescales(kv_dtype):
    """Keys whose scores jump far above everything before them, placed in
    the middle of a segment, on the first key of every split piece, and on a
    request's last key; plus a request whose whole first tile scores ~40
    below the rest.  The running maximum then moves by far more than the
    lazy-rescale threshold (2^8) mid-segment and across split boundaries."""
    lens = [12000, 6000, 3000, 2100]
    w = W.make_workload("dsv3", seed=24, seq_lens=lens, kv_dtype=kv_dtype,
                        k_scale=0.5 if kv_dtype == "e4m3" else 1.0)
    plan = B.mla_decode_plan(w.seq_lens, w.page_size, w.num_heads, w.q_len)
    segs = plan.segments()  # (worker, request, tile_begin, tile_end, slot)
    for b in range(3):
        d = _query_direction(w, b)
        starts = sorted({int(s[2]) * 64 for s in segs if s[1] == b and s[2] > 0})
        assert b > 1 or starts, "the long requests must be split"
        # alpha / scale sets the typical spike logit (natural-log units)
        spikes = [(lens[b] // 3, 15.0), (lens[b] // 2 + 5, 30.0), (lens[b] - 1, 45.0)]
        spikes += [(k, 12.0 + 8.0 * (i % 4)) for i, k in enumerate(starts)]
        for key, logit in spikes:
            _set_row(w, b, key, d * (logit / (w.scale * 2.1)))
    # request 3: its first tile far below everything after it
    d = _query_direction(w, 3)
    for key in range(64):
        _set_row(w, 3, key, -d * (40.0 / (w.scale * 2.1)))
    ref_out, ref_lse = oracle(w)
    assert 40.0 < np.nanmax(ref_lse) < 130.0  # sharp, within the exchange's precision range
    db, out, lse = run_gpu(w)
    check(w, out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("lens,widest", [
    ([4096] * 24, (2, 4)),      # splits of at most 4: four partials per load round
    ([4096] * 10, (5, 8)),      # 5-8: eight per round
    ([60000, 500, 33], (9, 128)),  # many: sixteen per round
])
def test_combine_group_sizes(lens, widest):
    """The combine loads the partials of 4, 8 or 16 splits per round, chosen
    for the widest split of the launch (past 8 splits a CTA also takes a
    sixteenth of the row instead of a quarter); each width merges like the
    oracle."""
    w = W.make_workload("dsv3", seed=25, seq_lens=lens)
    db, out, lse = run_gpu(w)
    segs = db.plan.segments()
    most = max(int((segs[:, 1] == b).sum()) for b in range(len(lens)))
    assert widest[0] <= most <= widest[1], most
    check(w, out, lse, *oracle(w))
