"""GPU parity of the RoPE + quantisation + cache-write kernel against the
oracle, bit for bit (every output is a code or a bit pattern decided in the
same float32 arithmetic on both sides), then the written cache driving the
decode."""

import numpy as np
import pytest
import torch

from oracle import kv_write_ref as K
from oracle import mla_ref as O
from paged_mla_decode_08_gb300 import binding as B
from paged_mla_decode_08_gb300 import runner as R
from paged_mla_decode_08_gb300 import workloads as W

from test_kv_write_oracle import roformer_cache
from test_parity import check

pytestmark = pytest.mark.gpu


def bf16(rng, shape, scale=1.0):
    return W.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def dev16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def make_step(seed, t, h, page, kv_dtype, pool_pages=40, max_pos=4096, scale=1.0):
    rng = np.random.default_rng(seed)
    q_nope, q_rope = bf16(rng, (t, h, 512), scale), bf16(rng, (t, h, 64), scale)
    k_nope, k_rope = bf16(rng, (t, 512), scale), bf16(rng, (t, 64), scale)
    pos = rng.integers(0, max_pos, size=t).astype(np.int64)
    slots = rng.choice(pool_pages * page, size=t, replace=False).astype(np.int64)
    cs = roformer_cache(max_pos).astype(np.float32)
    if kv_dtype == "bf16":
        kv = rng.integers(0, 1 << 16, size=(pool_pages, page, 576)).astype(np.uint16)
    else:
        kv = rng.integers(0, 256, size=(pool_pages, page, 576)).astype(np.uint8)
    return dict(q_nope=q_nope, q_rope=q_rope, k_nope=k_nope, k_rope=k_rope, pos=pos, slots=slots, cs=cs, kv=kv)


def run_kernel(st, q_dtype, kv_dtype, neox, with_q=True):
    t, h = st["q_rope"].shape[:2]
    kv = torch.from_numpy(st["kv"].view(np.int16) if kv_dtype == "bf16" else st["kv"]).cuda()
    if q_dtype == B.MLA_Q_E4M3:
        q_out = torch.zeros((t, h, 576), dtype=torch.uint8, device="cuda")
    else:
        q_out = torch.zeros((t, h, 64), dtype=torch.int16, device="cuda")
    B.mla_rope_quantize_cache_write(
        dev16(st["q_nope"]) if with_q else None, dev16(st["q_rope"]) if with_q else None,
        q_out if with_q else None, q_dtype, dev16(st["k_nope"]), dev16(st["k_rope"]),
        torch.from_numpy(st["pos"]).cuda(), torch.from_numpy(st["cs"]).cuda(), neox, kv,
        B.MLA_KV_BF16 if kv_dtype == "bf16" else B.MLA_KV_E4M3, torch.from_numpy(st["slots"]).cuda())
    torch.cuda.synchronize()
    err = B.mla_decode_device_error()
    kv_h = kv.cpu().numpy()
    return q_out.cpu().numpy(), (kv_h.view(np.uint16) if kv_dtype == "bf16" else kv_h), err


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("page", [32, 64])
@pytest.mark.parametrize("t,h", [(1, 1), (7, 16), (64, 128)])
def test_fp8_query_and_cache(neox, page, t, h):
    st = make_step(t * 131 + h, t, h, page, "e4m3", pool_pages=max(8, t))
    q_out, kv, err = run_kernel(st, B.MLA_Q_E4M3, "e4m3", neox)
    assert err == 0
    qc, kc, _, _ = K.rope_quantize_fp8(st["q_nope"], st["q_rope"], st["k_nope"], st["k_rope"], st["pos"], st["cs"],
                                       neox)
    assert np.array_equal(q_out, qc)
    assert np.array_equal(kv, K.kv_cache_write(st["kv"], kc, st["slots"], page))


@pytest.mark.parametrize("neox", [True, False])
def test_bf16_query_and_cache(neox):
    st = make_step(3, 33, 16, 64, "bf16")
    q_out, kv, err = run_kernel(st, B.MLA_Q_BF16, "bf16", neox)
    assert err == 0
    assert np.array_equal(q_out.view(np.uint16), K.rope_bf16(st["q_rope"], st["pos"], st["cs"], neox))
    rows = np.concatenate([st["k_nope"], K.rope_bf16(st["k_rope"], st["pos"], st["cs"], neox)], axis=1)
    assert np.array_equal(kv, K.kv_cache_write(st["kv"], rows, st["slots"], 64))


def test_bf16_query_with_fp8_cache_and_saturation():
    """Large values: the FP8 codes saturate at 448 (and rounding to zero
    keeps the sign) exactly as the oracle's."""
    st = make_step(4, 9, 8, 32, "e4m3", scale=300.0)
    st["k_nope"][0, :8] = W.f32_to_bf16_bits(np.array([1e5, -1e5, 460, -460, 1e-6, -1e-6, 0.0, -0.0],
                                                       dtype=np.float32))
    q_out, kv, err = run_kernel(st, B.MLA_Q_BF16, "e4m3", False)
    assert err == 0
    _, kc, _, _ = K.rope_quantize_fp8(st["q_nope"], st["q_rope"], st["k_nope"], st["k_rope"], st["pos"], st["cs"],
                                      False)
    assert np.array_equal(kv, K.kv_cache_write(st["kv"], kc, st["slots"], 32))
    assert np.array_equal(q_out.view(np.uint16), K.rope_bf16(st["q_rope"], st["pos"], st["cs"], False))


def test_plain_cache_write_without_rotation_or_query():
    st = make_step(5, 20, 4, 64, "bf16")
    kv = torch.from_numpy(st["kv"].view(np.int16)).cuda()
    B.mla_rope_quantize_cache_write(None, None, None, B.MLA_Q_BF16, dev16(st["k_nope"]), dev16(st["k_rope"]),
                                    None, None, False, kv, B.MLA_KV_BF16, torch.from_numpy(st["slots"]).cuda())
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    rows = np.concatenate([st["k_nope"], st["k_rope"]], axis=1)
    assert np.array_equal(kv.cpu().numpy().view(np.uint16), K.kv_cache_write(st["kv"], rows, st["slots"], 64))


def test_more_tokens_than_one_grid_column():
    """70,000 new tokens: the launch covers at most 65,535 tokens per grid
    column and loops over the rest.  Every cache row must be rewritten, and a
    sample of tokens on both sides of the 65,535 boundary must match the
    oracle bit for bit (query codes and cache rows)."""
    t = 70_000
    st = make_step(8, t, 1, 64, "e4m3", pool_pages=t // 64 + 8)
    q_out, kv, err = run_kernel(st, B.MLA_Q_E4M3, "e4m3", False)
    assert err == 0
    sample = np.unique(np.concatenate([np.arange(0, 64), np.arange(65_500, 65_600), np.arange(t - 64, t),
                                       np.random.default_rng(9).integers(0, t, 200)]))
    qc, kc, _, _ = K.rope_quantize_fp8(st["q_nope"][sample], st["q_rope"][sample], st["k_nope"][sample],
                                       st["k_rope"][sample], st["pos"][sample], st["cs"], False)
    assert np.array_equal(q_out[sample], qc)
    flat_new, flat_old = kv.reshape(-1, 576), st["kv"].reshape(-1, 576)
    assert np.array_equal(flat_new[st["slots"][sample]], kc)
    # rows of every token changed (a random 576-byte row rewritten with the same bytes is not a real risk)
    assert np.all(np.any(flat_new[st["slots"]] != flat_old[st["slots"]], axis=1))
    untouched = np.setdiff1d(np.arange(flat_old.shape[0]), st["slots"])
    assert np.array_equal(flat_new[untouched], flat_old[untouched])


def test_bad_positions_and_slots_are_reported_not_written():
    st = make_step(6, 4, 2, 64, "e4m3", pool_pages=8, max_pos=100)
    st["pos"][1] = 100      # past the table: token 1 untouched
    st["slots"][2] = 8 * 64  # past the cache: key 2 untouched, its query written
    q_out, kv, err = run_kernel(st, B.MLA_Q_E4M3, "e4m3", True)
    assert err in (0x601, 0x602)
    ok = [0, 3]
    qc, kc, _, _ = K.rope_quantize_fp8(st["q_nope"][ok], st["q_rope"][ok], st["k_nope"][ok], st["k_rope"][ok],
                                       st["pos"][ok], st["cs"], True)
    assert np.array_equal(q_out[ok], qc) and np.all(q_out[1] == 0)
    qc2, _, _, _ = K.rope_quantize_fp8(st["q_nope"][[2]], st["q_rope"][[2]], st["k_nope"][[2]], st["k_rope"][[2]],
                                       st["pos"][[2]], st["cs"], True)
    assert np.array_equal(q_out[2], qc2[0])
    assert np.array_equal(kv, K.kv_cache_write(st["kv"], kc, st["slots"][ok], 64))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_written_tokens_are_decoded(kv_dtype):
    """A decode step end to end: the new tokens' keys go into the cache at
    the next slot of each request (RoPE applied), the query's rope part is
    rotated, and the decode over the updated cache matches the oracle over
    the oracle-updated cache."""
    rng = np.random.default_rng(7)
    lens_before = np.array([100, 63, 2000, 0, 640], dtype=np.int32)
    w = W.make_workload("dsv3", seed=7, seq_lens=list(lens_before + 1), num_heads=16, kv_dtype=kv_dtype,
                        k_scale=1.0, pool_pages=200)
    t, h, page = w.batch, w.num_heads, w.page_size
    cs = roformer_cache(8192).astype(np.float32)
    pos = lens_before.astype(np.int64)   # the new token's position is the old length
    slots = np.array([w.block_table[b, lens_before[b] // page] * page + lens_before[b] % page for b in range(t)],
                     dtype=np.int64)
    k_nope, k_rope = bf16(rng, (t, 512)), bf16(rng, (t, 64))
    q_rope_raw = bf16(rng, (t, h, 64))
    db = R.upload(w)
    q_pe = torch.empty((t, h, 64), dtype=torch.bfloat16, device="cuda")
    B.mla_rope_quantize_cache_write(db.q_nope, dev16(q_rope_raw), q_pe, B.MLA_Q_BF16, dev16(k_nope), dev16(k_rope),
                                    torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(), False, db.kv,
                                    db.kv_dtype, torch.from_numpy(slots).cuda())
    db.q_pe = q_pe
    out, lse = R.decode(db)
    torch.cuda.synchronize()
    assert B.mla_decode_device_error() == 0
    if kv_dtype == "bf16":
        rows = np.concatenate([k_nope, K.rope_bf16(k_rope, pos, cs, False)], axis=1)
    else:
        _, rows, _, _ = K.rope_quantize_fp8(np.zeros((t, 1, 512), np.uint16), np.zeros((t, 1, 64), np.uint16),
                                            k_nope, k_rope, pos, cs, False)
    kv_new = K.kv_cache_write(w.kv_bits, rows, slots, page)
    q_pe_ref = K.rope_bf16(q_rope_raw, pos, cs, False)
    ref_out, ref_lse = O.mla_decode(w.q_nope_bits, q_pe_ref, kv_new, w.kv_dtype, w.block_table, w.seq_lens,
                                    w.q_len, page, w.scale, w.k_scale)
    check(w, out, lse, ref_out, ref_lse)
