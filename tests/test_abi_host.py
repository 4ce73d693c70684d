"""C ABI on the host: the library loads without a GPU, exports every function
include/mla_decode.h declares, and rejects bad arguments before any launch
(no GPU is touched by these tests)."""

import ctypes
import os
import re

import numpy as np
import pytest

from paged_mla_decode_08_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla_decode.h")


def declared_functions():
    with open(HEADER) as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "mla_decode_plan" in names and "mla_decode" in names
    lib = ctypes.CDLL(B.LIB)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
        assert n in B.SIGNATURES, f"{n} has no binding signature"


def test_version_and_constants():
    assert B.mla_decode_version() >= 100
    assert B.mla_planner_constants() == (64, 3, 4)
    assert B.load().mla_decode_last_error_string() is not None


FAKE = 1 << 20  # a 256-aligned non-NULL address; never dereferenced: every
                # case below is rejected on the host before any launch


def call_decode(plan, **over):
    kw = dict(q_nope=FAKE, q_pe=FAKE, num_tokens=plan.batch * plan.q_len, num_heads=plan.num_heads,
              kv=FAKE, kv_dtype=B.MLA_KV_BF16, num_pages=100, page_size=plan.page_size, bt=FAKE,
              bt_stride=64, seq_lens=FAKE, scale=0.07, k_scale=1.0, out=FAKE, lse=FAKE,
              ws=FAKE, ws_bytes=plan.workspace_bytes, stream=None)
    kw.update(over)
    return B.load().mla_decode(plan.handle, kw["q_nope"], kw["q_pe"], kw["num_tokens"], kw["num_heads"],
                               kw["kv"], kw["kv_dtype"], kw["num_pages"], kw["page_size"], kw["bt"],
                               kw["bt_stride"], kw["seq_lens"], kw["scale"], kw["k_scale"], kw["out"],
                               kw["lse"], kw["ws"], kw["ws_bytes"], kw["stream"])


@pytest.fixture
def split_plan():
    p = B.mla_decode_plan([4000, 3000, 100], 64, 128, 1, num_sms=148)
    assert p.workspace_bytes > 0
    return p


@pytest.mark.parametrize("over,code", [
    (dict(num_tokens=5), B.MLA_ERR_PLAN_MISMATCH),
    (dict(num_heads=64), B.MLA_ERR_PLAN_MISMATCH),
    (dict(page_size=32), B.MLA_ERR_PLAN_MISMATCH),
    (dict(kv_dtype=7), B.MLA_ERR_ARG),
    (dict(num_pages=0), B.MLA_ERR_ARG),
    (dict(num_pages=1 << 40), B.MLA_ERR_ARG),
    (dict(bt_stride=10), B.MLA_ERR_ARG),
    (dict(scale=0.0), B.MLA_ERR_ARG),
    (dict(scale=float("nan")), B.MLA_ERR_ARG),
    (dict(kv_dtype=B.MLA_KV_E4M3, k_scale=0.0), B.MLA_ERR_ARG),
    (dict(kv_dtype=B.MLA_KV_E4M3, k_scale=float("inf")), B.MLA_ERR_ARG),
    (dict(kv=FAKE + 8), B.MLA_ERR_ARG),
    (dict(q_nope=None), B.MLA_ERR_ARG),
    (dict(lse=None), B.MLA_ERR_ARG),
    (dict(ws=None), B.MLA_ERR_WORKSPACE),
    (dict(ws_bytes=100), B.MLA_ERR_WORKSPACE),
    (dict(ws=FAKE + 128), B.MLA_ERR_WORKSPACE),
])
def test_decode_rejects(split_plan, over, code):
    rc = call_decode(split_plan, **over)
    assert rc == code, B.load().mla_decode_last_error_string()
    assert B.load().mla_decode_last_error_string()


def call_host_io(plan, host_null=None, **over):
    kw = dict(q_nope=FAKE, q_pe=FAKE, num_tokens=plan.batch * plan.q_len, num_heads=plan.num_heads,
              kv=FAKE, kv_dtype=B.MLA_KV_BF16, num_pages=100, page_size=plan.page_size, bt=FAKE,
              bt_stride=64, seq_lens=FAKE, scale=0.07, k_scale=1.0, out=FAKE, lse=FAKE,
              ws=FAKE, ws_bytes=plan.workspace_bytes)
    kw.update(over)
    host = [FAKE] * 6
    if host_null is not None:
        host[host_null] = None
    return B.load().mla_decode_host_io(plan.handle, kw["q_nope"], kw["q_pe"], kw["num_tokens"], kw["num_heads"],
                                       kw["kv"], kw["kv_dtype"], kw["num_pages"], kw["page_size"], kw["bt"],
                                       kw["bt_stride"], kw["seq_lens"], kw["scale"], kw["k_scale"], kw["out"],
                                       kw["lse"], kw["ws"], kw["ws_bytes"], *host, None)


@pytest.mark.parametrize("host_null", range(6))
def test_host_io_rejects_null_host_pointer(split_plan, host_null):
    assert call_host_io(split_plan, host_null) == B.MLA_ERR_ARG
    assert "host pointer" in B.load().mla_decode_last_error_string().decode()


@pytest.mark.parametrize("over,code", [
    (dict(num_tokens=5), B.MLA_ERR_PLAN_MISMATCH),
    (dict(q_nope=None), B.MLA_ERR_ARG),
    (dict(ws=None), B.MLA_ERR_WORKSPACE),
])
def test_host_io_checks_device_arguments_like_decode(split_plan, over, code):
    assert call_host_io(split_plan, **over) == code


def test_decode_null_plan():
    rc = B.load().mla_decode(None, FAKE, FAKE, 1, 1, FAKE, 0, 1, 64, FAKE, 1, FAKE, 0.1, 1.0, FAKE, FAKE,
                             None, 0, None)
    assert rc == B.MLA_ERR_ARG


def no_gpu():
    """Cases whose arguments pass validation carry fake pointers: run them
    only where no GPU is visible, so the call stops at the device check and
    never launches."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("valid arguments on fake pointers would launch on a GPU")


def test_bf16_k_scale_is_ignored_not_rejected(split_plan):
    # a bf16 cache ignores k_scale (any value passes validation); without a
    # GPU the call then stops at the device check
    no_gpu()
    rc = call_decode(split_plan, k_scale=0.0)
    assert rc in (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED, B.MLA_OK)


def test_combine_rejects_small_workspace(split_plan):
    rc = B.load().mla_decode_combine(split_plan.handle, FAKE, FAKE, FAKE, 64, None)
    assert rc == B.MLA_ERR_WORKSPACE


def test_combine_without_splits_is_noop():
    p = B.mla_decode_plan([10], 64, 16, 1, num_sms=148)
    assert B.load().mla_decode_combine(p.handle, FAKE, FAKE, None, 0, None) == B.MLA_OK


def test_segment_capacity_limit():
    # more segments than one launch's parameter block holds
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan(np.full(5000, 10, dtype=np.int32), 64, 16, 1, num_sms=148)
    assert ei.value.code == B.MLA_ERR_ARG


def call_bt_tokens(**over):
    kw = dict(pool=FAKE, rows=10, cols=640, idx=FAKE, lens=FAKE, batch=3, page=64, bt=FAKE, mb=10)
    kw.update(over)
    return B.load().mla_block_table_from_tokens(kw["pool"], kw["rows"], kw["cols"], kw["idx"], kw["lens"],
                                                kw["batch"], kw["page"], kw["bt"], kw["mb"], None)


def call_bt_pages(**over):
    kw = dict(pool=FAKE, rows=10, cols=10, idx=FAKE, batch=3, bt=FAKE, mb=10)
    kw.update(over)
    return B.load().mla_block_table_from_pages(kw["pool"], kw["rows"], kw["cols"], kw["idx"], kw["batch"],
                                               kw["bt"], kw["mb"], None)


@pytest.mark.parametrize("over", [
    dict(page=16), dict(page=128), dict(lens=None), dict(lens=FAKE + 2), dict(pool=None), dict(idx=None),
    dict(bt=None), dict(batch=0), dict(mb=0), dict(mb=B.MLA_BLOCK_TABLE_MAX_BLOCKS + 1), dict(rows=0),
    dict(cols=0), dict(rows=1 << 40, cols=1 << 40), dict(bt=FAKE + 1),
])
def test_block_table_from_tokens_rejects(over):
    assert call_bt_tokens(**over) == B.MLA_ERR_ARG
    assert B.load().mla_decode_last_error_string()


@pytest.mark.parametrize("over", [
    dict(pool=None), dict(idx=None), dict(bt=None), dict(batch=-1), dict(mb=0), dict(rows=0), dict(cols=-5),
    dict(idx=FAKE + 3),
])
def test_block_table_from_pages_rejects(over):
    assert call_bt_pages(**over) == B.MLA_ERR_ARG


def test_block_table_valid_args_reach_device_check():
    # valid arguments pass validation; without a GPU the call then stops at
    # the device check (never at a launch)
    no_gpu()
    assert call_bt_tokens() in (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED, B.MLA_OK)
    assert call_bt_pages() in (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED, B.MLA_OK)


def call_ragged(plan, **over):
    kw = dict(q_nope=FAKE, q_pe=FAKE, num_tokens=5, num_heads=plan.num_heads, kv=FAKE, kv_dtype=B.MLA_KV_BF16,
              num_pages=100, page_size=plan.page_size, bt=FAKE, bt_stride=64, seq_lens=FAKE, cu=FAKE,
              scale=0.07, k_scale=1.0, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=plan.workspace_bytes, stream=None)
    kw.update(over)
    return B.load().mla_decode_ragged(plan.handle, kw["q_nope"], kw["q_pe"], kw["num_tokens"], kw["num_heads"],
                                      kw["kv"], kw["kv_dtype"], kw["num_pages"], kw["page_size"], kw["bt"],
                                      kw["bt_stride"], kw["seq_lens"], kw["cu"], kw["scale"], kw["k_scale"],
                                      kw["out"], kw["lse"], kw["ws"], kw["ws_bytes"], kw["stream"])


@pytest.fixture
def ragged_plan():
    p = B.mla_decode_plan_ragged([4000, 3000, 100], [1, 4, 2], 64, 16, num_sms=148)
    assert p.q_len == 4 and p.workspace_bytes > 0
    return p


@pytest.mark.parametrize("over,code", [
    (dict(cu=None), B.MLA_ERR_ARG),
    (dict(cu=FAKE + 2), B.MLA_ERR_ARG),
    (dict(num_tokens=0), B.MLA_ERR_PLAN_MISMATCH),
    (dict(num_tokens=13), B.MLA_ERR_PLAN_MISMATCH),   # > batch * max q_len = 12
    (dict(num_heads=8), B.MLA_ERR_PLAN_MISMATCH),
    (dict(ws_bytes=10), B.MLA_ERR_WORKSPACE),
    (dict(q_pe=None), B.MLA_ERR_ARG),
])
def test_ragged_decode_rejects(ragged_plan, over, code):
    assert call_ragged(ragged_plan, **over) == code


def test_ragged_plan_rules():
    # planned rows follow the largest query count; zero counts are allowed
    p = B.mla_decode_plan_ragged([10, 20, 30], [0, 8, 3], 64, 16, num_sms=148)
    assert p.q_len == 8
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan_ragged([10, 20], [1, 9], 64, 16, num_sms=148)   # 16 * 9 > 128 rows
    assert ei.value.code == B.MLA_ERR_ARG
    with pytest.raises(B.MlaError) as ei:
        B.mla_decode_plan_ragged([10, 20], [1, -1], 64, 16, num_sms=148)
    assert ei.value.code == B.MLA_ERR_ARG
    # the schedule ignores query counts: same segments as the uniform plan
    u = B.mla_decode_plan([4000, 3000, 100], 64, 16, 4, num_sms=148)
    r = B.mla_decode_plan_ragged([4000, 3000, 100], [1, 4, 2], 64, 16, num_sms=148)
    assert np.array_equal(u.segments(), r.segments()) and u.workspace_bytes == r.workspace_bytes


def test_ragged_valid_args_reach_device_check(ragged_plan):
    no_gpu()
    assert call_ragged(ragged_plan) in (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED, B.MLA_OK)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), B.MLA_ERR_ARG), (dict(q=FAKE + 8), B.MLA_ERR_ARG), (dict(num_tokens=5), B.MLA_ERR_PLAN_MISMATCH),
    (dict(num_heads=8), B.MLA_ERR_PLAN_MISMATCH), (dict(k_scale=0.0), B.MLA_ERR_ARG), (dict(ws=None), B.MLA_ERR_WORKSPACE),
])
def test_decode_fp8q_rejects(split_plan, over, code):
    kw = dict(q=FAKE, num_tokens=split_plan.batch * split_plan.q_len, num_heads=split_plan.num_heads, kv=FAKE,
              num_pages=100, page_size=split_plan.page_size, bt=FAKE, bt_stride=64, seq_lens=FAKE, cu=None,
              scale=0.07, k_scale=1.0, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=split_plan.workspace_bytes)
    kw.update(over)
    rc = B.load().mla_decode_fp8q(split_plan.handle, kw["q"], kw["num_tokens"], kw["num_heads"], kw["kv"],
                                  kw["num_pages"], kw["page_size"], kw["bt"], kw["bt_stride"], kw["seq_lens"],
                                  kw["cu"], kw["scale"], kw["k_scale"], kw["out"], kw["lse"], kw["ws"],
                                  kw["ws_bytes"], None)
    assert rc == code


def test_binding_refuses_a_missing_library(tmp_path):
    """The product path has no fallback: a missing shared library is an error."""
    missing = str(tmp_path / "libmladecode.so")
    with pytest.raises(RuntimeError, match="not built"):
        B.load(missing)


def call_rope_write(**over):
    kw = dict(q_nope=FAKE, q_rope=FAKE, num_tokens=4, num_heads=8, q_out=FAKE, q_out_dtype=B.MLA_Q_E4M3,
              k_nope=FAKE, k_rope=FAKE, positions=FAKE, cos_sin=FAKE, max_position=4096, is_neox=0,
              kv=FAKE, kv_dtype=B.MLA_KV_E4M3, num_pages=64, page_size=64, slots=FAKE, stream=None)
    kw.update(over)
    return B.load().mla_rope_quantize_cache_write(
        kw["q_nope"], kw["q_rope"], kw["num_tokens"], kw["num_heads"], kw["q_out"], kw["q_out_dtype"],
        kw["k_nope"], kw["k_rope"], kw["positions"], kw["cos_sin"], kw["max_position"], kw["is_neox"],
        kw["kv"], kw["kv_dtype"], kw["num_pages"], kw["page_size"], kw["slots"], kw["stream"])


@pytest.mark.parametrize("over", [
    dict(num_tokens=0), dict(num_heads=-1), dict(num_heads=(1 << 16) + 1),
    dict(num_tokens=1 << 30, num_heads=1 << 16),               # more items than one grid covers
    dict(q_out_dtype=7), dict(kv_dtype=5), dict(page_size=16), dict(num_pages=0), dict(num_pages=1 << 40),
    dict(k_nope=None), dict(k_rope=None), dict(kv=None), dict(slots=None),
    dict(q_rope=None), dict(q_out=None), dict(q_nope=None),   # the e4m3 query needs its latent part
    dict(positions=None), dict(max_position=0),               # a table needs positions
    dict(k_nope=FAKE + 8), dict(kv=FAKE + 4), dict(slots=FAKE + 4), dict(cos_sin=FAKE + 4), dict(q_out=FAKE + 8),
])
def test_rope_cache_write_rejects(over):
    assert call_rope_write(**over) == B.MLA_ERR_ARG


def test_rope_cache_write_valid_args_reach_device_check():
    no_gpu()
    ok = (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED, B.MLA_OK)
    assert call_rope_write() in ok
    # a plain cache write: no query at all, and no rotation table
    assert call_rope_write(num_heads=0, q_nope=None, q_rope=None, q_out=None, cos_sin=None, positions=None) in ok
    # a bf16 q_pe output needs no latent query input
    assert call_rope_write(q_out_dtype=B.MLA_Q_BF16, q_nope=None, kv_dtype=B.MLA_KV_BF16) in ok
