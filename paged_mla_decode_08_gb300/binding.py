"""Thin ctypes binding of libmladecode.so (the C ABI in include/mla_decode.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Torch tensors are accepted for convenience and are only used
for their device pointers and the current CUDA stream.  There is no fallback:
if the library is missing, loading fails loudly.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from .build import LIB

MLA_OK = 0
MLA_ERR_ARG = -1
MLA_ERR_WORKSPACE = -2
MLA_ERR_PLAN_MISMATCH = -3
MLA_ERR_CUDA = -4
MLA_ERR_UNSUPPORTED = -5
MLA_KV_BF16 = 0
MLA_KV_E4M3 = 1

# Every symbol the header declares, with its ctypes signature.
_c_int, _c_size, _vp, _i32p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
_DECODE_ARGS = [_vp, _vp, _vp, _c_int, _c_int, _vp, _c_int, ctypes.c_int64, _c_int, _vp, _c_int, _vp,
                ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _c_size, _vp]
SIGNATURES = {
    "mla_decode_plan": (_c_int, [_i32p, _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_vp),
                                 ctypes.POINTER(_c_size)]),
    "mla_plan_destroy": (None, [_vp]),
    "mla_decode": (_c_int, _DECODE_ARGS),
    "mla_decode_main": (_c_int, _DECODE_ARGS),
    "mla_decode_combine": (_c_int, [_vp, _vp, _vp, _vp, _c_size, _vp]),
    "mla_decode_noalloc": (_c_int, _DECODE_ARGS[:16] + [_vp]),
    "mla_decode_host_io": (_c_int, _DECODE_ARGS[:18] + [_vp] * 6 + [_vp]),
    "mla_decode_plan_ragged": (_c_int, [_i32p, _i32p, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_vp),
                                        ctypes.POINTER(_c_size)]),
    "mla_decode_ragged": (_c_int, _DECODE_ARGS[:12] + [_vp] + _DECODE_ARGS[12:]),
    "mla_decode_plan_device": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_vp),
                                        ctypes.POINTER(_c_size)]),
    "mla_plan_is_device": (_c_int, [_vp]),
    "mla_plan_read_device_schedule": (_c_int, [_vp, _vp, _i32p, _c_int, ctypes.POINTER(_c_int)]),
    "mla_rope_quantize_cache_write": (_c_int, [_vp, _vp, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp, _vp,
                                               ctypes.c_int64, _c_int, _vp, _c_int, ctypes.c_int64, _c_int, _vp,
                                               _vp]),
    "mla_decode_fp8q": (_c_int, [_vp, _vp, _c_int, _c_int, _vp, ctypes.c_int64, _c_int, _vp, _c_int, _vp, _vp,
                                 ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _c_size, _vp]),
    "mla_block_table_from_tokens": (_c_int, [_vp, ctypes.c_int64, ctypes.c_int64, _vp, _vp, _c_int, _c_int,
                                             _vp, _c_int, _vp]),
    "mla_block_table_from_pages": (_c_int, [_vp, ctypes.c_int64, ctypes.c_int64, _vp, _c_int, _vp, _c_int,
                                            _vp]),
    "mla_plan_workspace_bytes": (_c_size, [_vp]),
    "mla_plan_num_workers": (_c_int, [_vp]),
    "mla_plan_num_segments": (_c_int, [_vp]),
    "mla_plan_get_segments": (_c_int, [_vp, _i32p, _c_int]),
    "mla_plan_num_partial_slots": (_c_int, [_vp]),
    "mla_planner_constants": (None, [ctypes.POINTER(_c_int)] * 3),
    "mla_decode_device_error": (_c_int, [ctypes.POINTER(_c_int), _c_int]),
    "mla_decode_last_error_string": (ctypes.c_char_p, []),
    "mla_decode_version": (_c_int, []),
}

_lib: Optional[ctypes.CDLL] = None


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"MLA error {code}: {msg}")
        self.code = code


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (built by build.build()); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libmladecode.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != MLA_OK:
        raise MlaError(rc, load().mla_decode_last_error_string().decode())


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owner of an ``mla_plan*``; destroyed with the object."""

    def __init__(self, handle: int, workspace_bytes: int, batch: int, page_size: int,
                 num_heads: int, q_len: int):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.batch, self.page_size, self.num_heads, self.q_len = batch, page_size, num_heads, q_len

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.mla_plan_destroy(self.handle)
            self.handle = None

    @property
    def num_workers(self) -> int:
        return load().mla_plan_num_workers(self.handle)

    @property
    def num_partial_slots(self) -> int:
        return load().mla_plan_num_partial_slots(self.handle)

    @property
    def is_device(self) -> bool:
        return bool(load().mla_plan_is_device(self.handle))

    def device_segments(self, workspace) -> np.ndarray:
        """The schedule the last decode built in ``workspace`` (device plans;
        synchronises): (worker, request, tile_begin, tile_end, slot) rows."""
        lib = load()
        cap = 1920
        buf = np.zeros(5 * cap, dtype=np.int32)
        n = ctypes.c_int()
        got = lib.mla_plan_read_device_schedule(self.handle, _ptr(workspace), buf.ctypes.data_as(_i32p), cap,
                                                ctypes.byref(n))
        if got < 0:
            _check(got)
        return buf[: 5 * got].reshape(got, 5)

    def segments(self) -> np.ndarray:
        """(worker, request, tile_begin, tile_end, partial_slot) rows."""
        lib = load()
        n = lib.mla_plan_num_segments(self.handle)
        buf = np.zeros(5 * n, dtype=np.int32)
        got = lib.mla_plan_get_segments(self.handle, buf.ctypes.data_as(_i32p), n)
        if got < 0:
            _check(got)
        return buf.reshape(n, 5)


def mla_decode_plan(seq_lens_host, page_size: int, num_heads: int, q_len: int = 1,
                    num_sms: int = 0) -> Plan:
    lib = load()
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    handle = _vp()
    ws = _c_size()
    _check(lib.mla_decode_plan(lens.ctypes.data_as(_i32p), int(lens.shape[0]), page_size, num_heads,
                               q_len, num_sms, ctypes.byref(handle), ctypes.byref(ws)))
    return Plan(handle.value, ws.value, int(lens.shape[0]), page_size, num_heads, q_len)


def mla_decode_plan_device(batch: int, page_size: int, num_heads: int, q_len: int = 1, num_sms: int = 0) -> Plan:
    """A plan whose schedule is built on the device from the device lengths
    at every decode (graph-capturable for any lengths)."""
    lib = load()
    handle = _vp()
    ws = _c_size()
    _check(lib.mla_decode_plan_device(batch, page_size, num_heads, q_len, num_sms, ctypes.byref(handle),
                                      ctypes.byref(ws)))
    return Plan(handle.value, ws.value, batch, page_size, num_heads, q_len)


def mla_decode_plan_ragged(seq_lens_host, q_lens_host, page_size: int, num_heads: int, num_sms: int = 0) -> Plan:
    """Plan a batch whose requests carry ``q_lens_host[b]`` query tokens each."""
    lib = load()
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    qls = np.ascontiguousarray(np.asarray(q_lens_host, dtype=np.int32))
    if qls.shape != lens.shape:
        raise MlaError(MLA_ERR_ARG, "q_lens and seq_lens differ in length")
    handle = _vp()
    ws = _c_size()
    _check(lib.mla_decode_plan_ragged(lens.ctypes.data_as(_i32p), qls.ctypes.data_as(_i32p), int(lens.shape[0]),
                                      page_size, num_heads, num_sms, ctypes.byref(handle), ctypes.byref(ws)))
    return Plan(handle.value, ws.value, int(lens.shape[0]), page_size, num_heads, max(int(qls.max(initial=1)), 1))


def _decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table, seq_lens, scale, k_scale,
                 out, lse, workspace, workspace_bytes, stream):
    num_pages = kv_pages.shape[0]
    page_size = kv_pages.shape[1]
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (plan.handle, _ptr(q_nope), _ptr(q_pe), int(q_nope.shape[0]), int(q_nope.shape[1]),
            _ptr(kv_pages), kv_dtype, int(num_pages), int(page_size), _ptr(block_table),
            int(block_table.shape[1]), _ptr(seq_lens), float(scale), float(k_scale), _ptr(out), _ptr(lse),
            _ptr(workspace), int(workspace_bytes), _stream(stream))


def mla_decode(plan: Plan, q_nope, q_pe, kv_pages, kv_dtype: int, block_table, seq_lens, scale: float,
               k_scale: float, out, lse, workspace=None, workspace_bytes=None, stream=None):
    """Decode into ``out`` / ``lse`` (torch CUDA tensors) on ``stream``."""
    _check(load().mla_decode(*_decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table, seq_lens,
                                           scale, k_scale, out, lse, workspace, workspace_bytes, stream)))


def mla_decode_host_io(plan: Plan, q_nope, q_pe, kv_pages, kv_dtype: int, block_table, seq_lens, scale: float,
                       k_scale: float, out, lse, workspace, q_nope_host, q_pe_host, block_table_host, seq_lens_host,
                       out_host, lse_host, stream=None):
    """``mla_decode`` with the step's inputs copied in from, and its results
    copied out to, host tensors (pinned for asynchronous copies); the device
    tensors q_nope, q_pe, block_table and seq_lens are overwritten.  The host
    results are valid once ``stream`` has been synchronised."""
    args = _decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table, seq_lens, scale, k_scale, out, lse,
                        workspace, None, stream)
    _check(load().mla_decode_host_io(*args[:18], _ptr(q_nope_host), _ptr(q_pe_host), _ptr(block_table_host),
                                     _ptr(seq_lens_host), _ptr(out_host), _ptr(lse_host), args[18]))


def mla_decode_ragged(plan: Plan, q_nope, q_pe, kv_pages, kv_dtype: int, block_table, seq_lens, cu_seqlens_q,
                      scale: float, k_scale: float, out, lse, workspace=None, workspace_bytes=None, stream=None):
    """Decode a ragged batch (query rows of request b: cu_seqlens_q[b] ..
    cu_seqlens_q[b+1]-1) into ``out`` / ``lse``."""
    args = _decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table, seq_lens, scale, k_scale, out, lse,
                        workspace, workspace_bytes, stream)
    _check(load().mla_decode_ragged(*args[:12], _ptr(cu_seqlens_q), *args[12:]))


def mla_decode_fp8q(plan: Plan, q, kv_pages, block_table, seq_lens, scale: float, k_scale: float, out, lse,
                    workspace=None, workspace_bytes=None, cu_seqlens_q=None, stream=None):
    """Decode with the merged e4m3 query ``q`` [T, H, 576] over an e4m3 cache."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().mla_decode_fp8q(plan.handle, _ptr(q), int(q.shape[0]), int(q.shape[1]), _ptr(kv_pages),
                                  int(kv_pages.shape[0]), int(kv_pages.shape[1]), _ptr(block_table),
                                  int(block_table.shape[1]), _ptr(seq_lens), _ptr(cu_seqlens_q), float(scale),
                                  float(k_scale), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)))


def mla_decode_main(plan: Plan, q_nope, q_pe, kv_pages, kv_dtype: int, block_table, seq_lens, scale: float,
                    k_scale: float, out, lse, workspace=None, workspace_bytes=None, stream=None):
    _check(load().mla_decode_main(*_decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table,
                                                seq_lens, scale, k_scale, out, lse, workspace,
                                                workspace_bytes, stream)))


def mla_decode_combine(plan: Plan, out, lse, workspace=None, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().mla_decode_combine(plan.handle, _ptr(out), _ptr(lse), _ptr(workspace),
                                     int(workspace_bytes), _stream(stream)))


def mla_decode_noalloc(plan: Plan, q_nope, q_pe, kv_pages, kv_dtype: int, block_table, seq_lens,
                       scale: float, k_scale: float, out, lse, stream=None):
    """mla_decode without a workspace: the library's built-in scratch array
    (MLA_NOALLOC_SCRATCH_BYTES) holds the split partials.  For callers that
    cannot allocate device memory; calls that overlap on the GPU race."""
    args = _decode_args(plan, q_nope, q_pe, kv_pages, kv_dtype, block_table, seq_lens, scale, k_scale,
                        out, lse, None, 0, stream)
    _check(load().mla_decode_noalloc(*args[:16], args[18]))


MLA_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
MLA_BLOCK_TABLE_MAX_BLOCKS = 65535 * 256
MLA_Q_BF16 = 0
MLA_Q_E4M3 = 1


def mla_rope_quantize_cache_write(q_nope, q_rope, q_out, q_out_dtype: int, k_nope, k_rope, positions,
                                  cos_sin_cache, is_neox: bool, kv_pages, kv_dtype: int, out_cache_loc,
                                  stream=None):
    """RoPE + (FP8) quantisation of the new tokens' query into ``q_out`` and
    of their keys into the cache at ``out_cache_loc`` (torch CUDA tensors;
    q tensors may be None for a plain cache write)."""
    t = int(k_nope.shape[0])
    h = 0 if q_rope is None else int(q_rope.shape[1])
    max_pos = 0 if cos_sin_cache is None else int(cos_sin_cache.shape[0])
    _check(load().mla_rope_quantize_cache_write(
        _ptr(q_nope), _ptr(q_rope), t, h, _ptr(q_out), int(q_out_dtype), _ptr(k_nope), _ptr(k_rope),
        _ptr(positions), _ptr(cos_sin_cache), max_pos, 1 if is_neox else 0, _ptr(kv_pages), int(kv_dtype),
        int(kv_pages.shape[0]), int(kv_pages.shape[1]), _ptr(out_cache_loc), _stream(stream)))


def mla_block_table_from_tokens(req_to_token, req_pool_indices, seq_lens, page_size: int, block_table,
                                stream=None):
    """Fill ``block_table`` (int32 CUDA [batch, max_blocks]) from a token pool
    ``req_to_token`` (int32 CUDA [pool_rows, token_cols], contiguous)."""
    rows, cols = req_to_token.shape
    _check(load().mla_block_table_from_tokens(_ptr(req_to_token), int(rows), int(cols), _ptr(req_pool_indices),
                                              _ptr(seq_lens), int(block_table.shape[0]), int(page_size),
                                              _ptr(block_table), int(block_table.shape[1]), _stream(stream)))


def mla_block_table_from_pages(req_to_page, req_pool_indices, block_table, stream=None):
    """Fill ``block_table`` (int32 CUDA [batch, max_blocks]) from a page pool
    ``req_to_page`` (int32 CUDA [pool_rows, page_cols], contiguous)."""
    rows, cols = req_to_page.shape
    _check(load().mla_block_table_from_pages(_ptr(req_to_page), int(rows), int(cols), _ptr(req_pool_indices),
                                             int(block_table.shape[0]), _ptr(block_table),
                                             int(block_table.shape[1]), _stream(stream)))


def mla_planner_constants():
    a, b, c = _c_int(), _c_int(), _c_int()
    load().mla_planner_constants(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return a.value, b.value, c.value


def mla_decode_device_error(reset: bool = True) -> int:
    """Kernel-side error word (0 = no bounded wait timed out); synchronises."""
    code = _c_int()
    _check(load().mla_decode_device_error(ctypes.byref(code), 1 if reset else 0))
    return code.value


def mla_decode_version() -> int:
    return load().mla_decode_version()
