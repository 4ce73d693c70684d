"""Device-side plumbing around the binding: move a seeded workload's stored
bit patterns into torch CUDA tensors, plan, allocate outputs and workspace,
and call the library.  Torch only holds memory and streams here."""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding as B
from .workloads import KV_LORA_RANK, Workload


@dataclass
class DeviceBatch:
    w: Workload
    plan: B.Plan
    q_nope: torch.Tensor  # bf16 [T,H,512]
    q_pe: torch.Tensor  # bf16 [T,H,64]
    kv: torch.Tensor  # bf16 or uint8 [P,page,576]
    kv_dtype: int
    block_table: torch.Tensor  # int32 [B, stride]
    seq_lens: torch.Tensor  # int32 [B]
    out: torch.Tensor  # bf16 [T,H,512]
    lse: torch.Tensor  # fp32 [T,H]
    workspace: Optional[torch.Tensor]
    cu_seqlens_q: Optional[torch.Tensor] = None  # int32 [B+1] for a ragged batch


def _bits_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def upload(w: Workload, device="cuda", num_sms: int = 0, plan_seq_lens=None) -> DeviceBatch:
    """Copy ``w`` to ``device`` and plan it (``plan_seq_lens`` overrides the
    host lengths the plan is made from, e.g. upper bounds)."""
    lens = w.seq_lens if plan_seq_lens is None else np.asarray(plan_seq_lens, dtype=np.int32)
    if w.cu_seqlens_q is not None:
        plan = B.mla_decode_plan_ragged(lens, w.q_lens(), w.page_size, w.num_heads, num_sms)
    else:
        plan = B.mla_decode_plan(lens, w.page_size, w.num_heads, w.q_len, num_sms)
    if w.kv_dtype == "bf16":
        kv = _bits_to_bf16(w.kv_bits, device)
        kv_dtype = B.MLA_KV_BF16
    else:
        kv = torch.from_numpy(np.ascontiguousarray(w.kv_bits)).to(device)
        kv_dtype = B.MLA_KV_E4M3
    t, h = w.num_tokens, w.num_heads
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=device)
    return DeviceBatch(
        w=w, plan=plan,
        q_nope=_bits_to_bf16(w.q_nope_bits, device), q_pe=_bits_to_bf16(w.q_pe_bits, device),
        kv=kv, kv_dtype=kv_dtype,
        block_table=torch.from_numpy(np.ascontiguousarray(w.block_table)).to(device),
        seq_lens=torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device),
        out=torch.empty((t, h, KV_LORA_RANK), dtype=torch.bfloat16, device=device),
        lse=torch.empty((t, h), dtype=torch.float32, device=device),
        workspace=ws,
        cu_seqlens_q=None if w.cu_seqlens_q is None else torch.from_numpy(w.cu_seqlens_q).to(device),
    )


def decode(db: DeviceBatch, stream=None):
    if db.cu_seqlens_q is not None:
        B.mla_decode_ragged(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                            db.cu_seqlens_q, db.w.scale, db.w.k_scale, db.out, db.lse, db.workspace, None, stream)
    else:
        B.mla_decode(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                     db.w.scale, db.w.k_scale, db.out, db.lse, db.workspace, None, stream)
    return db.out, db.lse


def decode_main(db: DeviceBatch, stream=None):
    B.mla_decode_main(db.plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                      db.w.scale, db.w.k_scale, db.out, db.lse, db.workspace, None, stream)


def decode_combine(db: DeviceBatch, stream=None):
    B.mla_decode_combine(db.plan, db.out, db.lse, db.workspace, None, stream)
