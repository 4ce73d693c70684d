"""Strength of the oracle's pins: plant a plausible mistake in a copy of the
oracle (on the CPU, never in the CUDA path) and check that at least one pin of
``test_oracle.py`` rejects it."""

import inspect
import types

import pytest

from oracle import mla_ref as O

import test_oracle as P

# (name, text in the oracle, planted replacement)
MUTATIONS = [
    ("dropped rope term",
     " + qp @ rows[:, KV_LORA_RANK:].T", ""),
    ("value slice starts at the rope columns",
     "out = (p @ rows[:, :KV_LORA_RANK])", "out = (p @ rows[:, ROPE_DIM:])"),
    ("causal off by one",
     "v = max(n - q_len + 1 + i, 0)", "v = max(n - q_len + i, 0)"),
    ("log base 2 in lse",
     "lse = m[:, 0] + np.log(l)", "lse = m[:, 0] + np.log2(l)"),
    ("lse without the max",
     "lse = m[:, 0] + np.log(l)", "lse = np.log(l)"),
    ("page and slot swapped",
     "return kv_bits[pages, j % page_size]", "return kv_bits[pages, (j * 7) % page_size]"),
    ("block table indexed by token",
     "pages = np.asarray(bt_row, dtype=np.int64)[j // page_size]",
     "pages = np.asarray(bt_row, dtype=np.int64)[np.minimum(j, len(bt_row) - 1) // page_size]"),
    ("scale dropped",
     "s = scale * (qn @", "s = (qn @"),
    ("k_scale ignored",
     'dq = k_scale if kv_dtype == "e4m3" else 1.0', "dq = 1.0"),
    ("k_scale applied twice",
     "kv_dtype) * dq", "kv_dtype) * dq * dq"),
    ("merge weights not normalised",
     "wn = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)", "wn = w"),
    ("zero-length rows not -inf",
     "return np.zeros((h, KV_LORA_RANK)), np.full(h, -np.inf)",
     "return np.zeros((h, KV_LORA_RANK)), np.zeros(h)"),
]


def mutated(old, new):
    src = inspect.getsource(O)
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def caught(mod):
    checks = [
        lambda: P.pin_sdpa(mod.mla_decode) >= 1e-12,
        lambda: P.pin_absorption(mod.attend) >= 1e-10,
        lambda: P.pin_page_permutation(mod.mla_decode) != 0.0,
        lambda: P.pin_single_key(mod.mla_decode) >= 1e-13,
        lambda: P.pin_equal_scores(mod.mla_decode) >= 1e-13,
        lambda: P.pin_zero_length(mod.mla_decode) != 0.0,
        lambda: P.pin_draft_expansion(mod.mla_decode) != 0.0,
        lambda: P.pin_split_merge(mod.attend, mod.merge_splits) >= 1e-12,
        lambda: P.pin_fp8_scale(mod.mla_decode) >= 1e-12,
    ]
    hits = []
    for i, c in enumerate(checks):
        try:
            if c():
                hits.append(i)
        except Exception:  # a crash is a rejection too
            hits.append(i)
    return hits


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    assert caught(mutated(old, new)), f"no pin rejects: {name}"


def test_unmutated_passes_all_pins():
    assert caught(O) == []
