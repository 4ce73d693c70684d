"""Writes tiny_oracle.txt: the float64 oracle's output on the seeded tiny
workload (B=2, H=16, seq_lens {64,100}, page 64, seed 0).  Calls only the
oracle and the seeded input generator; nothing here comes from the CUDA path.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import mla_ref as O  # noqa: E402
from paged_mla_decode_08_gb300 import workloads as W  # noqa: E402


def main():
    w = W.make_workload("tiny", seed=0)
    out, lse = O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table,
                            w.seq_lens, w.q_len, w.page_size, w.scale, w.k_scale)
    fmt = lambda a: " ".join(repr(float(x)) for x in np.asarray(a).reshape(-1))  # noqa: E731
    with open(os.path.join(HERE, "tiny_oracle.txt"), "w") as f:
        f.write("# float64 oracle on workload 'tiny' (seed 0); written by make_golden.py\n")
        f.write(f"lse = {fmt(lse)}\n")
        f.write(f"out_every_97th = {fmt(out.reshape(-1)[::97])}\n")
        f.write(f"out_row_sums = {fmt(out.sum(axis=-1))}\n")


if __name__ == "__main__":
    main()
