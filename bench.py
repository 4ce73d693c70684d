"""Decode benchmark: weight-absorbed paged MLA decode on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config dsv3|tiny|long_skewed|spec_q4|fp8_kv] [--seed S]
                    [--soak SECONDS] [--cpu-seconds SECONDS] [--configs all|none|a,b]
                    [--profile [--pool-pages P]]

A step is one whole decode (split-KV main kernel + LSE combine) over one
resident batch of the DeepSeek-V3-shaped workload (B=64 requests, q_len=1,
H=128, kv_lora_rank 512 + rope 64, L ~ U[1024, 4096], page 64, shuffled
16384-page pool, seed 0).  L2 is flushed (a write of 2x the L2 size) between
steps, outside the timed events.  Rank 0 prints one JSON line; its
``configs`` object holds the same measurement for every other seeded
workload (tiny, long_skewed, spec_q4, fp8_kv), each with the roofline of its
main kernel, and ``host_plan_us`` / ``e2e_replan`` the cost of planning on
the host from the lengths of every step.

--impl reference times the float64 CPU oracle (the only reference this
decode has) on the host cores, same workload and metric.
"""

from __future__ import annotations

import os

# BLAS threads for the CPU oracle: every host core (set before numpy loads)
_CORES = os.cpu_count() or 1
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_mla_decode_08_gb300 import workloads as W  # noqa: E402

METRIC = "MLA decode tokens/s, KV HBM GB/s and tensor TFLOPS as % of roofline, 1×GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MAIN_KERNEL_SOURCES = ["mla_sm103.cu", "sm103_ptx.cuh", "mla_internal.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text):
    """Source text without comments and blank lines: what the compiled kernel
    depends on, so a comment edit keeps the profiles that match the code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash():
    """sha256 (first 16 hex digits) of the main kernel's sources, comments and
    blank lines removed."""
    h = hashlib.sha256()
    for f in MAIN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_mla_decode_08_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(config_name):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"mla_main_{config_name}_ncu.md")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        txt = fh.read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    hsh = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    if not m or not hsh or hsh.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


def workload_desc(w):
    return {
        "workload": f"{w.name}: {w.meta.get('desc', '')}",
        "batch": w.batch, "q_len": w.q_len, "num_heads": w.num_heads, "kv_dim": 576,
        "kv_lora_rank": 512, "page_size": w.page_size, "kv_dtype": w.kv_dtype,
        "pool_pages": w.num_pages, "seed": w.meta.get("seed", 0),
        "kv_tokens": int(w.seq_lens.sum()),
        "l2": "flushed between steps (write of 2x L2, outside the timed events)",
        "kv_cache": "resident in HBM (persistent state, like weights)",
    }


# ------------------------------------------------------------------ clocks


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.t0 = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t0 = time.time()
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        return rows

    @staticmethod
    def summarize(rows, peaks):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": peaks.get("sm_max_mhz"), "reasons": ["no samples"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle


def time_oracle(w, budget_s=10.0, max_s=30.0):
    """The float64 oracle as it stands, on the host cores; whole workload
    passes repeated until ``budget_s`` (request-sized steps, bounded)."""
    from oracle import mla_ref as O
    t0 = time.perf_counter()
    rows = 0
    passes = 0
    b = 0
    while True:
        O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
                     w.q_len, w.page_size, w.scale, w.k_scale, requests=[b])
        rows += w.q_len
        b += 1
        if b == w.batch:
            b = 0
            passes += 1
        el = time.perf_counter() - t0
        if (el >= budget_s and (passes >= 1 or el >= max_s)) or el >= max_s:
            break
    return rows / el, el, rows


def reference_arm(args, w, rank):
    if rank != 0:
        return
    st = W.workload_stats(w)
    from oracle import mla_ref as O
    # a step = one bounded sample of the workload: the first requests whose
    # KV adds up to ~1/8 of the batch (keeps K steps within a few minutes)
    target = st["kv_tokens"] / 8
    reqs, acc = [], 0
    for b in range(w.batch):
        reqs.append(b)
        acc += int(w.seq_lens[b])
        if acc >= target:
            break
    def step():
        O.mla_decode(w.q_nope_bits, w.q_pe_bits, w.kv_bits, w.kv_dtype, w.block_table, w.seq_lens,
                     w.q_len, w.page_size, w.scale, w.k_scale, requests=reqs)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    toks = len(reqs) * w.q_len * args.steps
    value = toks / el
    sample = f"requests 0..{reqs[-1]} of the workload ({acc} KV tokens) per step, float64 NumPy oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_desc(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _CORES, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm


def whole_job_rate(my_seconds, tokens_per_step, steps, world, dist=None, device=None):
    """Weak-scaling aggregate over replicas: every rank decodes its own copy
    of the workload for `steps` steps; the job's time is the slowest rank's
    (all-reduce MAX) and its tokens are all ranks' tokens.  Returns
    (tokens/s of the whole job, the job's seconds)."""
    import torch
    t = my_seconds
    if dist is not None and world > 1:
        buf = torch.tensor([my_seconds], dtype=torch.float64, device=device)
        dist.all_reduce(buf, op=dist.ReduceOp.MAX)
        t = float(buf.item())
    return tokens_per_step * steps * world / t, t


def our_arm(args, w, rank, world):
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    from paged_mla_decode_08_gb300 import runner as R
    from paged_mla_decode_08_gb300.build import build

    build()
    B.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=dev)
        dist = dist_mod
    peaks, peaks_kind = load_peaks()
    st = W.workload_stats(w)
    db = R.upload(w, device=dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    launches_per_step = 1 + (1 if db.plan.num_partial_slots > 0 else 0)

    def step():
        R.decode(db, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    # soak: keep the GPU busy with the same step so the clock sampler sees a
    # steady state even when K is small
    sampler = ClockSampler(dev.index)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(50):
            flush.zero_()
            step()
        torch.cuda.synchronize()

    K = args.steps
    # timed region: K steps of the public decode call (main kernel + combine,
    # the combine launched as a programmatic dependent of the main kernel)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        R.decode(db, stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - t0
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    # per-kernel split (an event between the launches, so no overlap): the
    # main kernel's own duration for the roofline line
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        evk[k][0].record(stream)
        R.decode_main(db, stream)
        evk[k][1].record(stream)
        R.decode_combine(db, stream)
        evk[k][2].record(stream)
    torch.cuda.synchronize()
    clock_rows = sampler.stop()
    main_ms = [e[0].elapsed_time(e[1]) for e in evk]
    comb_ms = [e[1].elapsed_time(e[2]) for e in evk]
    value, tot_s = whole_job_rate(sum(step_ms) / 1e3, st["tokens"], K, world, dist, dev)
    ms_per_step = tot_s * 1e3 / K

    # ---- the same host-planned step captured in a CUDA graph and replayed
    # (no per-launch host work; the lengths are fixed by the plan)
    graph_s = graph_step_seconds(lambda cs: R.decode(db, cs), dev, stream, flush, max(3, min(K, 200)))
    # ---- e2e: host buffers in, results back to the host, copies timed;
    # host-synchronous per step, and with the host link overlapped
    e2e_serial = e2e_measure(db, w, dev, stream, max(3, min(K, 200)))
    e2e = e2e_pipelined_measure(db, w, dev, stream, max(3, min(K, 200)))
    e2e_hio = e2e_host_io_measure(db, w, dev, stream, max(3, min(K, 200)))
    # ---- the step before the decode: block-table construction, timed alone
    bt_rows = block_table_measure(w, dev, stream, flush, max(3, min(K, 200)))
    # ---- ragged query counts (draft extend), the same decode kernels
    ragged = ragged_measure(dev, stream, flush, max(3, min(K, 200)), peaks)
    # ---- the same workload planned on the device (planner kernel in the step)
    devplan = device_plan_measure(db, w, dev, stream, flush, max(3, min(K, 200)), st)
    # ---- the step before: RoPE + FP8 quantisation + cache write of the new tokens
    rope_write = rope_write_measure(w, dev, stream, flush, max(3, min(K, 200)), peaks)
    # ---- a serving step that re-plans on the host from the new lengths
    e2e_rp = e2e_replan_measure(db, w, dev, stream, max(3, min(K, 200)))
    plan_us = host_plan_us(w)
    # ---- every other seeded workload, timed the same way
    names = [] if args.configs == "none" else (
        list(W.CONFIGS) if args.configs == "all" else [n for n in args.configs.split(",") if n])
    per_config = {}
    for name in names:
        if name == w.name:
            continue
        per_config[name] = config_measure(name, args.seed + rank, dev, stream, flush, max(3, min(K, 100)), peaks,
                                          peaks_kind)

    if rank != 0:
        return
    main_avg_s = statistics.mean(main_ms) / 1e3
    step_avg_s = statistics.mean(step_ms) / 1e3
    t_hbm = st["alg_bytes"] / (float(peaks["hbm_gbs"]) * 1e9)
    t_tc = st["flops"] / (float(peaks["bf16_tflops"]) * 1e12)
    rl = roofline_of(st, main_avg_s, peaks, peaks_kind, "bf16" if w.kv_dtype == "bf16" else "fp16")
    bound, achieved, peak, unit = rl["bound"], rl["achieved"], rl["peak"], rl["unit"]
    cpu_v, cpu_el, cpu_rows = time_oracle(w, budget_s=args.cpu_seconds)
    clocks = ClockSampler.summarize(clock_rows, peaks)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3-kv/fp16-mma",
        "data": "synthetic", "config": workload_desc(w),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                     "kernel": "main split-KV decode kernel", "peak_kind": peaks_kind,
                     "alg_bytes_per_launch": st["alg_bytes"], "alg_flops_per_launch": st["flops"]},
        "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
                         "sample": f"whole-request float64 oracle passes over the same workload, "
                                   f"{cpu_rows} query tokens in {cpu_el:.1f} s"},
        "e2e": e2e,
        "e2e_serial": e2e_serial,
        "e2e_host_io": e2e_hio,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "kv_gbs": st["kv_bytes"] / step_avg_s / 1e9,
        "tflops": st["flops"] / step_avg_s / 1e12,
        "step_roofline_frac": max(t_hbm, t_tc) / step_avg_s,
        "main_kernel_frac_of_roofline_time": max(t_hbm, t_tc) / main_avg_s,
        "main_ms": statistics.mean(main_ms), "combine_ms": statistics.mean(comb_ms),
        "main_ms_median": statistics.median(main_ms),
        "t_roof_us": {"hbm": t_hbm * 1e6, "tensor": t_tc * 1e6},
        "wall_s_timed_loop": wall,
        "block_table_build": bt_rows,
        "ragged_decode": ragged,
        "graph_replay": {"us_per_step": graph_s * 1e6, "tokens_per_s": st["tokens"] / graph_s,
                         "note": "the same decode step captured once in a CUDA graph and replayed; "
                                 "L2 flushed between replays"},
        "device_plan": devplan,
        "rope_quantize_write": rope_write,
        "segments": int(len(db.plan.segments())), "partial_slots": db.plan.num_partial_slots,
        "host_plan_us": plan_us,
        "e2e_replan": e2e_rp,
        "kernel_source_sha": kernel_source_hash(),
        "configs": per_config,
    }
    print(json.dumps(line), flush=True)


def roofline_of(st, main_s, peaks, peaks_kind, mma="bf16"):
    """Roofline of one main-kernel launch: the slower of the algorithmic
    bytes at the HBM peak and the algorithmic flops at the tensor peak of the
    MMA precision used (bf16 and fp16 MMAs share the measured bf16 rate)."""
    hbm_peak = float(peaks["hbm_gbs"])
    tc_peak = float(peaks["bf16_tflops"])
    t_hbm = st["alg_bytes"] / (hbm_peak * 1e9)
    t_tc = st["flops"] / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        achieved, peak, unit, bound = st["alg_bytes"] / main_s / 1e9, hbm_peak, "GB/s", "hbm"
    else:
        achieved, peak, unit, bound = st["flops"] / main_s / 1e12, tc_peak, "TFLOP/s", "tensor"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "peak_kind": peaks_kind, "mma": mma, "t_roof_us": max(t_hbm, t_tc) * 1e6,
            "alg_bytes_per_launch": st["alg_bytes"], "alg_flops_per_launch": st["flops"]}


def config_measure(name, seed, dev, stream, flush, K, peaks, peaks_kind):
    """One seeded workload timed like the headline step: K decode steps
    (main kernel + combine, L2 flushed before each, events on the launching
    stream), then K steps with an event between the two launches for the
    main kernel's own time; host plan cost; roofline of the main kernel."""
    import torch
    from paged_mla_decode_08_gb300 import runner as R
    w = W.make_workload(name, seed=seed)
    st = W.workload_stats(w)
    db = R.upload(w, device=dev)
    for _ in range(3):
        flush.zero_()
        R.decode(db, stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        R.decode(db, stream)
        ev[k][1].record(stream)
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        evk[k][0].record(stream)
        R.decode_main(db, stream)
        evk[k][1].record(stream)
        R.decode_combine(db, stream)
        evk[k][2].record(stream)
    torch.cuda.synchronize()
    step_s = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    main_s = statistics.mean(e[0].elapsed_time(e[1]) for e in evk) / 1e3
    comb_us = statistics.mean(e[1].elapsed_time(e[2]) for e in evk) * 1e3
    res = {
        "workload": workload_desc(w)["workload"], "tokens_per_s": st["tokens"] / step_s,
        "step_us": step_s * 1e6, "main_us": main_s * 1e6, "combine_us": comb_us,
        "kv_gbs": st["kv_bytes"] / step_s / 1e9, "tflops": st["flops"] / step_s / 1e12,
        "roofline": dict(roofline_of(st, main_s, peaks, peaks_kind, "bf16" if w.kv_dtype == "bf16" else "fp16"),
                         traffic=profiled_traffic(w.name)),
        "step_roofline_frac": roofline_of(st, step_s, peaks, peaks_kind)["frac"],
        "host_plan_us": host_plan_us(w), "segments": int(len(db.plan.segments())),
        "partial_slots": db.plan.num_partial_slots, "steps": K, "launches_per_step": 1 + (db.plan.num_partial_slots > 0),
        "kernel_source_sha": kernel_source_hash(),
    }
    del db
    torch.cuda.empty_cache()
    return res


def host_plan_us(w, reps=200):
    """Mean wall time of one mla_decode_plan call from the host lengths
    (through the Python binding, plan object freed each time)."""
    from paged_mla_decode_08_gb300 import binding as B
    lens = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    B.mla_decode_plan(lens, w.page_size, w.num_heads, w.q_len)
    t0 = time.perf_counter()
    for _ in range(reps):
        p = B.mla_decode_plan(lens, w.page_size, w.num_heads, w.q_len)
        del p
    return (time.perf_counter() - t0) / reps * 1e6


def e2e_replan_measure(db, w, dev, stream, K):
    """The e2e step of a host-planned serving loop: every step makes a new
    plan from the host lengths, then copies the query, block table and
    lengths in, decodes, and reads out and lse back (host-synchronous)."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    hq = db.q_nope.cpu().pin_memory()
    hp = db.q_pe.cpu().pin_memory()
    hbt = db.block_table.cpu().pin_memory()
    hsl = db.seq_lens.cpu().pin_memory()
    lens = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    ho = torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()
    hl = torch.empty(db.lse.shape, dtype=db.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hp, hbt, hsl))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl))

    def one():
        plan = B.mla_decode_plan(lens, w.page_size, w.num_heads, w.q_len)
        db.q_nope.copy_(hq, non_blocking=True)
        db.q_pe.copy_(hp, non_blocking=True)
        db.block_table.copy_(hbt, non_blocking=True)
        db.seq_lens.copy_(hsl, non_blocking=True)
        B.mla_decode(plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens, w.scale,
                     w.k_scale, db.out, db.lse, db.workspace, None, stream)
        ho.copy_(db.out, non_blocking=True)
        hl.copy_(db.lse, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(3):
        one()
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    el = time.perf_counter() - t0
    return {"value": w.num_tokens * K / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "note": "host plan made from the host lengths inside every step; otherwise as e2e"}


def block_table_measure(w, dev, stream, flush, K):
    """Both block-table builders over a request pool holding this workload's
    pages (pool rows = batch + 64), each launch timed with events after an L2
    flush.  Algorithmic bytes: one int32 pool read per live table entry plus
    the row index (and, for the token pool, the length) per request, and the
    whole int32 table written."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    pool = W.make_request_pool(w.block_table, w.seq_lens, w.page_size, pool_rows=w.batch + 64, seed=1)
    r2t = torch.from_numpy(pool.req_to_token).to(dev)
    r2p = torch.from_numpy(pool.req_to_page).to(dev)
    idx = torch.from_numpy(pool.req_pool_indices).to(dev)
    lens = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(dev)
    max_blocks = int(w.block_table.shape[1])
    bt = torch.empty((w.batch, max_blocks), dtype=torch.int32, device=dev)
    live = int(((w.seq_lens.astype(np.int64) + w.page_size - 1) // w.page_size).sum())
    table_bytes = w.batch * max_blocks * 4
    calls = {
        "from_tokens": (lambda: B.mla_block_table_from_tokens(r2t, idx, lens, w.page_size, bt, stream),
                        live * 4 + w.batch * 8 + table_bytes),
        "from_pages": (lambda: B.mla_block_table_from_pages(r2p, idx, bt, stream),
                       w.batch * min(max_blocks, r2p.shape[1]) * 4 + w.batch * 4 + table_bytes),
    }
    res = {}
    for name, (fn, alg) in calls.items():
        for _ in range(3):
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            fn()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        res[name] = {"us": us, "alg_bytes": alg, "achieved_gbs": alg / (us * 1e-6) / 1e9,
                     "bound": "latency", "launches": K}
    want = np.where(np.arange(max_blocks)[None, :] < ((w.seq_lens[:, None] + w.page_size - 1) // w.page_size),
                    w.block_table, 0)
    got = bt.cpu().numpy()
    res["last_table_matches_workload"] = bool(np.array_equal(got, want))
    return res


def graph_step_seconds(launch, dev, stream, flush, K):
    """Capture `launch(capture_stream)` once in a CUDA graph, then time K
    replays on `stream` (L2 flushed before each, outside the events).
    Returns the mean seconds per replay."""
    import torch
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            launch(cap)
    stream.wait_stream(cap)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            graph.replay()
            ev[k][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3


def device_plan_measure(db, w, dev, stream, flush, K, st):
    """The headline decode with a device plan: each step launches the planner
    kernel, the main kernel and the combine (what a CUDA graph captured once
    replays for any lengths).  Timed like the headline step."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    from paged_mla_decode_08_gb300 import runner as R
    plan = B.mla_decode_plan_device(w.batch, w.page_size, w.num_heads, w.q_len)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(db.out)
    lse = torch.empty_like(db.lse)

    def step():
        B.mla_decode(plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens, w.scale,
                     w.k_scale, out, lse, ws, None, stream)

    for _ in range(3):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    s_avg = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    # the two launches apart: planner + main kernel, then the combine
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        evk[k][0].record(stream)
        B.mla_decode_main(plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens, w.scale,
                          w.k_scale, out, lse, ws, None, stream)
        evk[k][1].record(stream)
        B.mla_decode_combine(plan, out, lse, ws, None, stream)
        evk[k][2].record(stream)
    torch.cuda.synchronize()
    main_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evk) * 1e3
    comb_us = statistics.mean(e[1].elapsed_time(e[2]) for e in evk) * 1e3
    # the same step captured once in a CUDA graph and replayed (the use the
    # device plan exists for: no host work and one graph launch per step)
    g_avg = graph_step_seconds(
        lambda cs: B.mla_decode(plan, db.q_nope, db.q_pe, db.kv, db.kv_dtype, db.block_table, db.seq_lens,
                                w.scale, w.k_scale, out, lse, ws, None, cs), dev, stream, flush, K)
    host_out = R.decode(db, stream)[0]
    diff = float((out.float() - host_out.float()).abs().max())  # the two plans split differently
    return {"us_per_step": s_avg * 1e6, "tokens_per_s": st["tokens"] / s_avg,
            "graph_us_per_step": g_avg * 1e6, "graph_tokens_per_s": st["tokens"] / g_avg,
            "planner_plus_main_us": main_us, "combine_us": comb_us,
            "segments": int(len(plan.device_segments(ws))), "launches_per_step": 3,
            "max_abs_diff_vs_host_plan": diff,
            "note": "planner + main + combine per step (eager launches; graph_*: one captured CUDA graph "
                    "replayed per step), L2 flushed between steps"}


def rope_write_measure(w, dev, stream, flush, K, peaks):
    """mla_rope_quantize_cache_write for one decode step of this workload's
    shape (one new token per request, all heads) on the pages' FP8 path:
    merged e4m3 query out, e4m3 key rows into a cache.  Algorithmic bytes:
    the bf16 query and key read once (1152 B per head and per key), the
    e4m3 rows written (576 B each), cos/sin rows and the index arrays."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    t, h = w.batch, w.num_heads
    g = torch.Generator(device=dev).manual_seed(0)
    q_nope = torch.randn((t, h, 512), generator=g, device=dev).to(torch.bfloat16)
    q_rope = torch.randn((t, h, 64), generator=g, device=dev).to(torch.bfloat16)
    k_nope = torch.randn((t, 512), generator=g, device=dev).to(torch.bfloat16)
    k_rope = torch.randn((t, 64), generator=g, device=dev).to(torch.bfloat16)
    max_pos = 8192
    inv = 10000.0 ** (-torch.arange(0, 64, 2, dtype=torch.float64, device=dev) / 64)
    ang = torch.arange(max_pos, dtype=torch.float64, device=dev)[:, None] * inv[None, :]
    cs = torch.cat([ang.cos(), ang.sin()], dim=1).float().contiguous()
    pos = torch.randint(0, max_pos, (t,), generator=g, device=dev, dtype=torch.int64)
    kv = torch.zeros((max(t, 64), w.page_size, 576), dtype=torch.uint8, device=dev)
    slots = torch.randperm(kv.shape[0] * w.page_size, generator=g, device=dev)[:t].to(torch.int64)
    q_out = torch.empty((t, h, 576), dtype=torch.uint8, device=dev)

    def step():
        B.mla_rope_quantize_cache_write(q_nope, q_rope, q_out, B.MLA_Q_E4M3, k_nope, k_rope, pos, cs, False, kv,
                                        B.MLA_KV_E4M3, slots, stream)

    for _ in range(3):
        step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    alg = t * (h + 1) * (1152 + 576) + t * (256 + 16)
    gbs = alg / (us * 1e-6) / 1e9
    return {"us": us, "alg_bytes": alg, "achieved_gbs": gbs, "hbm_frac": gbs / float(peaks["hbm_gbs"]),
            "tokens": t, "heads": h, "launches": K, "note": "e4m3 query + e4m3 cache rows; L2 flushed"}


def ragged_measure(dev, stream, flush, K, peaks):
    """The draft-extend workload (per-request query counts 1..4 packed by
    cu_seqlens_q), one mla_decode_ragged call per step between events after
    an L2 flush; roofline against the same HBM peak as the main line."""
    import torch
    from paged_mla_decode_08_gb300 import runner as R
    w = W.make_ragged_workload("draft_extend", seed=0)
    st = W.workload_stats(w)
    db = R.upload(w, device=dev)
    for _ in range(3):
        R.decode(db, stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        R.decode(db, stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    s_avg = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    gbs = st["alg_bytes"] / s_avg / 1e9
    return {"workload": workload_desc(w)["workload"], "us": s_avg * 1e6, "tokens_per_s": st["tokens"] / s_avg,
            "query_tokens": st["tokens"], "alg_bytes": st["alg_bytes"], "achieved_gbs": gbs,
            "hbm_frac": gbs / float(peaks["hbm_gbs"]), "launches_per_step": 1 + (db.plan.num_partial_slots > 0),
            "note": "decode step incl. combine; L2 flushed between steps"}


def e2e_measure(db, w, dev, stream, K):
    """The same decode through the public API starting from pinned host
    buffers: per step, copy the query, block table and lengths in, decode,
    copy out and lse back, wait for them on the host."""
    import torch
    from paged_mla_decode_08_gb300 import runner as R
    hq = db.q_nope.cpu().pin_memory()
    hp = db.q_pe.cpu().pin_memory()
    hbt = db.block_table.cpu().pin_memory()
    hsl = db.seq_lens.cpu().pin_memory()
    ho = torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory()
    hl = torch.empty(db.lse.shape, dtype=db.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hp, hbt, hsl))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl))

    def one():
        db.q_nope.copy_(hq, non_blocking=True)
        db.q_pe.copy_(hp, non_blocking=True)
        db.block_table.copy_(hbt, non_blocking=True)
        db.seq_lens.copy_(hsl, non_blocking=True)
        R.decode(db, stream)
        ho.copy_(db.out, non_blocking=True)
        hl.copy_(db.lse, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(3):
        one()
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    el = time.perf_counter() - t0
    return {"value": w.num_tokens * K / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "note": "host-synchronous per step, L2 not flushed; KV cache resident in HBM"}


def e2e_pipelined_measure(db, w, dev, stream, K, sets=4):
    """The e2e step with the host link overlapped: `sets` sets of per-step
    buffers; step k's inputs are copied in on one stream while earlier steps
    decode, and step k - 1's results are copied out on a third stream while
    step k decodes.  Every step still moves its own query, block table and
    lengths in and its output and lse out through pinned host memory; a
    step's inputs travel as one copy and its results as one (the tensors are
    views of one buffer each), and the host waits for every result copy (a
    step's buffers are reused `sets` steps later, after the host has its
    results).  The sets are independent batches in flight, as a server
    interleaving micro-batches has them.  With two sets the host's wait for
    step k - 2's results sits between step k - 1's decode and step k's copy
    in, and the decode stalls on that chain (100 us a step on the
    DeepSeek-V3-shaped batch); three sets give it one decode of slack (72.5
    us) and four hide the copies entirely (69.4 us, against 70.9 us for the
    decode alone while both copies run)."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B

    def packed(tensors, pinned):
        """One byte buffer holding `tensors` back to back (256-byte aligned),
        and views of it shaped like them."""
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-(t.numel() * t.element_size()) // 256) * 256
        buf = torch.empty(n, dtype=torch.uint8, device="cpu" if pinned else dev)
        if pinned:
            buf = buf.pin_memory()
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
        return buf, views

    ins = (db.q_nope, db.q_pe, db.block_table, db.seq_lens)
    outs = (db.out, db.lse)
    h_in, d_in, h_out, d_out = [], [], [], []
    for _ in range(sets):
        hb, hv = packed(ins, True)
        for v, t in zip(hv, ins):
            v.copy_(t.cpu())
        h_in.append((hb, hv))
        d_in.append(packed(ins, False))
        h_out.append(packed(outs, True))
        d_out.append(packed(outs, False))
    ws = [torch.empty_like(db.workspace) for _ in range(sets)]
    h2d = int(h_in[0][0].numel())
    d2h = int(h_out[0][0].numel())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(sets)]
    ev_dec = [torch.cuda.Event() for _ in range(sets)]
    ev_out = [torch.cuda.Event() for _ in range(sets)]

    def run(n):
        for k in range(n):
            i = k % sets
            if k >= sets:
                ev_out[i].synchronize()  # the host has step k - sets's results; its buffers are free
                s_in.wait_event(ev_dec[i])  # step k - sets no longer reads set i
            with torch.cuda.stream(s_in):
                d_in[i][0].copy_(h_in[i][0], non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            q, qp, bt, sl = d_in[i][1]
            o, l = d_out[i][1]
            B.mla_decode(db.plan, q, qp, db.kv, db.kv_dtype, bt, sl, w.scale, w.k_scale, o, l, ws[i], None, stream)
            ev_dec[i].record(stream)
            s_out.wait_event(ev_dec[i])
            with torch.cuda.stream(s_out):
                h_out[i][0].copy_(d_out[i][0], non_blocking=True)
            ev_out[i].record(s_out)
        for e in ev_out:
            e.synchronize()

    run(2 * sets)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(K)
    el = time.perf_counter() - t0
    last = h_out[(K - 1) % sets][1][0]
    same = bool(torch.equal(last.view(torch.int16).to(dev), db.out.view(torch.int16)))
    return {"value": w.num_tokens * K / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "result_matches_device_decode": same, "buffer_sets": sets,
            "note": f"copies of later steps in and step k-1 out overlap the decode of step k (three streams; "
                    f"{sets} buffer sets = {sets} independent batches in flight; one copy each way per step); "
                    f"L2 not flushed (the 191 MB KV stream exceeds it); KV cache resident in HBM"}


def e2e_host_io_measure(db, w, dev, stream, K, sets=4):
    """The e2e step through mla_decode_host_io, the call that takes the step's
    inputs from host memory and returns its results there: `sets` sets of
    buffers (pinned host and device) on as many streams, in turn, so one
    step's copies overlap the other steps' decodes.  Every step still moves
    its own query, block table and lengths in and its output and lse out;
    the host waits for a step's results before reusing its buffers `sets`
    steps later."""
    import torch
    from paged_mla_decode_08_gb300 import binding as B
    ins = (db.q_nope, db.q_pe, db.block_table, db.seq_lens)
    outs = (db.out, db.lse)
    h_in = [[t.cpu().pin_memory() for t in ins] for _ in range(sets)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] for _ in range(sets)]
    d_in = [[torch.empty_like(t) for t in ins] for _ in range(sets)]
    d_out = [[torch.empty_like(t) for t in outs] for _ in range(sets)]
    ws = [torch.empty_like(db.workspace) for _ in range(sets)]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0])
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    streams = [torch.cuda.Stream(device=dev) for _ in range(sets)]
    done = [torch.cuda.Event() for _ in range(sets)]

    def run(n):
        for k in range(n):
            i = k % sets
            if k >= sets:
                done[i].synchronize()  # the host holds step k - sets's results; set i is free
            q, qp, bt, sl = d_in[i]
            o, l = d_out[i]
            hq, hqp, hbt, hsl = h_in[i]
            ho, hl = h_out[i]
            B.mla_decode_host_io(db.plan, q, qp, db.kv, db.kv_dtype, bt, sl, w.scale, w.k_scale, o, l, ws[i],
                                 hq, hqp, hbt, hsl, ho, hl, streams[i])
            done[i].record(streams[i])
        for e in done:
            e.synchronize()

    run(2 * sets)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(K)
    el = time.perf_counter() - t0
    same = bool(torch.equal(h_out[(K - 1) % sets][0].view(torch.int16).to(dev), db.out.view(torch.int16)))
    return {"value": w.num_tokens * K / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "result_matches_device_decode": same,
            "call": "mla_decode_host_io", "buffer_sets": sets,
            "note": f"{sets} buffer sets on {sets} streams, in turn: one step's copies overlap the other "
                    f"steps' decodes; L2 not flushed; KV cache resident in HBM"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="dsv3", choices=list(W.CONFIGS))
    ap.add_argument("--seed", type=int, default=0, help="workload seed (rank r draws seed + r)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed steps before timing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="host time for the cpu_baseline sample of the oracle")
    ap.add_argument("--configs", default="all",
                    help="seeded workloads measured besides the headline one, into the line's 'configs' object: "
                         "'all' (default), 'none', or a comma-separated list of names")
    ap.add_argument("--profile", action="store_true",
                    help="run --warmup + 1 decode steps of --config and exit: a small, fixed launch sequence "
                         "for ncu captures (no timing, no JSON line)")
    ap.add_argument("--pool-pages", type=int, default=0,
                    help="with --profile: cache pool size in pages (0 = the workload's); the decode reads the "
                         "same pages either way, and a smaller pool keeps a capture's device memory small")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    # weak scaling: every rank decodes its own batch of the same shape
    extra = {"pool_pages": args.pool_pages} if (args.profile and args.pool_pages) else {}
    w = W.make_workload(args.config, seed=args.seed + rank, **extra)
    if args.impl == "reference":
        reference_arm(args, w, rank)
        return
    if args.profile:
        profile_run(args, w)
        return
    our_arm(args, w, rank, world)


def profile_run(args, w):
    """The launch sequence ncu captures: (warmup + 1) x [L2 flush, mla_decode]
    on the configured workload (main kernel then combine per step)."""
    import torch
    from paged_mla_decode_08_gb300 import runner as R
    from paged_mla_decode_08_gb300.build import build
    build()
    db = R.upload(w)
    flush = torch.empty(2 * int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20)),
                        dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup + 1):
        flush.zero_()
        R.decode(db)
    torch.cuda.synchronize()
    print(f"profile run: {args.warmup + 1} decode steps of {w.name}", flush=True)


if __name__ == "__main__":
    main()
