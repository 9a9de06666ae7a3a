"""Benchmark of one paged decode step on GB300.

A step is the whole hot path over one batch: copy-on-write block copies,
the new tokens' K/V writes, and the paged decode attention (split-KV with a
log-sum-exp merge).

Metric: KV bytes the step must read (sum of lengths x kv heads x head_dim x
2 bytes x K,V) per second of device time, plus tokens attended per second.

With no workload flag, one line is printed per measured case (the block
copy and the cache write on their own, every decode workload, the fp8
cache, beam search, chunked prefill, swap) and the LAST line is the headline:
the largest single-GPU decode workload, the fragmented MHA batch (256
sequences of up to 4096 tokens, 32 query = 32 kv heads, head_dim 128, bf16,
block 16, 8.6 GB of KV), with the roofline, the CPU baseline (the oracle)
and the end-to-end figure.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 1..6] [--block-size 8|16|32] [--kv bf16|fp8]
                    [--op decode|write|copy|prefill|swap]

With --kv fp8 the pools hold E4M3 codes (one byte per element, per-tensor
scales): the same step through the fp8 entry points, KV bytes halved.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV-read HBM GB/s (% of peak), tokens attended/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
KERNEL_SOURCES = ["paged_kv_cache_105_gb300/csrc/pa_decode.cu",
                  "paged_kv_cache_105_gb300/csrc/pa_ptx.cuh"]
PREFILL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_traffic.txt")
PREFILL_SOURCES = ["paged_kv_cache_105_gb300/csrc/pa_prefill.cu",
                   "paged_kv_cache_105_gb300/csrc/pa_tc.cuh",
                   "paged_kv_cache_105_gb300/csrc/pa_ptx.cuh"]
FALLBACK_HBM_GBS = 6800.0
# The headline: the largest single-GPU decode workload (the fragmented MHA
# batch, 8.6 GB of KV at block size 16).
HEADLINE = (3, 16)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5, 6],
                   help="one decode workload (default: every case, the headline last)")
    p.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32])
    p.add_argument("--partition-tokens", type=int, default=None)
    p.add_argument("--num-seqs", type=int, default=None,
                   help="configs 2-5: a smaller batch of the same shape (profiling)")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--op", choices=["decode", "write", "copy", "swap", "prefill"],
                   default="decode",
                   help="decode: the decode step (default); write: the cache write alone "
                        "(the GQA batch's new tokens); copy: the copy-on-write block copy "
                        "alone (the prefix-sharing batch's pairs); swap: block swap-out to "
                        "pinned host memory and swap-in back; prefill: a chunked-prefill step")
    p.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                   help="KV cache element type (fp8: E4M3 codes with per-tensor scales)")
    p.add_argument("--eager", action="store_true",
                   help="launch every call from Python instead of replaying CUDA graphs")
    return p.parse_args()


def build_workload(cfg, bs, num_seqs=None):
    """Config `cfg`; num_seqs shrinks configs 2-5 to a smaller batch of the
    same shape (for profiling captures that must stay small)."""
    from paged_kv_cache_105_gb300 import workloads as W
    kw = {} if num_seqs is None else {"num_seqs": num_seqs}
    if num_seqs is not None and cfg not in (2, 3, 4, 5):
        raise SystemExit("--num-seqs applies to configs 2-5")
    if cfg == 3:
        return W.config3(block_size=bs, **kw)
    if kw:
        return {2: W.config2, 4: W.config4, 5: W.config5}[cfg](**kw)
    return W.CONFIGS[cfg]()


def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def max_over_ranks(x, world, device):
    """The largest x over the ranks: the job takes as long as its slowest
    rank. Collective: every rank calls it, with world > 1 under an initialised
    process group (NCCL on the GPUs; gloo works for CPU tensors)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units all ranks processed per second: each of the `world` replicas does
    the same work, and `seconds` is the slowest rank's time."""
    return world * units_per_rank / seconds


def _code_tokens(text):
    """C/CUDA source without its comments and blank space: what the compiler
    sees, so that a comment edit does not invalidate a recorded capture."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_tokens(fh.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload_name, path=TRAFFIC_FILE, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from a committed ncu summary (decode by default),
    if it was taken on this workload with the current kernel source."""
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    key = f"traffic_bytes_per_launch[{workload_name}]"
    if kv.get("kernel_source_sha256") != kernel_hash(sources) or key not in kv:
        return None
    return float(kv[key])


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        if j.get("hbm_gbs"):
            return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _bits(t):
    import numpy as np
    import torch
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def cpu_oracle_step(wl, vals_cpu, seqs, fp8_scale=None, threads=1):
    """The oracle's copy -> write -> attention for the sequences `seqs`
    (a bounded sample of the workload); fp8_scale: E4M3 pools with that
    scale for K and V. threads > 1: the attention's (sequence, head) rows are
    split across that many threads (the oracle's calls release the GIL).
    Returns KV bytes of the sample."""
    import numpy as np
    from oracle import paref
    bits = _bits
    rows = np.array([(s, h) for s in seqs for h in range(wl.n_q_heads)], np.int32)
    if threads > 1:
        from concurrent.futures import ThreadPoolExecutor
        chunks = [c for c in np.array_split(rows, threads) if len(c)]
        attend = paref.attention_paged_fp8 if fp8_scale is not None else paref.attention_paged
        extra = (fp8_scale, fp8_scale) if fp8_scale is not None else ()

        def attention(q, kp, vp, bt, sl, scale, *sc, rows):
            with ThreadPoolExecutor(len(chunks)) as ex:
                list(ex.map(lambda c: attend(q, kp, vp, bt, sl, scale, *sc, rows=c), chunks))
    else:
        attention = None
    ntok = int(wl.seq_lens[list(seqs)].astype(np.int64).sum())
    if fp8_scale is not None:
        kp, vp = vals_cpu["k_pool"].numpy().copy(), vals_cpu["v_pool"].numpy().copy()
        paref.copy_blocks(kp.view(np.uint16), vp.view(np.uint16), wl.cow_pairs)
        paref.reshape_and_cache_fp8(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                                    wl.slot_mapping, fp8_scale, fp8_scale)
        (attention or paref.attention_paged_fp8)(bits(vals_cpu["q"]), kp, vp, wl.block_tables,
                                                 wl.seq_lens, wl.scale, fp8_scale, fp8_scale,
                                                 rows=rows)
        return ntok * wl.n_kv_heads * wl.head_dim * 1 * 2
    kp, vp = bits(vals_cpu["k_pool"]).copy(), bits(vals_cpu["v_pool"]).copy()
    paref.copy_blocks(kp, vp, wl.cow_pairs)
    paref.reshape_and_cache(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                            wl.slot_mapping)
    (attention or paref.attention_paged)(bits(vals_cpu["q"]), kp, vp, wl.block_tables,
                                         wl.seq_lens, wl.scale, rows=rows)
    return ntok * wl.n_kv_heads * wl.head_dim * 2 * 2


def cpu_sample_seqs(wl, budget_tokens):
    """Sequences (longest last) whose total length stays within a budget."""
    import numpy as np
    order = np.random.default_rng(0).permutation(wl.num_seqs)
    picked, tot = [], 0
    for s in order:
        L = int(wl.seq_lens[s])
        if picked and tot + L > budget_tokens:
            continue
        picked.append(int(s))
        tot += L
    return sorted(picked), tot


def run_reference(args):
    """The oracle as the reference arm, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = HEADLINE[0] if args.config is None else args.config
    bs = HEADLINE[1] if args.config is None else args.block_size
    wl = build_workload(cfg, bs, args.num_seqs)
    if hasattr(wl, "steps"):  # multi-step workload: the oracle times its first step
        wl = wl.steps[0]
    budget = 6000 if wl.n_q_heads * wl.head_dim >= 4096 else 20000
    seqs, tok = cpu_sample_seqs(wl, budget)
    fp8 = fp8_scale_of(args)
    vals = W_make_values_subset(wl, seqs, fp8=fp8 is not None)
    for _ in range(max(0, args.warmup)):
        cpu_oracle_step(vals["wl"], vals["vals"], vals["seqs"], fp8)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += cpu_oracle_step(vals["wl"], vals["vals"], vals["seqs"], fp8)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "kv_dtype": args.kv, "sample_seqs": len(seqs),
                       "sample_tokens": tok},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{len(seqs)} of {wl.num_seqs} sequences "
                                       f"({tok} tokens) per step, all query heads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def fp8_scale_of(args):
    if args.kv != "fp8":
        return None
    from paged_kv_cache_105_gb300 import workloads as W
    return W.FP8_SCALE


def W_make_values_subset(wl, seqs, fp8=False):
    """A self-contained sub-workload holding only `seqs` (tables remapped
    onto a compact pool), with values drawn for exactly those blocks, so the
    CPU baseline never allocates the full pool on the host."""
    import numpy as np
    from paged_kv_cache_105_gb300 import workloads as W
    bs = wl.block_size
    pair_src = {int(d): int(s) for s, d in wl.cow_pairs}
    need = []
    for s in seqs:
        nb = -(-int(wl.seq_lens[s]) // bs)
        for b in wl.block_tables[s, :nb]:
            need.append(int(b))
            if int(b) in pair_src:
                need.append(pair_src[int(b)])
    ids = list(dict.fromkeys(need))
    remap = {b: i for i, b in enumerate(ids)}
    maxb = wl.block_tables.shape[1]
    bt = np.full((len(seqs), maxb), -1, np.int32)
    slots, pairs = [], []
    for i, s in enumerate(seqs):
        nb = -(-int(wl.seq_lens[s]) // bs)
        bt[i, :nb] = [remap[int(b)] for b in wl.block_tables[s, :nb]]
        sl = int(wl.slot_mapping[s])
        slots.append(-1 if sl < 0 else remap[sl // bs] * bs + sl % bs)
        last = int(wl.block_tables[s, (int(wl.seq_lens[s]) - 1) // bs]) if nb else -1
        if last in pair_src:
            pairs.append((remap[pair_src[last]], remap[last]))
    sub = W.Workload(name=wl.name + "-sample", num_seqs=len(seqs), n_q_heads=wl.n_q_heads,
                     n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim, block_size=bs,
                     num_blocks=max(1, len(ids)), seq_lens=wl.seq_lens[seqs].astype(np.int32),
                     block_tables=bt, slot_mapping=np.array(slots, np.int32),
                     cow_pairs=np.array(pairs, np.int32).reshape(-1, 2),
                     free_order=np.arange(max(1, len(ids)), dtype=np.int32), seed=wl.seed)
    vals = W.make_values_fp8(sub, device="cpu") if fp8 else W.make_values(sub, device="cpu")
    return {"wl": sub, "vals": vals, "seqs": list(range(len(seqs)))}


class Env:
    """The process's GPU, rank and library, set up once for every line."""

    def __init__(self, args):
        import torch
        self.world, self.rank, self.local = dist_init(args)
        self.dev = torch.device("cuda", self.local)
        torch.cuda.set_device(self.dev)
        import __graft_entry__
        __graft_entry__.build()
        self.l2 = torch.cuda.get_device_properties(self.dev).L2_cache_size

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()


def release():
    """Free the device memory of the line just measured before the next."""
    import gc
    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


class L2Flush:
    """Between timed launches of a small kernel: a write over twice the L2
    size, then a read of it (torch kernels), so that the kernel starts from
    cold data and the L2 holds no dirty lines whose write-back would compete
    with it."""

    def __init__(self, env):
        import torch
        self.buf = torch.empty(2 * env.l2 // 4, dtype=torch.int32, device=env.dev)
        self.sink = torch.empty((), dtype=torch.int32, device=env.dev)

    def __call__(self):
        import torch
        self.buf.fill_(1)
        torch.amax(self.buf, dim=0, out=self.sink)


def time_small_kernel(env, fn, reps):
    """Median CUDA-event time (ms) of one launch of `fn` after an L2 flush,
    over `reps` launches, on the current stream."""
    import torch
    flush = L2Flush(env)
    stream = torch.cuda.current_stream(env.dev)
    for _ in range(5):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def small_op_line(args, env, what, wl, bytes_moved, ms, launches, note, kernel):
    peak, peak_kind = measured_peak()
    ms = max_over_ranks(ms, env.world, env.dev)
    gbs = whole_job_rate(bytes_moved, env.world, ms * 1e-3) / 1e9
    return {"metric": f"{what} read+write GB/s", "value": gbs, "unit": "GB/s",
            "n_gpus": env.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8 (bit copy)", "data": "synthetic",
            "config": {"workload": wl.name, "bytes_per_launch": bytes_moved,
                       "l2": "L2 flushed (a 2x L2 write, then a read of it) before every "
                             "timed launch",
                       "timing": f"median of {args.steps} launches, CUDA events around each"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None, "kernel": kernel,
                         "peak_source": f"{peak_kind} hbm_gbs", "note": note},
            "gpu_launches": launches}


def run_write(args, env):
    """a2 alone: the GQA batch's new tokens written into their slots."""
    import numpy as np
    import torch
    from paged_kv_cache_105_gb300 import binding as B
    from paged_kv_cache_105_gb300 import workloads as W
    wl = W.config2()
    vals = W.make_values(wl, device=env.dev)
    sm = torch.from_numpy(np.ascontiguousarray(wl.slot_mapping)).to(env.dev)
    err = torch.zeros(1, dtype=torch.int32, device=env.dev)

    def fn():
        B.pa_reshape_and_cache(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"], sm,
                               err_word=err)

    ms = time_small_kernel(env, fn, args.steps)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")
    row = wl.n_kv_heads * wl.head_dim * 2
    nbytes = 2 * 2 * wl.num_seqs * row + 4 * wl.num_seqs  # K, V read and written; slots
    us = ms * 1e3
    note = (f"launch-bound: {nbytes / 1e3:.0f} kB per launch would take "
            f"{nbytes / (measured_peak()[0] * 1e3):.2f} us at the copy peak; the launch "
            f"and its latency take the rest of {us:.1f} us")
    line = small_op_line(args, env, "reshape_and_cache (new tokens' K/V into the pool)", wl,
                         nbytes, ms, args.steps, note, "reshape_and_cache_kernel (pa_reshape_and_cache)")
    line["config"]["tokens"] = wl.num_seqs
    return line


def run_copy(args, env):
    """a1 alone: the prefix-sharing batch's copy-on-write block copies."""
    import numpy as np
    import torch
    from paged_kv_cache_105_gb300 import binding as B
    from paged_kv_cache_105_gb300 import workloads as W
    wl = W.config4()
    vals = W.make_values(wl, device=env.dev)
    pairs = torch.from_numpy(np.ascontiguousarray(wl.cow_pairs.reshape(-1, 2))).to(env.dev)
    err = torch.zeros(1, dtype=torch.int32, device=env.dev)

    def fn():
        B.pa_copy_blocks(vals["k_pool"], vals["v_pool"], pairs, err_word=err)

    ms = time_small_kernel(env, fn, args.steps)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")
    n = int(wl.cow_pairs.shape[0])
    block = wl.n_kv_heads * wl.block_size * wl.head_dim * 2
    nbytes = 2 * 2 * n * block + 8 * n  # K and V blocks read and written; pairs
    note = (f"{n} pairs, {nbytes / 1e6:.1f} MB per launch: {nbytes / (measured_peak()[0] * 1e3):.2f}"
            f" us at the copy peak; launch latency is a large share of {ms * 1e3:.1f} us")
    line = small_op_line(args, env, "copy_blocks (copy-on-write block copies)", wl, nbytes, ms,
                         args.steps, note, "copy_blocks_kernel (pa_copy_blocks)")
    line["config"]["pairs"] = n
    return line


def run_swap(args, env):
    """Preemption by swapping: every block the workload's tables use goes to a
    pinned host pool (swap-out) and comes back to the same ids (swap-in);
    one step = both. Compared with the copy engine moving the same bytes as
    one contiguous buffer each way (torch copy_, device <-> pinned host)."""
    import numpy as np
    import torch
    from paged_kv_cache_105_gb300 import binding as B
    from paged_kv_cache_105_gb300 import workloads as W
    dev = env.dev
    cfg = 2 if args.config is None else args.config
    wl = build_workload(cfg, args.block_size, args.num_seqs)
    fp8 = fp8_scale_of(args)
    vals = W.make_values_fp8(wl, device=dev) if fp8 is not None else W.make_values(wl, device=dev)
    gk, gv = vals["k_pool"], vals["v_pool"]
    ids = np.unique(wl.block_tables[wl.block_tables >= 0]).astype(np.int32)
    n = len(ids)
    hk = torch.empty((n,) + tuple(gk.shape[1:]), dtype=gk.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = torch.from_numpy(np.stack([ids, np.arange(n, dtype=np.int32)], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), ids], 1)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    block_bytes = gk[0].numel() * gk.element_size()
    moved = 2 * 2 * n * block_bytes  # K and V, out and in
    stream = torch.cuda.current_stream(dev)

    def step():
        B.pa_swap_blocks(hk, hv, gk, gv, out_pairs, err_word=err)
        B.pa_swap_blocks(gk, gv, hk, hv, in_pairs, err_word=err)

    dbuf = torch.empty(2 * n * block_bytes, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(dbuf.shape, dtype=torch.uint8).pin_memory()

    def ce_step():
        hbuf.copy_(dbuf, non_blocking=True)
        dbuf.copy_(hbuf, non_blocking=True)

    clocks = ClockSampler(env.local)
    clocks.start()
    res = {}
    for name, fn in (("kernel", step), ("copy_engine", ce_step)):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")
    res = {k: max_over_ranks(v, env.world, dev) for k, v in res.items()}
    world = env.world
    gbs = whole_job_rate(moved, world, res["kernel"] * 1e-3) / 1e9
    ce = whole_job_rate(moved, world, res["copy_engine"] * 1e-3) / 1e9
    return {"metric": "KV block swap, device <-> pinned host (out + in) GB/s", "value": gbs,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["kernel"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8 (byte copy)", "data": "synthetic",
            "config": {"workload": wl.name, "kv_dtype": args.kv, "blocks": n,
                       "block_bytes": block_bytes, "bytes_per_step": moved,
                       "l2": f"{moved / 2e6:.0f} MB per direction vs {env.l2 / 1e6:.0f} MB L2"},
            "roofline": {"bound": "chip-to-chip link", "achieved": gbs, "peak": ce,
                         "unit": "GB/s", "frac": gbs / ce, "traffic": None,
                         "kernel": "swap_blocks_kernel (pa_swap_blocks) x2",
                         "peak_source": "copy engine moving the same bytes as one contiguous "
                                        "buffer each way, measured in this run"},
            "gpu_launches": 2 * args.steps, "clocks": clk}


def run_prefill(args, env):
    """One chunked-prefill step = the chunk tokens' cache write + causal
    attention of every chunk token over its whole paged context. Metric:
    causal attention flops per second (4 * head_dim * query heads per visible
    (token, position) pair) against the measured bf16 tensor peak."""
    import numpy as np
    import torch
    from paged_kv_cache_105_gb300 import binding as B
    from paged_kv_cache_105_gb300 import workloads as W
    dev = env.dev
    wl = W.prefill_chunked()
    vals = W.make_prefill_values(wl, device=dev)
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).to(dev)
         for k in ("block_tables", "seq_lens", "cu_q", "slot_mapping")}
    out = torch.empty_like(vals["q"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def write():
        B.pa_reshape_and_cache(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                               t["slot_mapping"], err_word=err)

    def attend():
        B.pa_prefill(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                     t["seq_lens"], t["cu_q"], wl.scale, max_q_len=wl.max_q_len, err_word=err)

    write()
    attend()
    torch.cuda.synchronize()
    gs, ga = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(gs, stream=cap):
        write()
        attend()
    with torch.cuda.graph(ga, stream=cap):
        attend()
    torch.cuda.synchronize()
    clocks = ClockSampler(env.local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        gs.replay()
    torch.cuda.synchronize()
    t_pre = time.perf_counter()
    while time.perf_counter() - t_pre < 1.0:
        gs.replay()
        torch.cuda.synchronize()
    env.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        gs.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    env.barrier()
    # the prefill kernel alone: one event pair around 4 back-to-back replays,
    # repeated; the median per launch
    inner, reps = 4, max(20, min(50, args.steps))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a_, b_ in evs:
        a_.record(stream)
        for _ in range(inner):
            ga.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")
    world = env.world
    step_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    att_ms = statistics.median(a_.elapsed_time(b_) / inner for a_, b_ in evs)
    flops = wl.flops()
    value = whole_job_rate(flops, world, step_ms * 1e-3) / 1e12
    achieved = flops / (att_ms * 1e-3) / 1e12
    peak, kind = None, "fallback"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peak = json.load(f).get("bf16_tflops")
            kind = "measured"
    if not peak:
        peak = 1900.0
    return {"metric": "chunked-prefill causal attention TFLOP/s", "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "batched_tokens": wl.total_q,
                       "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads,
                       "head_dim": wl.head_dim, "block_size": wl.block_size,
                       "flops_per_step": flops, "kv_bytes": wl.kv_bytes(),
                       "arithmetic": "bf16 tcgen05.mma (M 128), fp32 accumulation in TMEM; "
                                     "P as a bf16 hi + lo pair read from TMEM, so the P V "
                                     "product runs twice",
                       "launch": "one CUDA graph replay per step (write, prefill)"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(wl.name, PREFILL_TRAFFIC_FILE,
                                                     PREFILL_SOURCES),
                         "kernel": "prefill_tc_kernel (pa_prefill)",
                         "peak_source": f"{kind} bf16_tflops (cuBLAS, burst)",
                         "timing": f"one CUDA event pair around {inner} back-to-back "
                                   f"prefill-only graph replays, median of {reps}",
                         "prefill_ms": att_ms},
            "gpu_launches": 2 * args.steps, "clocks": clk}


def run_decode(args, env, cfg, bs, kv="bf16", partition_tokens=None, num_seqs=None,
               cpu_baseline=False, e2e_steps=None):
    """The decode step of workload `cfg` (copy-on-write copies, the new
    tokens' writes, the decode and its merge) timed K times; returns the
    JSON line (rank 0) or None."""
    import numpy as np
    import torch
    from paged_kv_cache_105_gb300 import binding as B
    from paged_kv_cache_105_gb300 import workloads as W
    world, rank, dev = env.world, env.rank, env.dev

    # A workload is a list of decode steps over one pool: one step for the
    # single-step batches, T steps (forks, frees, copy-on-write between them)
    # for beam search; the timed steps cycle through them.
    wl0 = build_workload(cfg, bs, num_seqs)
    multi = isinstance(wl0, W.MultiStep)
    steps_wl = wl0.steps if multi else [wl0]
    wl = steps_wl[0]
    name = wl0.name
    T = len(steps_wl)
    fp8 = W.FP8_SCALE if kv == "fp8" else None
    P = wl.partition_tokens if partition_tokens is None else partition_tokens
    if fp8 is not None:
        P = 0  # the fp8 decode always runs the balanced split
    msl = max(w.max_seq_len for w in steps_wl)
    P_res = B.pa_decode_partition_tokens(wl.num_seqs, wl.n_kv_heads, wl.block_size, msl, P)
    eb = 1 if fp8 is not None else 2  # bytes per cached element
    base = W.make_values_fp8(wl, device=dev) if fp8 is not None else W.make_values(wl, device=dev)
    step_vals = ([{k: base[k] for k in ("q", "k_new", "v_new")}] if not multi else
                 [W.make_step_values(w, device=dev) for w in steps_wl])
    pools0 = {k: base[k] for k in ("k_pool", "v_pool")}
    pool_bytes = 2 * base["k_pool"].numel() * eb
    l2 = env.l2
    kv_min = min(w.kv_bytes(eb) for w in steps_wl)
    replicas = 1 if multi else max(1, math.ceil(3 * l2 / max(1, kv_min)))
    replicas = min(replicas, max(1, int(40e9 // max(1, pool_bytes))))
    reps = [pools0] + [{k: v.clone() for k, v in pools0.items()} for _ in range(replicas - 1)]
    maxw = max(w.block_tables.shape[1] for w in steps_wl)

    def idx_tensors(w, to):
        bt = np.full((w.num_seqs, maxw), W.PAD, np.int32)
        bt[:, :w.block_tables.shape[1]] = w.block_tables
        return {"bt": to(bt), "sl": to(w.seq_lens), "sm": to(w.slot_mapping),
                "pairs": to(np.ascontiguousarray(w.cow_pairs.reshape(-1, 2)))}

    tix = [idx_tensors(w, lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev))
           for w in steps_wl]
    outs = [torch.empty_like(base["q"]) for _ in reps]
    wss = [B.decode_workspace(wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                              wl.block_size, msl, P, device=dev) for _ in reps]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    npairs = [int(w.cow_pairs.shape[0]) for w in steps_wl]
    max_parts = 1 if P == 0 else -(-max(1, msl) // P)
    merge = 1 if (P == 0 or max_parts > 1) else 0
    launches = [(1 if npairs[k] else 0) + 2 + merge for k in range(T)]
    stream = torch.cuda.current_stream(dev)

    def api_write(r, k, pairs, k_new, v_new, sm):
        if fp8 is not None:
            if npairs[k]:
                B.pa_copy_blocks_fp8(r["k_pool"], r["v_pool"], pairs, err_word=err)
            B.pa_reshape_and_cache_fp8(k_new, v_new, r["k_pool"], r["v_pool"], sm, fp8, fp8,
                                       err_word=err)
            return
        if npairs[k]:
            B.pa_copy_blocks(r["k_pool"], r["v_pool"], pairs, err_word=err)
        B.pa_reshape_and_cache(k_new, v_new, r["k_pool"], r["v_pool"], sm, err_word=err)

    def api_decode(out, q, r, bt, sl, ws):
        if fp8 is not None:
            B.pa_decode_fp8(out, q, r["k_pool"], r["v_pool"], bt, sl, wl.scale, fp8, fp8,
                            max_seq_len=msl, workspace=ws, err_word=err)
        else:
            B.pa_decode(out, q, r["k_pool"], r["v_pool"], bt, sl, wl.scale, max_seq_len=msl,
                        workspace=ws, partition_tokens=P, err_word=err)

    def calls_write(j, k):
        sv, ti = step_vals[k], tix[k]
        api_write(reps[j], k, ti["pairs"], sv["k_new"], sv["v_new"], ti["sm"])

    def calls_decode(j, k):
        ti = tix[k]
        api_decode(outs[j], step_vals[k]["q"], reps[j], ti["bt"], ti["sl"], wss[j])

    def which(i):
        return i % replicas, i % T

    # Eager warm-up (also the library's one-time set-up), then, unless
    # --eager, CUDA graphs per (replica, step): the whole step (the decode is
    # a programmatic dependent of the cache write, so their launches overlap)
    # and the decode alone, as a serving engine replays its decode step.
    for i in range(replicas * T):
        calls_write(*which(i))
        calls_decode(*which(i))
    torch.cuda.synchronize()
    graphs = None
    if not args.eager:
        graphs = {}
        cap = torch.cuda.Stream(dev)
        for j in range(replicas):
            for k in range(T):
                gs, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=cap):
                    calls_write(j, k)
                    calls_decode(j, k)
                with torch.cuda.graph(gd, stream=cap):
                    calls_decode(j, k)
                graphs[(j, k)] = (gs, gd)
        torch.cuda.synchronize()

    def step(i, ev=None):
        j, k = which(i)
        if graphs is not None:
            graphs[(j, k)][0].replay()
            return
        calls_write(j, k)
        if ev is not None:
            ev[0].record(stream)
        calls_decode(j, k)
        if ev is not None:
            ev[1].record(stream)

    # Warm up with continuous load long enough for the clock sampler to see it.
    clocks = ClockSampler(env.local)
    clocks.start()
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    t_pre = time.perf_counter()
    i = 0
    while time.perf_counter() - t_pre < 1.0:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()
    env.barrier()
    torch.cuda.synchronize()
    dec_ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if graphs is None else [None] * args.steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(k, dec_ev[k])
    t1.record(stream)
    torch.cuda.synchronize()
    env.barrier()
    # The decode on its own, for the roofline: one event pair around `inner`
    # back-to-back decode-only graph replays (cycling the replicas, so every
    # launch reads cold data), repeated; per repeat the algorithmic bytes of
    # its launches over its time, and the median over the repeats.
    inner = max(replicas, 8)
    roof_reps = 50
    roof = []
    if graphs is not None:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(roof_reps)]
        idx = 0
        groups = []
        for a_, b_ in evs:
            a_.record(stream)
            g = []
            for _ in range(inner):
                graphs[which(idx)][1].replay()
                g.append(idx)
                idx += 1
            b_.record(stream)
            groups.append(g)
        torch.cuda.synchronize()
        for (a_, b_), g in zip(evs, groups):
            ms = a_.elapsed_time(b_)
            nb = sum(steps_wl[which(x)[1]].kv_bytes(eb) + steps_wl[which(x)[1]].io_bytes()
                     for x in g)
            roof.append((ms / inner, nb / (ms * 1e-3) / 1e9))
    # keep the load on a little past the timed region for the sampler
    t_post = time.perf_counter()
    while time.perf_counter() - t_post < 0.3:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()
    clk = clocks.stop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)

    timed = [steps_wl[i % T] for i in range(args.steps)]
    kv_total = sum(w.kv_bytes(eb) for w in timed)
    alg_total = sum(w.kv_bytes(eb) + w.io_bytes() for w in timed)
    kv_bytes = kv_total / args.steps
    alg_bytes = alg_total / args.steps
    tok_total = sum(w.tokens_attended for w in timed)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(kv_total, world, total_ms * 1e-3) / 1e9
    tokens_per_s = whole_job_rate(tok_total, world, total_ms * 1e-3)

    # ---- end to end through the public API, host buffers, copies timed
    e2e_steps = e2e_steps or args.e2e_steps or max(10, min(200, args.steps))
    # Each step's inputs (the new tokens' q, k, v and the index arrays) sit in
    # one page-locked host buffer, 256-byte aligned pieces, and go to the GPU
    # in one copy into a device staging buffer the calls read through views,
    # as a serving engine stages a step's inputs.
    def pack(tensors):
        lay, off = {}, 0
        for key, t in tensors.items():
            nb = t.numel() * t.element_size()
            lay[key] = (off, t.dtype, tuple(t.shape), nb)
            off += (nb + 255) // 256 * 256
        buf = torch.empty(max(off, 256), dtype=torch.uint8, pin_memory=True)
        for key, (o, _, _, nb) in lay.items():
            if nb:
                buf[o:o + nb].copy_(tensors[key].contiguous().reshape(-1).view(torch.uint8))
        return buf, lay

    host_pack, layouts = [], []
    for k in range(T):
        tens = {key: v.cpu() for key, v in step_vals[k].items()}
        tens.update(idx_tensors(steps_wl[k],
                                lambda a: torch.from_numpy(np.ascontiguousarray(a))))
        buf, lay = pack(tens)
        host_pack.append(buf)
        layouts.append(lay)
    stage = torch.empty(max(b.numel() for b in host_pack), dtype=torch.uint8, device=dev)
    dev_views = [{key: stage[o:o + nb].view(dt).view(shape)
                  for key, (o, dt, shape, nb) in lay.items()} for lay in layouts]
    host_out = torch.empty(base["q"].shape, dtype=torch.bfloat16, pin_memory=True)
    d2h = host_out.numel() * host_out.element_size()
    cur_stream = torch.cuda.current_stream(dev)
    # The public prepared-step object: checks and argument lists built once.
    dsteps = {}
    for j in range(replicas):
        for k in range(T):
            v = dev_views[k]
            dsteps[(j, k)] = B.DecodeStep(
                outs[j], v["q"], reps[j]["k_pool"], reps[j]["v_pool"], v["bt"], v["sl"],
                wl.scale, max_seq_len=msl, workspace=wss[j], k_new=v["k_new"], v_new=v["v_new"],
                slot_mapping=v["sm"], pairs=v["pairs"] if npairs[k] else None,
                partition_tokens=P, err_word=err,
                kv_scales=(fp8, fp8) if fp8 is not None else None)

    def e2e_body(j, k, sm_copies=True):
        # the step's inputs in, the step, its output out: by the library's
        # SM-driven pa_copy_host (one stream of kernels), or by the copy
        # engine (torch copies)
        hb = host_pack[k]
        if sm_copies:
            B.pa_copy_host(stage[:hb.numel()], hb)
        else:
            stage[:hb.numel()].copy_(hb, non_blocking=True)
        dsteps[(j, k)].enqueue()
        if sm_copies:
            B.pa_copy_host(host_out, outs[j])
        else:
            host_out.copy_(outs[j], non_blocking=True)

    def e2e_eager(i):
        e2e_body(*which(i))
        cur_stream.synchronize()  # the caller needs the result

    # The same step captured once per (replica, step) as a CUDA graph: the
    # input copy, the three library calls and the output copy, replayed and
    # synchronised every step, as a serving engine replays its decode step.
    e2e_graphs, graph_note = None, None
    try:
        e2e_graphs = {}
        cap2 = torch.cuda.Stream(dev)
        for sm_copies in (True, False):
            for j in range(replicas):
                for k in range(T):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=cap2):
                        e2e_body(j, k, sm_copies)
                    e2e_graphs[(j, k, sm_copies)] = g
        torch.cuda.synchronize()
    except Exception as ex:  # capture refused: eager only
        e2e_graphs, graph_note = None, f"graph capture failed ({type(ex).__name__}: {ex})"
        torch.cuda.synchronize()

    def e2e_graphed(i):
        e2e_graphs[which(i) + (True,)].replay()
        cur_stream.synchronize()

    def e2e_graphed_ce(i):
        e2e_graphs[which(i) + (False,)].replay()
        cur_stream.synchronize()

    def time_e2e(fn):
        for i in range(3):
            fn(i)
        env.barrier()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for i in range(e2e_steps):
            fn(i)
        w1 = time.perf_counter()
        env.barrier()
        sec = max_over_ranks(w1 - w0, world, dev)
        return whole_job_rate(sum(steps_wl[i % T].kv_bytes(eb) for i in range(e2e_steps)),
                              world, sec) / 1e9, sec / e2e_steps

    eager_value, eager_s = time_e2e(e2e_eager)
    ce_value = ce_s = None
    if e2e_graphs is not None:
        e2e_value, e2e_step_s = time_e2e(e2e_graphed)
        ce_value, ce_s = time_e2e(e2e_graphed_ce)
    else:
        e2e_value, e2e_step_s = eager_value, eager_s
    h2d = sum(host_pack[which(i)[1]].numel() for i in range(e2e_steps)) / e2e_steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")

    if rank != 0:
        return None

    peak, peak_kind = measured_peak()
    if roof:
        dec_ms = statistics.median(r[0] for r in roof)
        achieved = statistics.median(r[1] for r in roof)
        timing = (f"one CUDA event pair around {inner} back-to-back decode-only graph "
                  f"replays (replicas cycled), median over {len(roof)} repeats")
    else:
        per = [a.elapsed_time(b) for a, b in dec_ev]
        dec_ms = statistics.median(per)
        achieved = alg_bytes / (dec_ms * 1e-3) / 1e9
        timing = "CUDA events around each decode launch inside the timed steps, median"
    traffic = recorded_traffic(name + ("-fp8" if fp8 is not None else "") +
                               (f"-P{P_res}" if P_res > 0 else ""))
    kname = ("split_kernel<fp8> (pa_decode_fp8) + merge_kernel" if fp8 is not None else
             "split_kernel (pa_decode, balanced split) + merge_kernel" if P == 0 else
             "decode_kernel (pa_decode, fixed partitions) + merge_kernel")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": kname,
                "peak_source": f"{peak_kind} hbm_gbs",
                "alg_bytes_per_launch": alg_bytes,
                "timing": timing,
                "decode_ms": dec_ms}
    if multi or cfg == 4:
        roofline["note"] = ("logical bytes: shared blocks are read once per sequence that maps "
                            "them, mostly from L2 (L2-assisted); traffic gives the DRAM bytes")

    cpu = None
    if cpu_baseline and world == 1:
        budget = 6000 if wl.n_q_heads * wl.head_dim >= 4096 else 20000
        seqs, tok = cpu_sample_seqs(wl, budget)
        sub = W_make_values_subset(wl, seqs, fp8=fp8 is not None)
        cpu_oracle_step(sub["wl"], sub["vals"], sub["seqs"], fp8)  # load + warm
        c0 = time.perf_counter()
        reps_cpu = 0
        nbytes = 0
        while True:
            nbytes += cpu_oracle_step(sub["wl"], sub["vals"], sub["seqs"], fp8)
            reps_cpu += 1
            if time.perf_counter() - c0 > 10.0 or reps_cpu >= 1000:
                break
        cdt = time.perf_counter() - c0
        cpu = {"value": nbytes / cdt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(seqs)} of {wl.num_seqs} sequences ({tok} tokens, all "
                         f"{wl.n_q_heads} query heads){' of the first step' if multi else ''}"
                         f" x {reps_cpu} repetitions, {cdt:.1f} s, single thread"}
        # the same sample with the attention rows spread over every host core
        ncores = os.cpu_count() or 1
        if ncores > 1:
            c0 = time.perf_counter()
            reps_all, nbytes = 0, 0
            while True:
                nbytes += cpu_oracle_step(sub["wl"], sub["vals"], sub["seqs"], fp8,
                                          threads=ncores)
                reps_all += 1
                if time.perf_counter() - c0 > 5.0 or reps_all >= 1000:
                    break
            adt = time.perf_counter() - c0
            cpu["all_cores"] = {"value": nbytes / adt / 1e9, "unit": "GB/s", "cores": ncores,
                                "sample": f"the same sample x {reps_all} repetitions, "
                                          f"{adt:.1f} s, attention rows over {ncores} threads"}

    unique = None
    if multi:
        unique = [u * 2 * wl.n_kv_heads * wl.block_size * wl.head_dim * eb
                  for u in wl0.used_blocks]
    config = {"workload": name, "kv_dtype": kv, "num_seqs": wl.num_seqs,
              "tokens_attended": int(tok_total / args.steps), "n_q_heads": wl.n_q_heads,
              "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
              "block_size": wl.block_size, "partition_tokens": P_res,
              "cow_pairs": int(sum(npairs) / T), "kv_bytes_per_step": int(kv_bytes),
              "l2": (f"inputs rotated over {replicas} replicas "
                     f"({replicas * kv_min / 1e6:.0f} MB of KV vs {l2 / 1e6:.0f} MB L2)"
                     if not multi else
                     f"one pool; {kv_bytes / 1e6:.0f} MB of KV read per step (logical) over "
                     f"{max(unique) / 1e6:.0f} MB of unique blocks vs {l2 / 1e6:.0f} MB L2: "
                     "L2-assisted"),
              "arithmetic": ("bf16 operands, fp32 accumulation and softmax; P as a bf16 "
                             "hi + lo pair (two P V products)"
                             if fp8 is None else
                             "E4M3 codes and q as f16 mma operands, fp32 accumulation "
                             "and softmax; P as an f16 hi + lo pair; per-tensor scales"),
              "launch": "eager calls from Python" if args.eager else
                        "one CUDA graph replay per step (copy, write, decode, merge)",
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if multi:
        config["decode_steps"] = T
        config["steps_cycle"] = (f"the timed steps cycle through the {T} precomputed beam "
                                 "steps (forks, frees, copy-on-write) on one pool")
        config["sharing"] = {"used_blocks_last": wl0.used_blocks[-1],
                             "unshared_blocks_last": wl0.unshared_blocks[-1],
                             "saving": 1 - wl0.used_blocks[-1] / wl0.unshared_blocks[-1]}
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if fp8 is None else "e4m3 K/V, bf16 q/out",
        "data": "synthetic",
        "config": config,
        "tokens_attended_per_s": tokens_per_s,
        "pct_of_peak": 100.0 * value / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": e2e_step_s * 1e3,
                "launch": ("one CUDA graph replay per step (pa_copy_host in, DecodeStep."
                           "enqueue: copy_blocks, reshape_and_cache, decode, merge; "
                           "pa_copy_host out), then a stream synchronise"
                           if e2e_graphs is not None else graph_note),
                "copy_engine": ({"value": ce_value, "ms_per_step": ce_s * 1e3,
                                 "launch": "the same graph with the two copies done by the copy "
                                           "engine (torch copies) instead of pa_copy_host"}
                                if ce_value is not None else None),
                "eager": {"value": eager_value, "ms_per_step": eager_s * 1e3,
                          "launch": "the same calls issued from Python every step "
                                    "(pa_copy_host, DecodeStep.enqueue, pa_copy_host), then a "
                                    "stream synchronise"},
                "note": "every step: its inputs (q, k, v of the new tokens, block tables, "
                        "lengths, slots, copy pairs) copied in from one page-locked buffer, "
                        "the public calls, the output copied out to page-locked memory, "
                        "synchronised"},
        "gpu_launches": sum(launches[i % T] for i in range(args.steps)),
        "clocks": clk,
    }


def emit(line, env):
    if line is not None and env.rank == 0:
        print(json.dumps(line), flush=True)


def suite(args, env):
    """Every measured case, one line each; the headline last."""
    cases = [
        lambda: run_copy(args, env),
        lambda: run_write(args, env),
        lambda: run_decode(args, env, 1, 16, e2e_steps=20),
        lambda: run_decode(args, env, 2, 16, e2e_steps=50),
        lambda: run_decode(args, env, 2, 16, kv="fp8", e2e_steps=50),
        lambda: run_decode(args, env, 4, 16, e2e_steps=20),
        lambda: run_decode(args, env, 5, 16, e2e_steps=10),  # 512-token partitions
        lambda: run_decode(args, env, 5, 16, partition_tokens=0, e2e_steps=10),
        lambda: run_decode(args, env, 5, 16, kv="fp8", e2e_steps=10),
        lambda: run_decode(args, env, 6, 16, e2e_steps=20),
        lambda: run_decode(args, env, 3, 8, e2e_steps=10),
        lambda: run_decode(args, env, 3, 32, e2e_steps=10),
        lambda: run_prefill(args, env),
        lambda: run_swap(args, env),
    ]
    for case in cases:
        emit(case(), env)
        release()
    emit(run_decode(args, env, HEADLINE[0], HEADLINE[1], cpu_baseline=not args.no_cpu_baseline),
         env)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    env = Env(args)
    if args.op == "swap":
        emit(run_swap(args, env), env)
    elif args.op == "prefill":
        emit(run_prefill(args, env), env)
    elif args.op == "write":
        emit(run_write(args, env), env)
    elif args.op == "copy":
        emit(run_copy(args, env), env)
    elif args.config is None:
        if args.num_seqs is not None or args.partition_tokens is not None or args.kv != "bf16":
            # a flag that shapes one decode workload: the headline workload with it
            emit(run_decode(args, env, HEADLINE[0], args.block_size, kv=args.kv,
                            partition_tokens=args.partition_tokens, num_seqs=args.num_seqs,
                            cpu_baseline=not args.no_cpu_baseline), env)
        else:
            suite(args, env)
    else:
        emit(run_decode(args, env, args.config, args.block_size, kv=args.kv,
                        partition_tokens=args.partition_tokens, num_seqs=args.num_seqs,
                        cpu_baseline=not args.no_cpu_baseline), env)


if __name__ == "__main__":
    main()
