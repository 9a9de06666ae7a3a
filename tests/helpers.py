"""Shared test plumbing: run one decode step through the C ABI, and compute
the oracle's answer from the generator's inputs (never from GPU output)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W

ATOL = 1e-2       # max abs error, bf16 output vs fp64 oracle ...
BF16_ROUND = 2.0 ** -8  # ... or, where larger, the rounding bound of a bf16 output (|ref| > 2.56)
RTOL = 2e-2       # max element-wise relative error |gpu - ref| / max(|ref|, REL_FLOOR)
REL_FLOOR = 1e-2  # denominator floor: outputs are means of N(0, 1) values and can sit at 0
ROW_RTOL = 2e-2   # also: max over (seq, head) rows of ||gpu - ref||_2 / ||ref||_2

# Every compare() call appends (what, elements, max abs, max rel, max row rel,
# the reference value at the worst relative element); the session prints the
# maxima per workload at its end (tests/conftest.py).
PARITY_REPORT: list = []


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy array of its bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_dev(wl: W.Workload, device):
    d = dict(
        block_tables=torch.from_numpy(wl.block_tables).to(device),
        seq_lens=torch.from_numpy(wl.seq_lens).to(device),
        slot_mapping=torch.from_numpy(wl.slot_mapping).to(device),
        pairs=torch.from_numpy(np.ascontiguousarray(wl.cow_pairs.reshape(-1, 2))).to(device),
    )
    return d


def gpu_step(wl: W.Workload, vals: dict, partition_tokens=None, workspace=None, err=None,
             run_writes=True, max_seq_len=None):
    """copy_blocks -> reshape_and_cache -> decode on the tensors in `vals`
    (modified in place). Returns (out, err_word value)."""
    dev = vals["q"].device
    t = to_dev(wl, dev)
    P = wl.partition_tokens if partition_tokens is None else partition_tokens
    msl = wl.max_seq_len if max_seq_len is None else max_seq_len
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = B.decode_workspace(wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                       wl.block_size, msl, P, device=dev)
    out = torch.full_like(vals["q"], float("nan"))
    if run_writes:
        B.pa_copy_blocks(vals["k_pool"], vals["v_pool"], t["pairs"], err_word=err)
        B.pa_reshape_and_cache(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                               t["slot_mapping"], err_word=err)
    B.pa_decode(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                t["seq_lens"], wl.scale, max_seq_len=msl, workspace=workspace,
                partition_tokens=P, err_word=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def oracle_step(wl: W.Workload, vals_cpu: dict):
    """The oracle's copy -> write -> attention on host copies of the inputs.
    Returns (out fp64 [S,Hq,d], k_pool bits, v_pool bits)."""
    kp, vp = bits(vals_cpu["k_pool"]).copy(), bits(vals_cpu["v_pool"]).copy()
    paref.copy_blocks(kp, vp, wl.cow_pairs)
    paref.reshape_and_cache(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                            wl.slot_mapping)
    out = paref.attention_paged(bits(vals_cpu["q"]), kp, vp, wl.block_tables, wl.seq_lens,
                                wl.scale)
    return out, kp, vp


def sampled_oracle(wl: W.Workload, vals_dev: dict, seqs, fp8_scales=None):
    """Oracle rows for the sequences `seqs` of a workload too large to copy
    whole: gather (before the GPU step touches the pool) only the blocks
    those sequences read, plus their copy-on-write sources, into a compact
    host pool, remap ids, and run the oracle's step there. fp8_scales =
    (k_scale, v_scale) for uint8 E4M3 pools.
    Returns out fp64 [len(seqs), Hq, d]."""
    bs = wl.block_size
    seqs = list(seqs)
    pair_src = {int(dst): int(src) for src, dst in wl.cow_pairs}
    need = []
    for s in seqs:
        nb = -(-int(wl.seq_lens[s]) // bs)
        for b in wl.block_tables[s, :nb]:
            need.append(int(b))
            if int(b) in pair_src:
                need.append(pair_src[int(b)])
    ids = list(dict.fromkeys(need))
    remap = {b: i for i, b in enumerate(ids)}
    idx = torch.tensor(ids, dtype=torch.long, device=vals_dev["k_pool"].device)
    pool_np = bits if fp8_scales is None else (lambda t: t.cpu().numpy())
    kp = pool_np(vals_dev["k_pool"].index_select(0, idx)).copy()
    vp = pool_np(vals_dev["v_pool"].index_select(0, idx)).copy()
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
    sel = torch.tensor(seqs, dtype=torch.long, device=vals_dev["q"].device)
    q = bits(vals_dev["q"].index_select(0, sel))
    kn = bits(vals_dev["k_new"].index_select(0, sel))
    vn = bits(vals_dev["v_new"].index_select(0, sel))
    pairs = np.array(pairs, np.int32).reshape(-1, 2)
    slots = np.array(slots, np.int32)
    lens = wl.seq_lens[seqs].astype(np.int32)
    if fp8_scales is None:
        paref.copy_blocks(kp, vp, pairs)
        paref.reshape_and_cache(kn, vn, kp, vp, slots)
        return attention_threaded(paref.attention_paged, (q, kp, vp, bt, lens, wl.scale),
                                  len(seqs), wl.n_q_heads, wl.head_dim)
    ks, vs = fp8_scales
    paref.copy_blocks(kp.view(np.uint16), vp.view(np.uint16), pairs)  # a byte copy
    paref.reshape_and_cache_fp8(kn, vn, kp, vp, slots, ks, vs)
    return attention_threaded(paref.attention_paged_fp8, (q, kp, vp, bt, lens, wl.scale, ks, vs),
                              len(seqs), wl.n_q_heads, wl.head_dim)


def attention_threaded(fn, args, num_seqs, n_q_heads, head_dim, threads=None):
    """The oracle's attention `fn(*args, rows=...)` over every (sequence, head)
    row, the rows split across host threads (each oracle call releases the
    interpreter lock). Same result as one call: rows are independent."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    rows = np.array([(s, h) for s in range(num_seqs) for h in range(n_q_heads)], np.int32)
    threads = threads or max(1, min(32, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(rows, threads) if len(c)]
    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda c: fn(*args, rows=c), chunks))
    return np.concatenate(parts, 0).reshape(num_seqs, n_q_heads, head_dim)


class Parity(tuple):
    """(max_abs, max_rel) of one comparison, plus the row-wise figure."""

    def __new__(cls, max_abs, max_rel, max_row_rel):
        obj = super().__new__(cls, (max_abs, max_rel))
        obj.max_abs, obj.max_rel, obj.max_row_rel = max_abs, max_rel, max_row_rel
        return obj

    def __str__(self):
        return (f"max_abs={self.max_abs:.2e} max_rel={self.max_rel:.2e} "
                f"max_row_rel={self.max_row_rel:.2e}")


def compare(gpu_out: torch.Tensor, ref: np.ndarray, what="") -> Parity:
    """bf16 GPU output vs fp64 oracle, element by element: |gpu - ref| <=
    max(ATOL, BF16_ROUND * |ref|) and |gpu - ref| / max(|ref|, REL_FLOOR) <=
    RTOL for every element. The second term of the absolute bar is the
    rounding of a bf16 output itself: a value of magnitude 4 or more lies up
    to 2^-9 * 2^e (half a bf16 step, 2^e <= |ref|) from both neighbouring bf16
    values, more than 1e-2, whatever the kernel computes. The row-wise
    relative L2 error is computed and asserted as well."""
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel_el = err / np.maximum(np.abs(ref), REL_FLOOR)
    worst = int(np.argmax(rel_el)) if rel_el.size else 0
    max_rel = float(rel_el.flat[worst]) if rel_el.size else 0.0
    num = np.sqrt((err ** 2).sum(-1))
    den = np.sqrt((ref ** 2).sum(-1))
    rel = np.where(den > 0, num / np.maximum(den, 1e-30), num)
    max_row = float(rel.max()) if rel.size else 0.0
    PARITY_REPORT.append((what, int(err.size), max_abs, max_rel, max_row,
                          float(ref.flat[worst]) if ref.size else 0.0))
    where = np.unravel_index(worst, ref.shape) if ref.size else ()
    bar = np.maximum(ATOL, BF16_ROUND * np.abs(ref))
    over = err > bar
    if over.any():
        i = int(np.argmax(err - bar))
        raise AssertionError(f"{what}: abs err {err.flat[i]:.3e} > {bar.flat[i]:.3e} at "
                             f"{tuple(int(j) for j in np.unravel_index(i, ref.shape))} "
                             f"(ref {ref.flat[i]:.4e}, gpu {g.flat[i]:.4e})")
    assert max_rel <= RTOL, (f"{what}: max element rel err {max_rel:.3e} > {RTOL} at "
                             f"{tuple(int(i) for i in where)} (ref {ref.flat[worst]:.4e}, "
                             f"gpu {g.flat[worst]:.4e})")
    assert max_row <= ROW_RTOL, f"{what}: max row rel err {max_row:.3e} > {ROW_RTOL}"
    return Parity(max_abs, max_rel, max_row)


# ------------------------------------------------------------------ fp8 cache

def gpu_step_fp8(wl: W.Workload, vals: dict, k_scale, v_scale, workspace=None, err=None,
                 run_writes=True):
    """copy_blocks_fp8 -> reshape_and_cache_fp8 -> decode_fp8 (pools are
    uint8 E4M3 codes, modified in place). Returns (out, err_word value)."""
    dev = vals["q"].device
    t = to_dev(wl, dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = B.decode_workspace(wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                       wl.block_size, wl.max_seq_len, 0, device=dev)
    out = torch.full_like(vals["q"], float("nan"))
    if run_writes:
        B.pa_copy_blocks_fp8(vals["k_pool"], vals["v_pool"], t["pairs"], err_word=err)
        B.pa_reshape_and_cache_fp8(vals["k_new"], vals["v_new"], vals["k_pool"],
                                   vals["v_pool"], t["slot_mapping"], k_scale, v_scale,
                                   err_word=err)
    B.pa_decode_fp8(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                    t["seq_lens"], wl.scale, k_scale, v_scale, max_seq_len=wl.max_seq_len,
                    workspace=workspace, err_word=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def oracle_step_fp8(wl: W.Workload, vals_cpu: dict, k_scale, v_scale):
    """The oracle's step over uint8 E4M3 pools. Returns (out, k codes, v codes)."""
    kp = vals_cpu["k_pool"].numpy().copy()
    vp = vals_cpu["v_pool"].numpy().copy()
    # a block copy moves bytes: the oracle's copy on a 16-bit view of the codes
    paref.copy_blocks(kp.view(np.uint16), vp.view(np.uint16), wl.cow_pairs)
    paref.reshape_and_cache_fp8(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                                wl.slot_mapping, k_scale, v_scale)
    out = paref.attention_paged_fp8(bits(vals_cpu["q"]), kp, vp, wl.block_tables, wl.seq_lens,
                                    wl.scale, k_scale, v_scale)
    return out, kp, vp
