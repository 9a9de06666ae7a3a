"""GPU parity of chunked-prefill attention against the fp64 oracle: the
chunk's K/V written by the cache write, then causal attention over the whole
paged context. Same bar as decode, element by element: |gpu - ref| <= 1e-2
and |gpu - ref| / max(|ref|, 1e-2) <= 2e-2, and every (token, head) row
within 2e-2 relative L2 error."""
import numpy as np
import pytest
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import bits, compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_prefill(wl, vals, err=None, max_q_len=None):
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).to(DEV)
         for k in ("block_tables", "seq_lens", "cu_q", "slot_mapping")}
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_reshape_and_cache(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                           t["slot_mapping"], err_word=err)
    out = torch.full_like(vals["q"], float("nan"))
    B.pa_prefill(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                 t["seq_lens"], t["cu_q"], wl.scale,
                 max_q_len=wl.max_q_len if max_q_len is None else max_q_len, err_word=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def oracle_prefill(wl, vals_cpu, rows=None):
    kp, vp = bits(vals_cpu["k_pool"]).copy(), bits(vals_cpu["v_pool"]).copy()
    paref.reshape_and_cache(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                            wl.slot_mapping)
    out = paref.prefill_paged(bits(vals_cpu["q"]), kp, vp, wl.block_tables, wl.seq_lens,
                              wl.cu_q, wl.scale, rows=rows)
    return out, kp, vp


def oracle_prefill_threaded(wl, vals_cpu, rows):
    """oracle_prefill's rows, split across host threads (independent rows)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    kp, vp = bits(vals_cpu["k_pool"]).copy(), bits(vals_cpu["v_pool"]).copy()
    paref.reshape_and_cache(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                            wl.slot_mapping)
    q = bits(vals_cpu["q"])
    chunks = [c for c in np.array_split(rows, max(1, min(32, os.cpu_count() or 1))) if len(c)]
    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda c: paref.prefill_paged(q, kp, vp, wl.block_tables,
                                                          wl.seq_lens, wl.cu_q, wl.scale,
                                                          rows=c), chunks))
    return np.concatenate(parts, 0)


CASES = [
    # contexts, chunks
    ([0, 37, 300, 16, 5], [50, 1, 64, 16, 130]),
    ([0], [1]),
    ([1000, 0], [3, 200]),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (12, 4), (16, 1), (64, 2)])
def test_prefill_parity(d, bs, heads):
    Hq, Hkv = heads
    for i, (ctx, ch) in enumerate(CASES):
        wl = W.prefill_batch(ctx, ch, block_size=bs, Hq=Hq, Hkv=Hkv, d=d,
                             seed=i * 100 + bs + Hq, name=f"prefill-{i}-bs{bs}-q{Hq}kv{Hkv}")
        vals_cpu = W.make_prefill_values(wl)
        ref, kp, vp = oracle_prefill(wl, vals_cpu)
        vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
        out, err = gpu_prefill(wl, vals)
        assert err == 0
        assert np.array_equal(bits(vals["k_pool"]), kp)
        compare(out, ref, wl.name)


def test_single_token_chunks_equal_decode():
    # c_s = 1 for every sequence is a decode step: compare with pa_decode
    lens = [1, 17, 300, 64, 1000]
    wl = W.prefill_batch([L - 1 for L in lens], [1] * len(lens), Hq=32, Hkv=8, seed=3)
    vals = {k: v.to(DEV) for k, v in W.make_prefill_values(wl).items()}
    out, err = gpu_prefill(wl, vals)
    assert err == 0
    dec = torch.empty_like(out)
    bt = torch.from_numpy(wl.block_tables).to(DEV)
    sl = torch.from_numpy(wl.seq_lens).to(DEV)
    ws = B.decode_workspace(wl.num_seqs, 32, 8, 128, 16, wl.max_seq_len, 0, device=DEV)
    B.pa_decode(dec, vals["q"], vals["k_pool"], vals["v_pool"], bt, sl, wl.scale,
                max_seq_len=wl.max_seq_len, workspace=ws)
    torch.cuda.synchronize()
    diff = (out.float() - dec.float()).abs().max().item()
    assert diff <= 1e-2


def test_chunked_prefill_full_size_sampled():
    # every head of every 32nd chunk token and of the chunk edges: 9,472 rows
    wl = W.prefill_chunked()
    vals_cpu = W.make_prefill_values(wl)
    toks = sorted(set(range(0, wl.total_q, 32)) |
                  {1023, 1024, 4095, 4096, 7167, 7168, 8191, 1, 31, 33})
    rows = np.array([(t, h) for t in toks for h in range(wl.n_q_heads)], np.int32)
    ref = oracle_prefill_threaded(wl, vals_cpu, rows)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_prefill(wl, vals)
    assert err == 0
    got = out[torch.from_numpy(rows[:, 0]).long(), torch.from_numpy(rows[:, 1]).long()]
    compare(got, ref, wl.name)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("num_seqs", [255, 256, 257, 300])
def test_many_sequences_every_row(num_seqs):
    # Up to 256 sequences the blocks take the tiles longest first, beyond
    # that in the grid's own order; either way every tile exactly once (the
    # output starts as NaN, so a tile left out shows). Some chunks are empty.
    wl = W.prefill_mix(num_seqs, Hq=12, Hkv=4, d=64, seed=11)
    assert (wl.chunk_lens == 0).any()
    vals_cpu = W.make_prefill_values(wl)
    ref, kp, vp = oracle_prefill(wl, vals_cpu)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_prefill(wl, vals)
    assert err == 0
    compare(out, ref, wl.name)


def test_many_tiles_few_sequences_every_row():
    # 32 sequences with more (sequence, query tile) pairs than threads in a
    # block: the tiles are ranked by one warp, each lane trying its own cost
    # (16 heads per kv head: 16-token query tiles, 10 to 16 per sequence)
    ctx = [(7 * k) % 150 for k in range(32)]
    ch = [150 + (37 * k) % 100 for k in range(32)]
    wl = W.prefill_batch(ctx, ch, Hq=16, Hkv=1, d=64, seed=12, name="prefill-32seq-g16")
    assert sum(-(-c // 16) for c in ch) > 352
    vals_cpu = W.make_prefill_values(wl)
    ref = oracle_prefill_threaded(wl, vals_cpu, np.array(
        [(t, h) for t in range(wl.total_q) for h in range(wl.n_q_heads)], np.int32))
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_prefill(wl, vals)
    assert err == 0
    compare(out.reshape(-1, wl.head_dim), ref, wl.name)


def test_short_max_q_len_is_flagged():
    wl = W.prefill_batch([10, 0], [40, 100], Hq=32, Hkv=8, d=64, seed=5)  # 64-token tiles
    vals_cpu = W.make_prefill_values(wl)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_prefill(wl, vals, max_q_len=64)
    assert err & B.PA_DEV_ERR_SEQ_LEN
    # the grid covers each chunk's first 64 tokens (max_q_len): those rows
    # are still right, the second chunk's rows from 64 on stay unwritten
    ref, _, _ = oracle_prefill(wl, vals_cpu)
    keep = np.r_[0:40, 40:104]
    compare(out[torch.from_numpy(keep).long()], ref[keep], wl.name + "-truncated")
    assert torch.isnan(out[104:].float()).all()


def test_bad_block_id_flagged():
    wl = W.prefill_batch([40, 70], [8, 8], Hq=8, Hkv=2, d=64, seed=6)
    wl.block_tables[1, 2] = wl.num_blocks + 7
    vals = {k: v.to(DEV) for k, v in W.make_prefill_values(wl).items()}
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).to(DEV)
         for k in ("block_tables", "seq_lens", "cu_q")}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(vals["q"])
    B.pa_prefill(out, vals["q"], vals["k_pool"], vals["v_pool"], t["block_tables"],
                 t["seq_lens"], t["cu_q"], wl.scale, max_q_len=wl.max_q_len, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PA_DEV_ERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
