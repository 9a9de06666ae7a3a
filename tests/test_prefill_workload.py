"""The chunked-prefill batch builder against an independent replay by the
oracle's allocator (tables and the chunk tokens' slots), and its flop
count against a direct sum."""
import numpy as np

from oracle import paref
from paged_kv_cache_105_gb300 import workloads as W


def test_prefill_batch_replays_on_the_oracle_allocator():
    wl = W.prefill_batch([0, 37, 300, 16], [50, 1, 64, 16], block_size=16, Hq=8, Hkv=2,
                         d=64, seed=4)
    a = paref.Allocator(wl.num_blocks, wl.block_size, free_order=wl.free_order)
    seqs = [a.add_seq() for _ in range(wl.num_seqs)]
    ctx = wl.seq_lens - wl.chunk_lens
    for s, L in zip(seqs, ctx):
        for _ in range(int(L)):
            a.append(s)
    slots = []
    for s, c in zip(seqs, wl.chunk_lens):
        for _ in range(int(c)):
            slot, pair = a.append(s)
            assert pair is None
            slots.append(slot)
    assert np.array_equal(np.array(slots, np.int32), wl.slot_mapping)
    for i, s in enumerate(seqs):
        t = a.table(s)
        assert np.array_equal(wl.block_tables[i, :len(t)], t)
        assert a.seq_len(s) == wl.seq_lens[i]
    assert np.array_equal(wl.cu_q, np.concatenate([[0], np.cumsum(wl.chunk_lens)]))


def test_chunked_prefill_flops_by_direct_sum():
    wl = W.prefill_chunked()
    assert wl.total_q == 8192 and wl.max_seq_len == 8192
    pairs = sum(p + 1 for L, c in zip(wl.seq_lens, wl.chunk_lens) for p in range(L - c, L))
    assert wl.visible_pairs() == pairs
    assert wl.flops() == 4 * 128 * 32 * pairs
