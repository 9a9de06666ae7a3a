"""The seeded workload builder against an independent replay by the oracle's
allocator: same tables, slots and copy-on-write pairs."""
import numpy as np
import pytest

from oracle import paref
from paged_kv_cache_105_gb300 import workloads as W


def replay(wl):
    a = paref.Allocator(wl.num_blocks, wl.block_size, free_order=wl.free_order)
    slots, pairs, stepped = [], [], []
    for op in wl.ops:
        if op[0] == "add":
            a.add_seq()
        elif op[0] == "append":
            for _ in range(op[2]):
                a.append(op[1])
        elif op[0] == "fork":
            a.fork(op[1])
        elif op[0] == "free":
            a.free(op[1])
        elif op[0] == "step":
            slot, pair = a.append(op[1])
            slots.append(slot)
            stepped.append(op[1])
            if pair:
                pairs.append(pair)
    return a, slots, pairs, stepped


def check(wl):
    a, slots, pairs, stepped = replay(wl)
    assert len(stepped) == wl.num_seqs
    for i, s in enumerate(stepped):
        t = a.table(s)
        assert np.array_equal(wl.block_tables[i, :len(t)], t)
        assert np.all(wl.block_tables[i, len(t):] == W.PAD)
        assert a.seq_len(s) == wl.seq_lens[i]
    assert np.array_equal(np.array(slots, np.int32), wl.slot_mapping)
    assert np.array_equal(np.array(pairs, np.int32).reshape(-1, 2), wl.cow_pairs)
    return a


def test_worked_example_config():
    wl = W.config1()
    assert list(wl.seq_lens) == list(W.WORKED_EXAMPLE_LENGTHS)
    assert paref.paged_slots(wl.seq_lens, wl.block_size) == 2608
    a = check(wl)
    assert wl.num_blocks - a.num_free == 163
    # the ids are the first 163 of the seeded permutation, in (seq, block) order
    used = np.concatenate([wl.block_tables[s, :paref.blocks_for(L, 16)]
                           for s, L in enumerate(wl.seq_lens)])
    assert np.array_equal(used, wl.free_order[:163])
    assert len(wl.cow_pairs) == 0


def test_gqa_batch_config():
    wl = W.config2()
    assert wl.num_seqs == 64 and wl.group == 4 and wl.head_dim == 128
    assert wl.seq_lens.min() >= 1 and wl.seq_lens.max() <= 2048
    assert 150 <= np.median(wl.seq_lens) <= 600
    need = sum(paref.blocks_for(L, 16) for L in wl.seq_lens)
    assert wl.num_blocks == int(np.ceil(1.25 * need))
    check(wl)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_churned_config_small(bs):
    wl = W.config3(block_size=bs, num_seqs=24, max_len=300, phantoms=48, n_heads=4)
    a = check(wl)
    # fragmented: the tables are not runs of consecutive ids
    flat = np.concatenate([wl.block_tables[s, :paref.blocks_for(L, bs)]
                           for s, L in enumerate(wl.seq_lens)])
    assert np.mean(np.diff(flat) == 1) < 0.9
    assert len(set(flat.tolist())) == len(flat)


def test_prefix_sharing_config():
    wl = W.config4()
    a = check(wl)
    prefix = wl.block_tables[:, :64]
    assert np.all(prefix == prefix[0])
    # read by all 128 decoded sequences and by their 128 siblings
    assert all(a.refcount(int(b)) == 256 for b in prefix[0])
    n_cow = int(np.sum((wl.seq_lens - 1) % 16 != 0))
    assert len(wl.cow_pairs) == n_cow
    for src, dst in wl.cow_pairs:
        assert a.refcount(int(src)) == 1 and a.refcount(int(dst)) == 1
    assert set(wl.cow_pairs[:, 1].tolist()).isdisjoint(wl.cow_pairs[:, 0].tolist())


def test_long_context_config_small():
    wl = W.config5(num_seqs=3, seq_len=2000)
    check(wl)
    assert wl.partition_tokens == 512


def test_custom_with_empty_sequence():
    wl = W.custom([0, 1, 16, 17], block_size=16, seed=3)
    a, slots, pairs, stepped = replay(wl)
    assert stepped == [1, 2, 3]                   # no token for the empty one
    assert wl.slot_mapping[0] == -1
    assert np.array_equal(np.array(slots, np.int32), wl.slot_mapping[1:])
    assert np.all(wl.block_tables[0] == W.PAD)
    for s in (1, 2, 3):
        t = a.table(s)
        assert np.array_equal(wl.block_tables[s, :len(t)], t)


def test_values_are_seeded_and_poison_only_tails():
    import torch
    wl = W.config1()
    a = W.make_values(wl)
    b = W.make_values(wl)
    for name in a:
        assert torch.equal(a[name].view(torch.int16), b[name].view(torch.int16))
    p = W.make_values(wl, poison_tails=True)
    kp = p["k_pool"].float()
    bad = ~torch.isfinite(kp)
    for s, L in enumerate(wl.seq_lens):
        for i in range(L):
            blk = wl.block_tables[s, i // 16]
            assert not bad[blk, :, i % 16].any()
    assert bad.any()
