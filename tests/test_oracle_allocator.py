"""Pins of the oracle's free-list allocator: on-demand blocks, refcounts,
fork and copy-on-write, free, exhaustion."""
import numpy as np
import pytest

from oracle import paref


def test_seventeenth_token_allocates(golden):
    g = golden("block_table_examples.json")
    bs = g["block_size"]
    a = paref.Allocator(8, bs)
    s = a.add_seq()
    took = []
    for t in range(1, 33):
        before = a.num_free
        a.append(s)
        if a.num_free < before:
            took.append(t)
    assert took == g["allocating_tokens_1_to_32"]


def test_sequence_b_and_80_token_request(golden):
    g = golden("block_table_examples.json")
    bs = g["block_size"]
    a = paref.Allocator(16, bs)
    s = a.add_seq()
    for _ in range(g["seq_b_tokens"]):
        a.append(s)
    assert len(a.table(s)) == g["seq_b_blocks"]
    assert g["seq_b_tokens"] - (len(a.table(s)) - 1) * bs == g["seq_b_last_used"]
    r = a.add_seq()
    for _ in range(80):
        a.append(r)
    assert len(a.table(r)) == g["request_80_tokens_blocks"]
    assert a.free(r) == g["request_80_tokens_blocks"]


def test_slots_follow_the_table():
    bs = 4
    order = [5, 2, 7, 0, 1, 3, 4, 6]
    a = paref.Allocator(8, bs, free_order=order)
    s = a.add_seq()
    slots = [a.append(s)[0] for _ in range(10)]
    # blocks are handed out in free_order; slot = block * bs + offset
    assert list(a.table(s)) == [5, 2, 7]
    assert slots == [20, 21, 22, 23, 8, 9, 10, 11, 28, 29]


def test_copy_on_write_diagram():
    # Three sequences share three blocks, the last partly filled; the first
    # writer copies the shared last block, the others keep the original.
    bs = 16
    a = paref.Allocator(10, bs, free_order=list(range(10)))
    root = a.add_seq()
    for _ in range(41):
        a.append(root)
    s1 = a.fork(root)
    s2 = a.fork(root)
    a.free(root)
    shared = list(a.table(s1))
    assert shared == [0, 1, 2]
    assert [a.refcount(b) for b in shared] == [2, 2, 2]
    slot, pair = a.append(s1)
    assert pair == (2, 3)
    assert list(a.table(s1)) == [0, 1, 3]
    assert list(a.table(s2)) == [0, 1, 2]
    assert a.refcount(2) == 1 and a.refcount(3) == 1
    assert a.refcount(0) == 2 and a.refcount(1) == 2
    assert slot == 3 * bs + 41 % bs
    # s2 is now the only owner of block 2: it writes in place.
    slot2, pair2 = a.append(s2)
    assert pair2 is None and slot2 == 2 * bs + 41 % bs
    # a full shared block is never copied: the next token opens a new block
    b = a.add_seq()
    for _ in range(16):
        a.append(b)
    c = a.fork(b)
    _, p = a.append(c)
    assert p is None and a.table(c)[0] == a.table(b)[0]


def test_exhaustion_leaves_state_unchanged():
    a = paref.Allocator(2, 4)
    s = a.add_seq()
    for _ in range(8):
        a.append(s)
    before = (list(a.table(s)), a.num_free, a.seq_len(s))
    with pytest.raises(paref.OutOfBlocks):
        a.append(s)
    assert (list(a.table(s)), a.num_free, a.seq_len(s)) == before
    # copy-on-write also needs a block
    a2 = paref.Allocator(1, 4)
    r = a2.add_seq()
    a2.append(r)
    f = a2.fork(r)
    with pytest.raises(paref.OutOfBlocks):
        a2.append(f)
    assert a2.refcount(0) == 2 and a2.seq_len(f) == 1


def test_free_returns_blocks_lifo():
    a = paref.Allocator(6, 2, free_order=[0, 1, 2, 3, 4, 5])
    s = a.add_seq()
    for _ in range(6):
        a.append(s)
    assert list(a.table(s)) == [0, 1, 2]
    assert a.free(s) == 3
    # walked from the last entry to the first: the first block is on top
    assert list(a.free_list()) == [0, 1, 2, 3, 4, 5]
    t = a.add_seq()
    a.append(t)
    assert list(a.table(t)) == [0]


def test_random_ops_invariants():
    rng = np.random.default_rng(7)
    nb, bs = 64, 4
    a = paref.Allocator(nb, bs, free_order=rng.permutation(nb))
    live = []
    for step in range(3000):
        op = rng.integers(0, 10)
        if op < 6 and live:
            s = live[rng.integers(len(live))]
            try:
                L0, T0 = a.seq_len(s), len(a.table(s))
                a.append(s)
                L = a.seq_len(s)
                assert L == L0 + 1
                assert len(a.table(s)) == -(-L // bs)
                assert len(a.table(s)) - T0 in (0, 1)
            except paref.OutOfBlocks:
                pass
        elif op < 7 and live:
            live.append(a.fork(live[rng.integers(len(live))]))
        elif op < 8 and live:
            s = live.pop(rng.integers(len(live)))
            a.free(s)
        else:
            live.append(a.add_seq())
        if step % 50 == 0:
            ref = a.refcounts()
            counted = np.zeros(nb, dtype=np.int64)
            for s in live:
                for b in a.table(s):
                    counted[b] += 1
            assert np.array_equal(ref, counted)        # refcount conservation
            fl = set(a.free_list().tolist())
            used = set(np.nonzero(counted)[0].tolist())
            assert len(fl) == a.num_free              # no duplicates
            assert fl.isdisjoint(used)
            assert fl | used == set(range(nb))        # free list + live = pool
            for s in live:                            # tail waste bound
                w = len(a.table(s)) * bs - a.seq_len(s)
                assert 0 <= w <= bs - 1
