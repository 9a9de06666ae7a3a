"""The beam-search / parallel-sampling workload: the generator against an
independent replay by the oracle's allocator, the sharing accounting
against closed forms, and the copy-on-write structure of every step."""
import numpy as np
import pytest

from oracle import paref
from paged_kv_cache_105_gb300 import workloads as W


def replay_multistep(ms):
    """Replay the whole log on the oracle's allocator; after each step check
    the tables, lengths, slots and pairs that step's Workload carries."""
    a = paref.Allocator(ms.num_blocks, ms.block_size, free_order=ms.free_order)
    t, slots, pairs, stepped = 0, [], [], []
    for i, op in enumerate(ms.ops):
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
        if t < len(ms.op_end) and i + 1 == ms.op_end[t]:
            wl = ms.steps[t]
            assert len(stepped) == wl.num_seqs
            for j, s in enumerate(stepped):
                tab = a.table(s)
                assert np.array_equal(wl.block_tables[j, :len(tab)], tab)
                assert np.all(wl.block_tables[j, len(tab):] == W.PAD)
                assert a.seq_len(s) == wl.seq_lens[j]
            assert np.array_equal(np.array(slots, np.int32), wl.slot_mapping)
            assert np.array_equal(np.array(pairs, np.int32).reshape(-1, 2), wl.cow_pairs)
            assert ms.num_blocks - a.num_free == ms.used_blocks[t]
            # refcount conservation: every table entry holds one reference
            live = np.concatenate([wl.block_tables[j][wl.block_tables[j] >= 0]
                                   for j in range(wl.num_seqs)])
            rc = a.refcounts()
            assert rc.sum() == len(live)
            t, slots, pairs, stepped = t + 1, [], [], []
    assert t == len(ms.steps)


def test_beam_search_replays_on_the_oracle_allocator():
    replay_multistep(W.beam_search(requests=4, beams=6, steps=40, prompt_median=200,
                                   keep=0.6, seed=3))


def test_beam_search_default_size_replays():
    ms = W.beam_search()
    assert len(ms.steps) == 32 and ms.steps[0].num_seqs == 16 * 8
    replay_multistep(ms)
    # re-selection forks produce copy-on-write pairs at staggered steps
    assert sum(len(w.cow_pairs) > 0 for w in ms.steps) == len(ms.steps)
    assert all(u <= v for u, v in zip(ms.used_blocks, ms.unshared_blocks))


@pytest.mark.parametrize("P", [100, 96, 1, 17])
def test_parallel_sampling_block_counts_closed_form(P):
    # keep = 1: beams never re-select, so they share exactly the prompt. With
    # bs = 16, after step t (length P + t + 1) a request holds the floor(P/16)
    # full prompt blocks once, and each of the W beams owns
    # ceil((P + t + 1)/16) - floor(P/16) blocks (its copy of the partial prompt
    # block included); without sharing each beam would own ceil((P+t+1)/16).
    R, Wb, T, bs = 3, 5, 40, 16
    ms = W.beam_search(requests=R, beams=Wb, steps=T, prompt_median=P, prompt_sigma=0.0,
                       prompt_lo=1, keep=1.0, block_size=bs, seed=1)
    for t in range(T):
        L = P + t + 1
        own = -(-L // bs) - P // bs
        assert ms.used_blocks[t] == R * (P // bs + Wb * own)
        assert ms.unshared_blocks[t] == R * Wb * (-(-L // bs))
        # copies happen only on the first step, and only for a partial prompt block
        want = R * (Wb - 1) if (t == 0 and P % bs) else 0
        assert len(ms.steps[t].cow_pairs) == want


def test_copy_pairs_are_disjoint_and_fresh():
    ms = W.beam_search(requests=6, beams=8, steps=24, prompt_median=150, keep=0.5, seed=9)
    for w in ms.steps:
        src, dst = w.cow_pairs[:, 0], w.cow_pairs[:, 1]
        assert len(set(dst)) == len(dst)                 # no destination twice
        assert not set(dst) & set(src)                    # no destination is a source
        # every destination is now some sequence's last block, at the new token
        last = {int(w.block_tables[i, (int(w.seq_lens[i]) - 1) // w.block_size])
                for i in range(w.num_seqs)}
        assert set(int(x) for x in dst) <= last
