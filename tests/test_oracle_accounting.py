"""Pins of the oracle's allocation arithmetic to numbers the pages print."""
import random

import pytest

from oracle import paref


def pct1(x):
    return round(100.0 * x, 1)


def test_worked_example(golden):
    g = golden("worked_example.json")
    lens, bs = g["lengths"], g["page"]
    assert paref.used_tokens(lens) == g["used_tokens"]
    assert [paref.blocks_for(L, bs) for L in lens] == g["pages"]
    assert [paref.blocks_for(L, bs) * bs for L in lens] == g["alloc"]
    assert [paref.tail_waste(L, bs) for L in lens] == g["tail_waste"]
    paged = paref.paged_slots(lens, bs)
    naive = paref.naive_slots(len(lens), g["reserve_max_len"])
    assert paged == g["paged_alloc_total"]
    assert naive == g["naive_alloc_total"]
    used = g["used_tokens"]
    assert pct1(1 - used / paged) == g["paged_waste_pct_1dp"]
    assert pct1(1 - used / naive) == g["naive_waste_pct_1dp"]
    assert paref.capacity(g["pool_slots"], naive, len(lens)) == g["naive_capacity"]
    assert paref.capacity(g["pool_slots"], paged, len(lens)) == g["paged_capacity"]


def _fragmentation_lengths(n, max_len):
    # The page's own generator: stdlib random, seed 0, lognormal(5.5, 0.9).
    rnd = random.Random(0)
    return [min(max_len, int(rnd.lognormvariate(5.5, 0.9))) for _ in range(n)]


def test_fragmentation_experiment(golden):
    g = golden("fragmentation.json")
    lens = _fragmentation_lengths(g["N"], g["max_len"])
    used = paref.used_tokens(lens)
    assert used == g["tokens_stored"]
    naive = paref.naive_slots(len(lens), g["max_len"])
    assert naive == g["naive_alloc"]
    assert pct1(used / naive) == g["naive_util_pct_1dp"]
    paged = paref.paged_slots(lens, 16)
    assert paged == g["paged_alloc_bs16"]
    assert pct1(used / paged) == g["paged_util_pct_1dp_bs16"]
    assert round(used / len(lens)) == g["mean_length_0dp"]
    assert round((paged - used) / len(lens), 1) == g["wasted_per_seq_1dp"]
    assert max(paref.tail_waste(L, 16) for L in lens) <= g["max_waste_per_seq"]
    for bs, util in g["sweep_util_pct_1dp"].items():
        assert pct1(used / paref.paged_slots(lens, int(bs))) == util, bs


def test_fragmentation_max_len_32768(golden):
    g = golden("fragmentation.json")
    lens = _fragmentation_lengths(g["N"], 32768)
    used = paref.used_tokens(lens)
    assert pct1(used / paref.naive_slots(len(lens), 32768)) == \
        g["max_len_32768_naive_util_pct_1dp"]
    assert pct1(used / paref.paged_slots(lens, 16)) == g["max_len_32768_paged_util_pct_1dp"]


def test_waste_table(golden):
    g = golden("waste_table.json")
    bs = g["block_size"]
    for row in g["rows"]:
        L = row["len"]
        assert paref.blocks_for(L, bs) == row["blocks"]
        assert paref.tail_waste(L, bs) == row["wasted"]
        alloc = paref.blocks_for(L, bs) * bs
        assert pct1(paref.tail_waste(L, bs) / alloc) == row["waste_pct_1dp"]


def test_capacity_example(golden):
    g = golden("capacity_example.json")
    per_tok = g["kv_bytes_per_token"]
    bpt = (per_tok["layers"] * per_tok["kv_heads"] * per_tok["head_dim"]
           * per_tok["k_and_v"] * per_tok["bytes_per_elem"])
    assert bpt == per_tok["total"]
    assert g["block_size"] * bpt == g["block_bytes"]
    assert g["pool_bytes"] // g["block_bytes"] == g["pool_blocks"]
    bs = g["block_size"]
    assert paref.blocks_for(g["answer_tokens"], bs) == g["answer_blocks"]
    assert bs - paref.tail_waste(g["answer_tokens"], bs) == g["answer_last_block_tokens"]
    assert paref.tail_waste(g["answer_tokens"], bs) == g["answer_last_block_free"]
    assert paref.blocks_for(g["system_prompt_tokens"], bs) == g["system_prompt_blocks"]
    assert paref.tail_waste(g["system_prompt_tokens"], bs) == 0


@pytest.mark.parametrize("bs", [1, 2, 8, 16, 32, 128])
def test_tail_waste_bound(bs):
    # At most block_size - 1 empty slots per sequence, zero on a boundary.
    for L in range(0, 4 * bs + 3):
        w = paref.tail_waste(L, bs)
        assert 0 <= w <= bs - 1
        assert (w == 0) == (L % bs == 0)
        assert paref.blocks_for(L, bs) * bs == L + w


def test_capacity_is_floor():
    assert paref.capacity(40960, 2608, 5) == 78          # 40960 / 521.6 = 78.5
    assert paref.capacity(100, 10, 1) == 10
    assert paref.capacity(99, 10, 1) == 9
    assert paref.capacity(100, 0, 1) == 0


def _grow(alloc, lens):
    """Sequences of the given lengths, grown one token at a time."""
    seqs = [alloc.add_seq() for _ in lens]
    for s, L in zip(seqs, lens):
        for _ in range(L):
            alloc.append(s)
    return seqs


def test_allocator_utilisation_fragmentation(golden):
    # The Try It experiment grown through the allocator itself: the live pool
    # holds the experiment's stored tokens in its paged slots (98.0% at bs 16).
    g = golden("fragmentation.json")
    lens = _fragmentation_lengths(g["N"], g["max_len"])
    pool = g["paged_alloc_bs16"] // 16 + 100
    alloc = paref.Allocator(pool, 16)
    _grow(alloc, lens)
    tokens, slots, blocks = alloc.usage()
    assert tokens == g["tokens_stored"]
    assert slots == g["paged_alloc_bs16"]
    assert blocks == g["paged_alloc_bs16"] // 16
    assert pct1(alloc.utilisation()) == g["paged_util_pct_1dp_bs16"]
    assert alloc.cache_usage() == blocks / pool


def test_allocator_utilisation_worked_example(golden):
    g = golden("worked_example.json")
    alloc = paref.Allocator(256, g["page"])
    _grow(alloc, g["lengths"])
    assert alloc.usage() == (g["used_tokens"], g["paged_alloc_total"],
                             g["paged_alloc_total"] // g["page"])
    assert alloc.utilisation() == g["used_tokens"] / g["paged_alloc_total"]
    assert pct1(1 - alloc.utilisation()) == g["paged_waste_pct_1dp"]


def test_allocator_utilisation_counts_a_shared_block_once():
    # 20 tokens at bs 16: blocks of 16 and 4 tokens. A fork shares both; its
    # next token lands in the shared partial block, which is copied first.
    alloc = paref.Allocator(8, 16)
    (s,) = _grow(alloc, [20])
    assert alloc.usage() == (20, 32, 2)
    f = alloc.fork(s)
    assert alloc.usage() == (20, 32, 2)                  # nothing new held
    _, pair = alloc.append(f)
    assert pair is not None
    assert alloc.usage() == (16 + 4 + 5, 48, 3)          # the copy holds 5 tokens
    alloc.free(s)                                        # its partial block goes back
    assert alloc.usage() == (16 + 5, 32, 2)
    alloc.free(f)
    assert alloc.usage() == (0, 0, 0)
    assert alloc.utilisation() == 0.0 and alloc.cache_usage() == 0.0
