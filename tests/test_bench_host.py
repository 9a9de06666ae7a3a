"""Host-side helpers of bench.py (no GPU): the traffic record's source key,
the bounded CPU sample and the all-core oracle timing path."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import paref  # noqa: E402
from paged_kv_cache_105_gb300 import workloads as W  # noqa: E402


def test_code_tokens_ignore_comments_and_blank_space():
    a = "int f(int x) {  // the answer\n  return x + 1; /* one\n more */ }\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_tokens(a) == bench._code_tokens("int f(int x) { return x + 1; }")
    assert bench._code_tokens(a) != bench._code_tokens(c)


def test_kernel_hash_is_keyed_on_the_listed_sources():
    h1 = bench.kernel_hash(bench.KERNEL_SOURCES)
    h2 = bench.kernel_hash(bench.PREFILL_SOURCES)
    assert len(h1) == 64 and len(h2) == 64 and h1 != h2


def test_cpu_sample_stays_within_its_budget():
    wl = W.config2()
    seqs, tok = bench.cpu_sample_seqs(wl, 3000)
    assert tok == int(wl.seq_lens[seqs].astype(np.int64).sum())
    assert tok <= 3000 or len(seqs) == 1
    assert len(set(seqs)) == len(seqs)


def test_oracle_rows_agree_across_threads():
    # the all-core baseline calls the oracle from several threads at once
    from concurrent.futures import ThreadPoolExecutor
    wl = W.custom([40, 300, 17], n_q_heads=8, n_kv_heads=2, head_dim=64, seed=5)
    vals = W.make_values(wl)
    bits = lambda t: t.view(__import__("torch").int16).numpy().view(np.uint16)
    q, kp, vp = bits(vals["q"]), bits(vals["k_pool"]), bits(vals["v_pool"])
    rows = np.array([(s, h) for s in range(wl.num_seqs) for h in range(8)], np.int32)
    whole = paref.attention_paged(q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, rows=rows)
    chunks = np.array_split(rows, 4)
    with ThreadPoolExecutor(4) as ex:
        parts = list(ex.map(lambda c: paref.attention_paged(q, kp, vp, wl.block_tables,
                                                             wl.seq_lens, wl.scale, rows=c),
                            chunks))
    assert np.array_equal(np.concatenate(parts), whole)
