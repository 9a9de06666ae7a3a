"""Seeded synthetic decode-step workloads (input generation only).

Each builder returns the host-side state a block manager hands to the
kernels for one decode step: sequence lengths, block tables, the slot of
every new token and the copy-on-write pairs. Values (Q, the new K/V and the
pool contents) are drawn by ``make_values``. Nothing here computes
attention, writes the cache or copies blocks.

The tables come from a small LIFO free-list simulation (``_Tables``) that
mirrors how a paged block manager hands out blocks: a block is taken when
the previous one is full ("03 · PagedAttention", "Blocks and block tables"),
blocks are uniform so a free list suffices ("PagedAttention", "Pros"), and
a write into a shared block first takes a copy ("PagedAttention",
copy-on-write diagram). Every workload also carries an operation log so
that an independent allocator can replay it and must reach the same tables.

Length conventions: ``seq_lens[s]`` is the number of tokens attended in the
step, including the new token, which sits at position ``seq_lens[s] - 1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAD = -1  # table entries past a sequence's last block


@dataclass
class Workload:
    name: str
    num_seqs: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray        # int32 [S], attended lengths
    block_tables: np.ndarray    # int32 [S, max_blocks], PAD beyond each table
    slot_mapping: np.ndarray    # int32 [S], slot of each sequence's new token
    cow_pairs: np.ndarray       # int32 [n_pairs, 2] (src, dst)
    free_order: np.ndarray      # int32 [num_blocks], initial hand-out order
    ops: list = field(default_factory=list)  # replayable allocator log
    seed: int = 0
    partition_tokens: int = 0   # 0: let the library choose
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def tokens_attended(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def kv_bytes(self, elem_bytes: int = 2) -> int:
        """K+V bytes one decode step must read: sum_s len_s * Hkv * d * 2 (K,V)."""
        return self.tokens_attended * self.n_kv_heads * self.head_dim * elem_bytes * 2

    def io_bytes(self, elem_bytes: int = 2) -> int:
        """Non-KV bytes of one decode: q, out, the tables actually read, lengths."""
        S, Hq, d = self.num_seqs, self.n_q_heads, self.head_dim
        nblk = int(np.sum((self.seq_lens.astype(np.int64) + self.block_size - 1)
                          // self.block_size))
        return 2 * S * Hq * d * elem_bytes + 4 * nblk + 4 * S


class _Tables:
    """Minimal LIFO block hand-out used only to build synthetic tables."""

    def __init__(self, free_order, block_size):
        self.bs = block_size
        self.stack = list(np.asarray(free_order, dtype=np.int64)[::-1])
        self.ref = {}
        self.tables = []
        self.lens = []
        self.alive = []
        self.ops = []

    def _pop(self):
        if not self.stack:
            raise RuntimeError("synthetic pool exhausted")
        b = int(self.stack.pop())
        self.ref[b] = 1
        return b

    def add(self):
        self.tables.append([])
        self.lens.append(0)
        self.alive.append(True)
        self.ops.append(("add",))
        return len(self.tables) - 1

    def grow(self, s, n):
        """Append n tokens to s; its last block must not be shared."""
        if n <= 0:
            return
        L = self.lens[s]
        need = -(-(L + n) // self.bs) - len(self.tables[s])
        if L % self.bs and self.ref[self.tables[s][-1]] > 1:
            raise RuntimeError("grow() into a shared block")
        if need > len(self.stack):
            raise RuntimeError("synthetic pool exhausted")
        for _ in range(need):
            self.tables[s].append(self._pop())
        self.lens[s] = L + n
        self.ops.append(("append", s, n))

    def fork(self, s):
        t = list(self.tables[s])
        for b in t:
            self.ref[b] += 1
        self.tables.append(t)
        self.lens.append(self.lens[s])
        self.alive.append(True)
        self.ops.append(("fork", s))
        return len(self.tables) - 1

    def free(self, s):
        for b in reversed(self.tables[s]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                del self.ref[b]
                self.stack.append(b)
        self.tables[s] = []
        self.lens[s] = 0
        self.alive[s] = False
        self.ops.append(("free", s))

    def step(self, s):
        """The decode step's one new token: returns (slot, cow pair or None)."""
        L = self.lens[s]
        pair = None
        if L % self.bs == 0:
            self.tables[s].append(self._pop())
        else:
            j = L // self.bs
            old = self.tables[s][j]
            if self.ref[old] > 1:
                new = self._pop()
                self.ref[old] -= 1
                self.tables[s][j] = new
                pair = (old, new)
        self.lens[s] = L + 1
        self.ops.append(("step", s))
        blk = self.tables[s][L // self.bs]
        return blk * self.bs + L % self.bs, pair


def _finish(name, tb: _Tables, seqs, free_order, *, Hq, Hkv, d, num_blocks, seed,
            slots, pairs, partition_tokens=0, note=""):
    lens = np.array([tb.lens[s] for s in seqs], dtype=np.int32)
    maxb = max(1, max((len(tb.tables[s]) for s in seqs), default=1))
    bt = np.full((len(seqs), maxb), PAD, dtype=np.int32)
    for i, s in enumerate(seqs):
        bt[i, :len(tb.tables[s])] = tb.tables[s]
    cp = np.array(pairs, dtype=np.int32).reshape(-1, 2)
    return Workload(name=name, num_seqs=len(seqs), n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d,
                    block_size=tb.bs, num_blocks=num_blocks, seq_lens=lens, block_tables=bt,
                    slot_mapping=np.array(slots, dtype=np.int32), cow_pairs=cp,
                    free_order=np.asarray(free_order, dtype=np.int32), ops=tb.ops,
                    seed=seed, partition_tokens=partition_tokens, note=note)


def _two_phase(name, lens, *, bs, num_blocks, Hq, Hkv, d, seed, rng, partition_tokens=0,
               note=""):
    """Sequences with L-1 cached tokens each (taken in sequence order from a
    shuffled free list), then the step appends token L-1 to each in turn."""
    free_order = rng.permutation(num_blocks)
    tb = _Tables(free_order, bs)
    seqs = [tb.add() for _ in lens]
    for s, L in zip(seqs, lens):
        tb.grow(s, int(L) - 1)
    slots, pairs = [], []
    for s in seqs:
        slot, pair = tb.step(s)
        slots.append(slot)
        if pair:
            pairs.append(pair)
    return _finish(name, tb, seqs, free_order, Hq=Hq, Hkv=Hkv, d=d, num_blocks=num_blocks,
                   seed=seed, slots=slots, pairs=pairs, partition_tokens=partition_tokens,
                   note=note)


def _lognormal_lengths(rng, n, median, sigma, lo, hi):
    z = rng.standard_normal(n)
    return np.clip(np.rint(np.exp(np.log(median) + sigma * z)), lo, hi).astype(np.int64)


# ------------------------------------------------------------------ configs

WORKED_EXAMPLE_LENGTHS = (512, 37, 1900, 128, 4)


def config1(seed: int = 1) -> Workload:
    """Worked example: lengths 512/37/1900/128/4, block 16, a 256-block pool
    handed out in a seeded random order, 8 q / 8 kv heads, head_dim 64."""
    rng = np.random.default_rng(seed)
    return _two_phase("worked-example-5seq-bs16-mha8-d64", WORKED_EXAMPLE_LENGTHS, bs=16,
                      num_blocks=256, Hq=8, Hkv=8, d=64, seed=seed, rng=rng)


def config2(seed: int = 2, num_seqs: int = 64, block_size: int = 16) -> Workload:
    """GQA decode batch: 64 sequences, lengths lognormal (median 300, sigma 1,
    clipped to [1, 2048]), 32 q / 8 kv heads, head_dim 128, pool 1.25x need."""
    rng = np.random.default_rng(seed)
    lens = _lognormal_lengths(rng, num_seqs, 300.0, 1.0, 1, 2048)
    need = int(sum(-(-int(L) // block_size) for L in lens))
    nb = int(math.ceil(1.25 * need))
    return _two_phase(f"gqa-decode-{num_seqs}seq-lognorm300-bs{block_size}-q32kv8-d128", lens,
                      bs=block_size, num_blocks=nb, Hq=32, Hkv=8, d=128, seed=seed, rng=rng)


def config3(block_size: int = 16, seed: int = 3, num_seqs: int = 256, max_len: int = 4096,
            n_heads: int = 32, phantoms: int = 512) -> Workload:
    """MHA decode over a fragmented pool: lengths uniform on [1, max_len];
    32 q = 32 kv heads, head_dim 128; the tables come from a free list after
    churn: phantom sequences grow round-robin until the pool is ~90% full, a
    seeded half of them is freed, then the real sequences grow round-robin,
    freeing further phantoms (seeded order) whenever the pool runs dry."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len + 1, size=num_seqs)
    need = int(sum(-(-int(L) // block_size) for L in lens))
    nb = int(math.ceil(1.25 * need)) + 64
    free_order = np.arange(nb)
    tb = _Tables(free_order, block_size)
    ph_lens = rng.integers(1, max_len + 1, size=phantoms)
    ph = [tb.add() for _ in range(phantoms)]
    target = int(0.9 * nb)
    used = 0
    # Round-robin growth, one block-round at a time (token-round-robin takes
    # blocks in exactly this order).
    done = False
    for b in range(-(-max_len // block_size)):
        for s, L in zip(ph, ph_lens):
            if used >= target:
                done = True
                break
            lo = b * block_size
            if lo < L:
                tb.grow(s, min(int(L), lo + block_size) - lo)
                used += 1
        if done:
            break
    victims = list(rng.permutation(phantoms))
    for s in victims[: phantoms // 2]:
        tb.free(ph[s])
    spare = victims[phantoms // 2:]
    real = [tb.add() for _ in range(num_seqs)]
    for b in range(-(-max_len // block_size)):
        for s, L in zip(real, lens):
            lo = b * block_size
            hi = min(int(L) - 1, lo + block_size)  # L-1 tokens before the step
            if lo < hi:
                while not tb.stack:
                    tb.free(ph[spare.pop(0)])
                tb.grow(s, hi - lo)
    slots, pairs = [], []
    for s in real:
        if tb.lens[s] % block_size == 0:
            while not tb.stack:
                tb.free(ph[spare.pop(0)])
        slot, pair = tb.step(s)
        slots.append(slot)
        if pair:
            pairs.append(pair)
    return _finish(f"mha-decode-{num_seqs}seq-uniform{max_len}-bs{block_size}-h{n_heads}-d128"
                   "-churned", tb, real, free_order, Hq=n_heads, Hkv=n_heads, d=128,
                   num_blocks=nb, seed=seed, slots=slots, pairs=pairs)


def config4(seed: int = 4, num_seqs: int = 128, prefix_tokens: int = 1024,
            block_size: int = 16) -> Workload:
    """Prefix sharing with copy-on-write: every sequence maps the same
    1024-token prefix (64 blocks) and owns a suffix of lognormal length
    (median 200, sigma 1, clipped to [1, 1024]). Each sequence has a sibling
    fork taken before this step (as in parallel sampling or beam search), so
    its partially filled last block is shared; the step's write into it
    copies the block first. 32 q / 8 kv heads, head_dim 128."""
    rng = np.random.default_rng(seed)
    suffix = _lognormal_lengths(rng, num_seqs, 200.0, 1.0, 1, 1024)
    pre_blocks = -(-prefix_tokens // block_size)
    need = pre_blocks + int(sum(-(-(int(x)) // block_size) + 1 for x in suffix))
    nb = int(math.ceil(1.25 * need))
    free_order = rng.permutation(nb)
    tb = _Tables(free_order, block_size)
    root = tb.add()
    tb.grow(root, prefix_tokens)
    seqs = [tb.fork(root) for _ in range(num_seqs)]
    tb.free(root)
    for s, x in zip(seqs, suffix):
        tb.grow(s, int(x) - 1)
        tb.fork(s)  # sibling, not decoded in this step
    slots, pairs = [], []
    for s in seqs:
        slot, pair = tb.step(s)
        slots.append(slot)
        if pair:
            pairs.append(pair)
    return _finish(f"prefix-share-cow-{num_seqs}seq-prefix{prefix_tokens}-q32kv8-d128", tb,
                   seqs, free_order, Hq=32, Hkv=8, d=128, num_blocks=nb, seed=seed,
                   slots=slots, pairs=pairs)


def config5(seed: int = 5, num_seqs: int = 16, seq_len: int = 32768,
            partition_tokens: int = 512) -> Workload:
    """Long-context split-KV: 16 sequences of 32768 tokens, block 16, blocks
    placed at random in a pool of 1.25x need, 64 q / 8 kv heads, head_dim 128,
    KV partitions of 512 tokens."""
    rng = np.random.default_rng(seed)
    need = num_seqs * (-(-seq_len // 16))
    nb = int(math.ceil(1.25 * need))
    return _two_phase(f"long-context-{num_seqs}x{seq_len}-bs16-q64kv8-d128", [seq_len] * num_seqs,
                      bs=16, num_blocks=nb, Hq=64, Hkv=8, d=128, seed=seed, rng=rng,
                      partition_tokens=partition_tokens)


def custom(lens, *, block_size=16, n_q_heads=8, n_kv_heads=8, head_dim=128, seed=0,
           extra_blocks=8, partition_tokens=0, name="custom") -> Workload:
    """Any lengths (0 allowed: no token, no write) in the two-phase layout."""
    rng = np.random.default_rng(seed)
    lens = [int(L) for L in lens]
    need = sum(-(-L // block_size) for L in lens)
    nb = max(1, need + extra_blocks)
    free_order = rng.permutation(nb)
    tb = _Tables(free_order, block_size)
    seqs = [tb.add() for _ in lens]
    for s, L in zip(seqs, lens):
        tb.grow(s, L - 1)
    slots, pairs = [], []
    for s, L in zip(seqs, lens):
        if L == 0:
            slots.append(-1)
            continue
        slot, pair = tb.step(s)
        slots.append(slot)
        if pair:
            pairs.append(pair)
    return _finish(name, tb, seqs, free_order, Hq=n_q_heads, Hkv=n_kv_heads, d=head_dim,
                   num_blocks=nb, seed=seed, slots=slots, pairs=pairs,
                   partition_tokens=partition_tokens)


@dataclass
class PrefillWorkload:
    """One chunked-prefill step: sequence s has seq_lens[s] - chunk_lens[s]
    cached tokens and appends a chunk of chunk_lens[s] tokens (rows
    cu_q[s]..cu_q[s+1]-1 of the batch), whose K/V go to slot_mapping[row]."""
    name: str
    num_seqs: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray      # int32 [S], cached tokens after the chunk
    chunk_lens: np.ndarray    # int32 [S]
    cu_q: np.ndarray          # int32 [S + 1]
    block_tables: np.ndarray  # int32 [S, max_blocks]
    slot_mapping: np.ndarray  # int32 [total_q]
    free_order: np.ndarray
    ops: list = field(default_factory=list)
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_q_len(self) -> int:
        return int(self.chunk_lens.max()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def visible_pairs(self) -> int:
        """Sum over query tokens of the positions each attends to (p + 1)."""
        tot = 0
        for L, c in zip(self.seq_lens.astype(np.int64), self.chunk_lens.astype(np.int64)):
            tot += c * (L - c) + c * (c + 1) // 2
        return int(tot)

    def flops(self) -> int:
        """Causal attention flops: 2 (QK) + 2 (PV) multiply-adds of head_dim per
        visible (query token, position) pair and query head."""
        return 4 * self.head_dim * self.n_q_heads * self.visible_pairs()

    def kv_bytes(self, elem_bytes: int = 2) -> int:
        """K+V bytes of every cached position of every sequence, read once."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.n_kv_heads * \
            self.head_dim * elem_bytes * 2


def prefill_batch(contexts, chunks, *, block_size: int = 16, Hq: int = 32, Hkv: int = 8,
                  d: int = 128, seed: int = 0, extra_blocks: int = 8,
                  name: str = "") -> PrefillWorkload:
    """Sequences with contexts[s] cached tokens each, then a chunk of
    chunks[s] tokens per sequence, blocks handed out from a seeded shuffled
    free list (history first, sequence by sequence, then the chunks)."""
    rng = np.random.default_rng(seed)
    ctx = [int(x) for x in contexts]
    ch = [int(x) for x in chunks]
    nb = sum(-(-(a + b) // block_size) for a, b in zip(ctx, ch)) + extra_blocks
    free_order = rng.permutation(nb)
    tb = _Tables(free_order, block_size)
    seqs = [tb.add() for _ in ctx]
    for sq, a in zip(seqs, ctx):
        tb.grow(sq, a)
    slots = []
    for sq, a, b in zip(seqs, ctx, ch):
        tb.grow(sq, b)
        for pos in range(a, a + b):
            slots.append(tb.tables[sq][pos // block_size] * block_size + pos % block_size)
    lens = np.array([a + b for a, b in zip(ctx, ch)], np.int32)
    maxb = max(1, max(len(tb.tables[sq]) for sq in seqs))
    bt = np.full((len(seqs), maxb), PAD, np.int32)
    for i, sq in enumerate(seqs):
        bt[i, :len(tb.tables[sq])] = tb.tables[sq]
    cu = np.concatenate([[0], np.cumsum(ch)]).astype(np.int32)
    name = name or f"prefill-{len(ctx)}seq-q{Hq}kv{Hkv}-d{d}-bs{block_size}"
    return PrefillWorkload(name=name, num_seqs=len(ctx), n_q_heads=Hq, n_kv_heads=Hkv,
                           head_dim=d, block_size=block_size, num_blocks=nb, seq_lens=lens,
                           chunk_lens=np.array(ch, np.int32), cu_q=cu, block_tables=bt,
                           slot_mapping=np.array(slots, np.int32),
                           free_order=np.asarray(free_order, np.int32), ops=tb.ops, seed=seed)


def prefill_chunked(seed: int = 7) -> PrefillWorkload:
    """A chunked-prefill step of 8192 batched tokens: eight 8192-token prompts,
    each at a different chunk (chunk 1024 tokens, contexts 0, 1024, ..., 7168
    already cached); block 16, 32 q / 8 kv heads, head_dim 128."""
    return prefill_batch([1024 * k for k in range(8)], [1024] * 8, seed=seed,
                         name="chunked-prefill-8x1024-ctx0to7168-bs16-q32kv8-d128")


def prefill_mix(num_seqs: int, *, max_context: int = 200, max_chunk: int = 48,
                seed: int = 0, **kw) -> PrefillWorkload:
    """A mixed batch of many sequences: contexts uniform in [0, max_context),
    chunks uniform in [0, max_chunk) (some empty), seeded; other arguments as
    prefill_batch."""
    rng = np.random.default_rng(seed * 7919 + num_seqs)
    ctx = rng.integers(0, max_context, num_seqs)
    ch = rng.integers(0, max_chunk, num_seqs)
    kw.setdefault("name", f"prefill-mix-{num_seqs}seq")
    return prefill_batch(ctx, ch, seed=seed, **kw)


def make_prefill_values(wl: PrefillWorkload, device="cpu", seed=None):
    """bf16 N(0, 1): q and the chunk's new K/V [total_q, ...], the pools."""
    import torch

    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + 53)
    TQ, Hq, Hkv, d, bs, NB = (wl.total_q, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                              wl.block_size, wl.num_blocks)
    bf = torch.bfloat16
    return {"q": torch.randn((TQ, Hq, d), generator=g, device=device, dtype=bf),
            "k_new": torch.randn((TQ, Hkv, d), generator=g, device=device, dtype=bf),
            "v_new": torch.randn((TQ, Hkv, d), generator=g, device=device, dtype=bf),
            "k_pool": torch.randn((NB, Hkv, bs, d), generator=g, device=device, dtype=bf),
            "v_pool": torch.randn((NB, Hkv, bs, d), generator=g, device=device, dtype=bf)}


@dataclass
class MultiStep:
    """Several decode steps over one pool. steps[t] is step t's Workload (the
    tables, lengths, slots and copy-on-write pairs after that step's forks,
    frees and appends); ops is the whole allocator log and op_end[t] the log
    length after step t; used_blocks[t] counts pool blocks in use after step
    t and unshared_blocks[t] what the same tables would take without
    sharing (sum over sequences of ceil(len / block_size))."""
    name: str
    steps: list
    ops: list
    op_end: list
    free_order: np.ndarray
    num_blocks: int
    used_blocks: list
    unshared_blocks: list

    @property
    def block_size(self) -> int:
        return self.steps[0].block_size


def beam_search(*, requests: int = 16, beams: int = 8, steps: int = 32,
                prompt_median: float = 1000.0, prompt_sigma: float = 0.5,
                prompt_lo: int = 32, prompt_hi: int = 4096, keep: float = 0.7,
                block_size: int = 16, Hq: int = 32, Hkv: int = 8, d: int = 128,
                seed: int = 6, name: str = "") -> MultiStep:
    """Beam search (or, with keep=1, parallel sampling) over a shared prompt.

    Each request's prompt (lognormal length, seeded) is cached once; `beams`
    sequences fork from it. Every step first re-selects the beams (from the
    second step on): beam j keeps its own lineage with probability `keep`,
    else it continues a uniformly drawn beam of the same request, so beams
    diverge and re-converge at staggered times. The first child of a parent
    continues the parent's sequence, further children fork it, parents with
    no child are freed. Then every beam appends its new token; a token that
    lands in a block shared with a sibling copies the block first. Sequences
    are ordered (request, beam) in every step."""
    rng = np.random.default_rng(seed)
    P = _lognormal_lengths(rng, requests, prompt_median, prompt_sigma, prompt_lo, prompt_hi)
    per_beam = -(-(P.astype(np.int64) + steps) // block_size)
    nb = int(beams * per_beam.sum()) + beams * requests  # never exhausted
    free_order = rng.permutation(nb)
    tb = _Tables(free_order, block_size)
    cur = []
    for r in range(requests):
        root = tb.add()
        tb.grow(root, int(P[r]))
        cur.append([root] + [tb.fork(root) for _ in range(beams - 1)])
    name = name or (f"beam-search-{requests}x{beams}beams-prompt{int(prompt_median)}"
                    f"-{steps}steps-keep{keep:g}-bs{block_size}-q{Hq}kv{Hkv}-d{d}")
    out, op_end, used, unshared = [], [], [], []
    for t in range(steps):
        slots, pairs, seqs = [], [], []
        for r in range(requests):
            if t > 0:
                parents = [j if rng.random() < keep else int(rng.integers(0, beams))
                           for j in range(beams)]
                taken, new = set(), []
                for p in parents:
                    if p in taken:
                        new.append(tb.fork(cur[r][p]))
                    else:
                        taken.add(p)
                        new.append(cur[r][p])
                for p in range(beams):
                    if p not in taken:
                        tb.free(cur[r][p])
                cur[r] = new
            for sq in cur[r]:
                slot, pair = tb.step(sq)
                slots.append(slot)
                seqs.append(sq)
                if pair:
                    pairs.append(pair)
        out.append(_finish(f"{name}-step{t}", tb, seqs, free_order, Hq=Hq, Hkv=Hkv, d=d,
                           num_blocks=nb, seed=seed * 1000 + t, slots=slots, pairs=pairs))
        op_end.append(len(tb.ops))
        used.append(len(tb.ref))
        unshared.append(int(sum(-(-tb.lens[sq] // block_size) for sq in seqs)))
    for w in out:
        w.ops = []  # the log lives in the MultiStep
    return MultiStep(name=name, steps=out, ops=list(tb.ops), op_end=op_end,
                     free_order=np.asarray(free_order, np.int32), num_blocks=nb,
                     used_blocks=used, unshared_blocks=unshared)


def config6(seed: int = 6) -> MultiStep:
    """Beam search: 16 requests x 8 beams over prompts of lognormal length
    (median 1000, sigma 0.5, clipped to [32, 4096]), 32 decode steps, beams
    keep their lineage with probability 0.7 per step; block 16, 32 q / 8 kv
    heads, head_dim 128."""
    return beam_search(seed=seed)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5, 6: config6}


# ------------------------------------------------------------------ values

BF16_NAN = 0x7FC0
BF16_POS_INF = 0x7F80


def make_values(wl: Workload, device="cpu", seed=None, poison_tails: bool = False):
    """Draw Q, the new K/V and the pool contents, bf16 ~ N(0, 1), seeded.

    Returns a dict of torch tensors on ``device``: q [S,Hq,d], k_new/v_new
    [S,Hkv,d] (one new token per sequence), k_pool/v_pool [NB,Hkv,bs,d].
    With ``poison_tails`` the slots past each sequence's last token in its
    last block (and, for a copy-on-write pair, the source block's slots from
    the new token on) hold NaN/Inf bit patterns: they must never reach an
    output.
    """
    import torch

    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + 17)
    S, Hq, Hkv, d, bs, NB = (wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                             wl.block_size, wl.num_blocks)
    bf = torch.bfloat16
    out = {
        "q": torch.randn((S, Hq, d), generator=g, device=device, dtype=bf),
        "k_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf),
        "v_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf),
        "k_pool": torch.randn((NB, Hkv, bs, d), generator=g, device=device, dtype=bf),
        "v_pool": torch.randn((NB, Hkv, bs, d), generator=g, device=device, dtype=bf),
    }
    if poison_tails:
        poison_blocks, poison_from = [], []
        pair_src = {int(dst): int(src) for src, dst in wl.cow_pairs}
        for s in range(S):
            L = int(wl.seq_lens[s])
            if L == 0:
                continue
            j = (L - 1) // bs
            blk = int(wl.block_tables[s, j])
            off = (L - 1) % bs
            poison_blocks.append(blk)
            poison_from.append(off + 1)
            if blk in pair_src:
                poison_blocks.append(pair_src[blk])
                poison_from.append(off)
        for blk, start in zip(poison_blocks, poison_from):
            if start < bs:
                for name, bits in (("k_pool", BF16_NAN), ("v_pool", BF16_POS_INF)):
                    view = out[name].view(torch.int16)
                    view[blk, :, start:, :] = bits - (1 << 16 if bits >= 1 << 15 else 0)
    return out


def make_step_values(wl: Workload, device="cpu", seed=None):
    """The per-step inputs alone (q, k_new, v_new; bf16 N(0, 1), seeded by the
    step's workload): for multi-step runs whose pools persist across steps."""
    import torch

    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + 41)
    S, Hq, Hkv, d = wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    bf = torch.bfloat16
    return {"q": torch.randn((S, Hq, d), generator=g, device=device, dtype=bf),
            "k_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf),
            "v_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf)}


# fp8 (E4M3) cache contents. A full fp8 cache stands for K/V ~ N(0, 1) that
# earlier steps stored with a per-tensor scale chosen so that about 4.5
# standard deviations reach the largest code (448): scale = 4.5 / 448, a
# value that is not a power of two, so the cache write's division rounds.
FP8_SCALE = 4.5 / 448.0
E4M3_NAN = 0x7F


def make_values_fp8(wl: Workload, device="cpu", seed=None, poison_tails: bool = False,
                    k_scale: float = FP8_SCALE, v_scale: float = FP8_SCALE):
    """Like make_values, but k_pool/v_pool are uint8 E4M3 codes.

    The pool codes are N(0, 1) / scale drawn in fp32 (on ``device``, seeded)
    and cast by torch to float8_e4m3fn (torch's own conversion: how one draws fp8 data,
    not the library's cache write). q and the new K/V stay bf16 N(0, 1).
    With ``poison_tails`` the same slots as in make_values hold the NaN
    code 0x7F in both pools."""
    import torch

    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + 29)
    S, Hq, Hkv, d, bs, NB = (wl.num_seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                             wl.block_size, wl.num_blocks)
    bf = torch.bfloat16

    def codes(scale):
        c = torch.empty((NB, Hkv, bs, d), dtype=torch.uint8, device=device)
        step = max(1, (1 << 26) // max(1, Hkv * bs * d))  # bounded fp32 temporaries
        for b0 in range(0, NB, step):
            b1 = min(NB, b0 + step)
            x = torch.randn((b1 - b0, Hkv, bs, d), generator=g, device=device,
                            dtype=torch.float32) / scale
            c[b0:b1] = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        return c

    out = {
        "q": torch.randn((S, Hq, d), generator=g, device=device, dtype=bf),
        "k_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf),
        "v_new": torch.randn((S, Hkv, d), generator=g, device=device, dtype=bf),
        "k_pool": codes(k_scale),
        "v_pool": codes(v_scale),
    }
    if poison_tails:
        pair_src = {int(dst): int(src) for src, dst in wl.cow_pairs}
        for s in range(S):
            L = int(wl.seq_lens[s])
            if L == 0:
                continue
            blk = int(wl.block_tables[s, (L - 1) // bs])
            off = (L - 1) % bs
            spans = [(blk, off + 1)]
            if blk in pair_src:
                spans.append((pair_src[blk], off))
            for b, start in spans:
                if start < bs:
                    out["k_pool"][b, :, start:, :] = E4M3_NAN
                    out["v_pool"][b, :, start:, :] = E4M3_NAN
    return out
