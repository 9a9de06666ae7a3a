"""Randomised GPU parity: seeded random batch shapes (sequence count and
lengths, block size, head dim, GQA group, split mode, bf16 or fp8 cache)
through the whole decode step, each against the fp64 oracle on every output
and the pool bytes exactly; and seeded random chunked-prefill batches, every
output row against the oracle. The seeds are fixed, so a failure
reproduces."""
import numpy as np
import pytest
import torch

from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import (bits, compare, gpu_step, gpu_step_fp8, oracle_step,
                           oracle_step_fp8)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 200))
    kind = rng.integers(0, 3)
    if kind == 0:    # short, many zeros and boundaries
        lens = rng.integers(0, 70, size=n)
    elif kind == 1:  # lognormal mix
        lens = np.clip(np.round(np.exp(np.log(200) + rng.normal(size=n))), 0, 6000)
    else:            # a few long ones among short ones
        lens = rng.integers(0, 40, size=n)
        lens[rng.integers(0, n, size=max(1, n // 20))] = rng.integers(2000, 20000)
    bs = int(rng.choice([8, 16, 32]))
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 8, 16]))
    P = int(rng.choice([0, 0, 64, 256, 512]))
    return dict(lens=[int(x) for x in lens], bs=bs, d=d, hkv=hkv, hq=hkv * g, P=P,
                seed=seed)


@pytest.mark.parametrize("seed", range(16))
def test_random_batches_bf16(seed):
    c = random_case(seed)
    wl = W.custom(c["lens"], block_size=c["bs"], n_q_heads=c["hq"], n_kv_heads=c["hkv"],
                  head_dim=c["d"], seed=c["seed"], partition_tokens=c["P"],
                  name=f"random-{seed}")
    vals_cpu = W.make_values(wl, poison_tails=True)
    ref, kp, vp = oracle_step(wl, vals_cpu)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_step(wl, vals)
    assert err == 0
    assert np.array_equal(bits(vals["k_pool"]), kp)
    assert np.array_equal(bits(vals["v_pool"]), vp)
    compare(out, ref, wl.name)


@pytest.mark.parametrize("seed", range(8))
def test_random_batches_fp8(seed):
    c = random_case(100 + seed)
    wl = W.custom(c["lens"], block_size=c["bs"], n_q_heads=c["hq"], n_kv_heads=c["hkv"],
                  head_dim=128, seed=c["seed"], name=f"random-fp8-{seed}")
    vals_cpu = W.make_values_fp8(wl, poison_tails=True)
    ref, kp, vp = oracle_step_fp8(wl, vals_cpu, W.FP8_SCALE, W.FP8_SCALE)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_step_fp8(wl, vals, W.FP8_SCALE, W.FP8_SCALE)
    assert err == 0
    assert np.array_equal(vals["k_pool"].cpu().numpy(), kp)
    assert np.array_equal(vals["v_pool"].cpu().numpy(), vp)
    compare(out, ref, wl.name)


def random_prefill_case(seed):
    rng = np.random.default_rng(2000 + seed)
    n = int(rng.integers(1, 41))  # up to 32: the block-wide or one-warp ranking; beyond: the search
    ctx = rng.integers(0, 400, size=n)
    ch = rng.integers(0, 200, size=n)
    ch[rng.random(n) < 0.15] = 0  # some sequences without a chunk
    if ch.max() == 0:
        ch[0] = 1
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 3, 4, 8, 16]))
    while hkv * g > 16:
        hkv //= 2
    return dict(ctx=[int(x) for x in ctx], ch=[int(x) for x in ch], bs=int(rng.choice([8, 16, 32])),
                d=int(rng.choice([64, 128])), hkv=hkv, hq=hkv * g, seed=seed)


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill_batches(seed):
    # seeded random chunked-prefill batches (sequence count, contexts, chunk
    # lengths with some empty, block size, head dim, group size), every output
    # row against the oracle
    from tests.test_gpu_prefill import gpu_prefill, oracle_prefill_threaded
    c = random_prefill_case(seed)
    wl = W.prefill_batch(c["ctx"], c["ch"], block_size=c["bs"], Hq=c["hq"], Hkv=c["hkv"],
                         d=c["d"], seed=c["seed"], name=f"random-prefill-{seed}")
    vals_cpu = W.make_prefill_values(wl)
    rows = np.array([(t, h) for t in range(wl.total_q) for h in range(wl.n_q_heads)], np.int32)
    ref = oracle_prefill_threaded(wl, vals_cpu, rows)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, err = gpu_prefill(wl, vals)
    assert err == 0
    compare(out.reshape(-1, wl.head_dim), ref, wl.name)
