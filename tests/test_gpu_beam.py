"""GPU parity over many decode steps of beam search / parallel sampling:
forks, frees and copy-on-write between steps, one pool throughout. Every
step's output against the fp64 oracle (same bar as single steps); the pools
byte-exact after the last step."""
import numpy as np
import pytest
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import attention_threaded, bits, compare, gpu_step

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def oracle_pools_step(wl, kp, vp, step_vals):
    """The oracle's copy -> write on persistent host pools (in place)."""
    paref.copy_blocks(kp, vp, wl.cow_pairs)
    paref.reshape_and_cache(bits(step_vals["k_new"]), bits(step_vals["v_new"]), kp, vp,
                            wl.slot_mapping)


@pytest.mark.parametrize("keep", [0.5, 1.0])
def test_beam_steps_full_parity(keep):
    ms = W.beam_search(requests=3, beams=4, steps=24, prompt_median=120, keep=keep, Hq=8,
                       Hkv=2, d=64, seed=12)
    base = W.make_values(ms.steps[0])
    kp, vp = bits(base["k_pool"]).copy(), bits(base["v_pool"]).copy()
    pools = {"k_pool": base["k_pool"].to(DEV), "v_pool": base["v_pool"].to(DEV)}
    n_pairs = 0
    for wl in ms.steps:
        sv = W.make_step_values(wl)
        oracle_pools_step(wl, kp, vp, sv)
        ref = paref.attention_paged(bits(sv["q"]), kp, vp, wl.block_tables, wl.seq_lens,
                                    wl.scale)
        vals = dict(pools, **{k: v.to(DEV) for k, v in sv.items()})
        out, err = gpu_step(wl, vals)
        assert err == 0
        compare(out, ref, wl.name)
        n_pairs += len(wl.cow_pairs)
    assert n_pairs > 0
    assert np.array_equal(bits(pools["k_pool"]), kp)
    assert np.array_equal(bits(pools["v_pool"]), vp)


def test_beam_search_full_size():
    # every step's pool bytes; every output of three of the 32 steps
    ms = W.config6()
    base = W.make_values(ms.steps[0], device=DEV)
    kp, vp = bits(base["k_pool"]).copy(), bits(base["v_pool"]).copy()
    for t, wl in enumerate(ms.steps):
        sv = W.make_step_values(wl, device=DEV)
        oracle_pools_step(wl, kp, vp, sv)
        vals = dict(base, **sv)
        out, err = gpu_step(wl, vals)
        assert err == 0
        if t in (0, 13, len(ms.steps) - 1):
            ref = attention_threaded(paref.attention_paged,
                                     (bits(sv["q"]), kp, vp, wl.block_tables, wl.seq_lens,
                                      wl.scale), wl.num_seqs, wl.n_q_heads, wl.head_dim)
            compare(out, ref, wl.name)
    assert np.array_equal(bits(base["k_pool"]), kp)
    assert np.array_equal(bits(base["v_pool"]), vp)
