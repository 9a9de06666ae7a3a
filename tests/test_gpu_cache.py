"""GPU parity of the cache writes: pa_copy_blocks and pa_reshape_and_cache
are bit-exact against the oracle over the whole pool (so every byte they
must not touch is untouched), and bad ids are skipped and flagged."""
import numpy as np
import pytest
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import bits, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def random_bits_values(wl, seed):
    """Pools and new K/V as arbitrary 16-bit patterns (NaN payloads too)."""
    g = torch.Generator().manual_seed(seed)
    def rb(*shape):
        return torch.randint(-(1 << 15), 1 << 15, shape, generator=g,
                             dtype=torch.int16).view(torch.bfloat16)
    S, Hkv, d, bs, NB = wl.num_seqs, wl.n_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks
    return {"k_new": rb(S, Hkv, d), "v_new": rb(S, Hkv, d),
            "k_pool": rb(NB, Hkv, bs, d), "v_pool": rb(NB, Hkv, bs, d)}


def run_writes(wl, vals_cpu, slot_mapping=None, pairs=None):
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    t = to_dev(wl, DEV)
    if slot_mapping is not None:
        t["slot_mapping"] = torch.tensor(slot_mapping, dtype=torch.int32, device=DEV)
    if pairs is not None:
        t["pairs"] = torch.tensor(pairs, dtype=torch.int32, device=DEV).reshape(-1, 2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_copy_blocks(vals["k_pool"], vals["v_pool"], t["pairs"], err_word=err)
    B.pa_reshape_and_cache(vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"],
                           t["slot_mapping"], err_word=err)
    torch.cuda.synchronize()
    return vals, int(err.item())


def oracle_writes(vals_cpu, slot_mapping, pairs):
    kp, vp = bits(vals_cpu["k_pool"]).copy(), bits(vals_cpu["v_pool"]).copy()
    paref.copy_blocks(kp, vp, np.asarray(pairs, np.int32).reshape(-1, 2))
    paref.reshape_and_cache(bits(vals_cpu["k_new"]), bits(vals_cpu["v_new"]), kp, vp,
                            np.asarray(slot_mapping, np.int32))
    return kp, vp


@pytest.mark.parametrize("cfg", ["c1", "c2", "c4", "c3_bs8", "c3_bs32"])
def test_step_writes_bit_exact(cfg):
    wl = {"c1": W.config1, "c2": W.config2, "c4": W.config4,
          "c3_bs8": lambda: W.config3(block_size=8, num_seqs=64, max_len=1024, phantoms=96),
          "c3_bs32": lambda: W.config3(block_size=32, num_seqs=64, max_len=1024,
                                       phantoms=96)}[cfg]()
    vals_cpu = random_bits_values(wl, 11)
    vals, err = run_writes(wl, vals_cpu)
    assert err == 0
    kp, vp = oracle_writes(vals_cpu, wl.slot_mapping, wl.cow_pairs)
    assert np.array_equal(bits(vals["k_pool"]), kp)
    assert np.array_equal(bits(vals["v_pool"]), vp)
    if cfg == "c4":
        assert len(wl.cow_pairs) > 100


@pytest.mark.parametrize("d,bs,hkv", [(64, 8, 1), (64, 32, 3), (128, 16, 8), (128, 8, 2)])
def test_writes_all_shapes_with_padding_and_bad_ids(d, bs, hkv):
    wl = W.custom([5, 17, 33, 40], block_size=bs, n_q_heads=hkv, n_kv_heads=hkv, head_dim=d,
                  seed=d + bs)
    vals_cpu = random_bits_values(wl, 12)
    NB = wl.num_blocks
    slots = [int(wl.slot_mapping[0]), -1, NB * bs + 3, int(wl.slot_mapping[3])]
    pairs = [[0, NB - 1], [NB, 1], [2, -5], [1, NB - 2]]
    vals, err = run_writes(wl, vals_cpu, slot_mapping=slots, pairs=pairs)
    assert err & B.PA_DEV_ERR_SLOT
    assert err & B.PA_DEV_ERR_PAIR
    assert not err & ~(B.PA_DEV_ERR_SLOT | B.PA_DEV_ERR_PAIR)
    kp, vp = oracle_writes(vals_cpu, slots, pairs)
    assert np.array_equal(bits(vals["k_pool"]), kp)
    assert np.array_equal(bits(vals["v_pool"]), vp)


def test_copy_blocks_many_pairs_full_size():
    # Config-4 sized pool, one copy for every block pair (src, dst) disjoint.
    wl = W.config4()
    vals_cpu = random_bits_values(wl, 13)
    NB = wl.num_blocks
    rng = np.random.default_rng(0)
    perm = rng.permutation(NB)
    half = NB // 2
    pairs = np.stack([perm[:half], perm[half:2 * half]], axis=1).astype(np.int32)
    vals, err = run_writes(wl, vals_cpu, slot_mapping=[-1] * wl.num_seqs, pairs=pairs)
    assert err == 0
    kp, vp = oracle_writes(vals_cpu, [-1] * wl.num_seqs, pairs)
    assert np.array_equal(bits(vals["k_pool"]), kp)
    assert np.array_equal(bits(vals["v_pool"]), vp)
