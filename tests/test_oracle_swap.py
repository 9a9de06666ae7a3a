"""Pins of the oracle's block swap (preemption by swapping blocks out to host
memory and back)."""
import numpy as np

from oracle import paref


def pools(rng, nb, shape=(2, 16, 8), dtype=np.uint16):
    k = rng.integers(0, 1 << 16, (nb,) + shape).astype(dtype)
    v = rng.integers(0, 1 << 16, (nb,) + shape).astype(dtype)
    return k, v


def test_swap_matches_fancy_indexing():
    rng = np.random.default_rng(0)
    sk, sv = pools(rng, 30)
    dk, dv = pools(rng, 12)
    pairs = np.array([[3, 0], [29, 11], [7, 5], [0, 6]], np.int32)
    wk, wv = dk.copy(), dv.copy()
    wk[pairs[:, 1]] = sk[pairs[:, 0]]
    wv[pairs[:, 1]] = sv[pairs[:, 0]]
    assert paref.swap_blocks(dk, dv, sk, sv, pairs) == 0
    assert np.array_equal(dk, wk) and np.array_equal(dv, wv)


def test_swap_out_then_in_restores_the_blocks_under_new_ids():
    rng = np.random.default_rng(1)
    gk, gv = pools(rng, 40)
    g0k, g0v = gk.copy(), gv.copy()
    hk, hv = np.zeros((10,) + gk.shape[1:], gk.dtype), np.zeros((10,) + gv.shape[1:], gv.dtype)
    victim = np.array([5, 17, 33, 2], np.int32)          # blocks of a preempted sequence
    host_ids = np.array([9, 0, 4, 1], np.int32)
    assert paref.swap_blocks(hk, hv, gk, gv, np.stack([victim, host_ids], 1)) == 0
    gk[victim] = 0                                        # the device blocks are reused
    back = np.array([20, 21, 22, 23], np.int32)           # fresh device ids on swap-in
    assert paref.swap_blocks(gk, gv, hk, hv, np.stack([host_ids, back], 1)) == 0
    assert np.array_equal(gk[back], g0k[victim]) and np.array_equal(gv[back], g0v[victim])


def test_swap_skips_out_of_range_pairs_and_touches_nothing_else():
    rng = np.random.default_rng(2)
    sk, sv = pools(rng, 8, dtype=np.uint8)
    dk, dv = pools(rng, 8, dtype=np.uint8)
    d0 = dk.copy()
    pairs = np.array([[8, 0], [0, 8], [-1, 1], [1, 2]], np.int32)
    assert paref.swap_blocks(dk, dv, sk, sv, pairs) == 3
    assert np.array_equal(dk[2], sk[1])
    keep = [0, 1, 3, 4, 5, 6, 7]
    assert np.array_equal(dk[keep], d0[keep])
