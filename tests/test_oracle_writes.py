"""Pins of the oracle's cache write and block copy: exactly the named bytes
change, nothing else does."""
import numpy as np

from oracle import paref


def pools(rng, nb, hkv, bs, d):
    kp = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    return kp, vp


def test_reshape_and_cache_writes_only_the_slots():
    rng = np.random.default_rng(0)
    nb, hkv, bs, d, T = 6, 3, 8, 16, 5
    kp, vp = pools(rng, nb, hkv, bs, d)
    k = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    slots = np.array([0, 13, -1, 47, 48 * 10], np.int32)   # pad, then one out of range
    kp0, vp0 = kp.copy(), vp.copy()
    skipped = paref.reshape_and_cache(k, v, kp, vp, slots)
    assert skipped == 1
    touched = np.zeros((nb, bs), bool)
    for t, s in enumerate(slots):
        if 0 <= s < nb * bs:
            b, o = divmod(int(s), bs)
            touched[b, o] = True
            assert np.array_equal(kp[b, :, o], k[t])
            assert np.array_equal(vp[b, :, o], v[t])
    mask = ~touched[:, None, :, None].repeat(hkv, 1).repeat(d, 3)
    assert np.array_equal(kp[mask], kp0[mask])
    assert np.array_equal(vp[mask], vp0[mask])


def test_copy_blocks_duplicates_and_leaves_the_rest():
    rng = np.random.default_rng(1)
    nb, hkv, bs, d = 8, 2, 4, 8
    kp, vp = pools(rng, nb, hkv, bs, d)
    kp0, vp0 = kp.copy(), vp.copy()
    pairs = np.array([[1, 5], [2, 6], [0, 99]], np.int32)
    assert paref.copy_blocks(kp, vp, pairs) == 1
    for s, t in [(1, 5), (2, 6)]:
        assert np.array_equal(kp[t], kp0[s]) and np.array_equal(vp[t], vp0[s])
    for b in (0, 1, 2, 3, 4, 7):
        assert np.array_equal(kp[b], kp0[b]) and np.array_equal(vp[b], vp0[b])


def test_copy_then_write_is_the_cow_step():
    # Copy the shared block first, then write the new token into the copy:
    # the copy holds the shared tokens plus the new one, the original is intact.
    rng = np.random.default_rng(2)
    nb, hkv, bs, d = 4, 1, 4, 4
    kp, vp = pools(rng, nb, hkv, bs, d)
    a = paref.Allocator(nb, bs, free_order=[0, 1, 2, 3])
    s = a.add_seq()
    for _ in range(2):
        a.append(s)
    f = a.fork(s)
    slot, pair = a.append(f)
    assert pair == (0, 1) and slot == 1 * bs + 2
    orig = kp[0].copy()
    k = rng.integers(0, 1 << 16, size=(1, hkv, d), dtype=np.uint16)
    paref.copy_blocks(kp, vp, np.array([pair], np.int32))
    paref.reshape_and_cache(k, k.copy(), kp, vp, np.array([slot], np.int32))
    assert np.array_equal(kp[1, :, :2], orig[:, :2])
    assert np.array_equal(kp[1, :, 2], k[0])
    assert np.array_equal(kp[0], orig)
