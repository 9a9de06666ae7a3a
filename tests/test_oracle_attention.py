"""Pins of the oracle's fp64 attention to closed forms, invariants and
special cases that the mathematics fixes."""
import math

import numpy as np
import pytest

from oracle import paref


def bf16_bits(x):
    """float array -> bf16 bit patterns (round to nearest even)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def paged_layout(k_seq, v_seq, lens, bs, nb, rng):
    """Scatter per-sequence contiguous K/V [L, Hkv, d] into a pool through a
    random block table. Returns pools and tables (a test-side layout)."""
    Hkv, d = k_seq[0].shape[1:]
    maxb = max(1, max(-(-L // bs) for L in lens))
    ids = rng.permutation(nb)
    kp = bf16_bits(rng.standard_normal((nb, Hkv, bs, d)))
    vp = bf16_bits(rng.standard_normal((nb, Hkv, bs, d)))
    bt = np.full((len(lens), maxb), -1, dtype=np.int32)
    nxt = 0
    for s, L in enumerate(lens):
        for j in range(-(-L // bs)):
            bt[s, j] = ids[nxt]
            nxt += 1
        for i in range(L):
            kp[bt[s, i // bs], :, i % bs, :] = k_seq[s][i]
            vp[bt[s, i // bs], :, i % bs, :] = v_seq[s][i]
    return kp, vp, bt


def rand_case(rng, lens, Hq, Hkv, d):
    q = bf16_bits(rng.standard_normal((len(lens), Hq, d)))
    k = [bf16_bits(rng.standard_normal((L, Hkv, d))) for L in lens]
    v = [bf16_bits(rng.standard_normal((L, Hkv, d))) for L in lens]
    return q, k, v


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(0)
    q, k, v = rand_case(rng, [1], 4, 2, 16)
    kp, vp, bt = paged_layout(k, v, [1], 16, 4, rng)
    out = paref.attention_paged(q, kp, vp, bt, np.array([1], np.int32), 0.25)
    for h in range(4):
        assert np.array_equal(out[0, h], bits_to_f64(v[0][0, h // 2]))


def test_zero_length_row_is_zero():
    rng = np.random.default_rng(1)
    q, k, v = rand_case(rng, [0, 3], 2, 2, 8)
    kp, vp, bt = paged_layout(k, v, [0, 3], 4, 4, rng)
    out = paref.attention_paged(q, kp, vp, bt, np.array([0, 3], np.int32), 0.5)
    assert np.all(out[0] == 0.0)
    assert np.any(out[1] != 0.0)


@pytest.mark.parametrize("how", ["q_zero", "scale_zero", "equal_keys"])
def test_uniform_weights_give_the_mean(how):
    # Equal scores make every weight 1/n: the output is the plain mean of V.
    rng = np.random.default_rng(2)
    L, Hq, Hkv, d = 37, 4, 4, 16
    q, k, v = rand_case(rng, [L], Hq, Hkv, d)
    scale = 0.3
    if how == "q_zero":
        q[:] = bf16_bits(np.zeros(q.shape))
    elif how == "scale_zero":
        scale = 0.0
    else:
        k[0][:] = k[0][0:1]
    kp, vp, bt = paged_layout(k, v, [L], 8, 8, rng)
    out = paref.attention_paged(q, kp, vp, bt, np.array([L], np.int32), scale)
    mean = bits_to_f64(v[0]).mean(axis=0)            # [Hkv, d]
    np.testing.assert_allclose(out[0], mean, rtol=0, atol=1e-12)


def test_two_keys_logistic_closed_form():
    # q = e0 and keys with only coordinate 0 set give scores scale*a, scale*b;
    # the weights are the logistic function of their difference. Large
    # scores check that the exponentials cannot overflow.
    d = 8
    for a, b, scale in [(1.0, -2.0, 1.0), (3.0, 0.5, 0.7), (1000.0, 999.0, 1.0),
                        (-800.0, -801.5, 1.0), (6.0, 6.0, 2.0)]:
        q = np.zeros((1, 1, d), np.float32)
        q[0, 0, 0] = 1.0
        k = np.zeros((2, 1, d), np.float32)
        k[0, 0, 0], k[1, 0, 0] = a, b
        v = np.zeros((2, 1, d), np.float32)
        v[0, 0, :] = np.arange(d)
        v[1, 0, :] = -np.arange(d) * 0.5 + 3
        qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
        a_, b_ = bits_to_f64(kb)[0, 0, 0], bits_to_f64(kb)[1, 0, 0]
        w0 = 1.0 / (1.0 + math.exp(scale * (b_ - a_)))
        want = w0 * bits_to_f64(vb)[0, 0] + (1 - w0) * bits_to_f64(vb)[1, 0]
        got = paref.attention_contiguous(qb[0], kb, vb, scale)[0]
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)
        rng = np.random.default_rng(3)
        kp, vp, bt = paged_layout([kb], [vb], [2], 4, 3, rng)
        got_p = paref.attention_paged(qb, kp, vp, bt, np.array([2], np.int32), scale)[0, 0]
        np.testing.assert_allclose(got_p, want, rtol=1e-13, atol=1e-13)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    L, d = 50, 32
    q, k, v = rand_case(rng, [L], 1, 1, d)
    k[0][17] = bf16_bits(bits_to_f64(q[0]) * 4.0)   # aligned with q: by far the top score
    kp, vp, bt = paged_layout(k, v, [L], 16, 6, rng)
    out = paref.attention_paged(q, kp, vp, bt, np.array([L], np.int32), 10.0)
    np.testing.assert_allclose(out[0, 0], bits_to_f64(v[0][17, 0]), atol=1e-9)


def test_gqa_equals_mha_on_replicated_heads():
    rng = np.random.default_rng(5)
    lens, Hq, Hkv, d, G = [9, 40, 1], 8, 2, 16, 4
    q, k, v = rand_case(rng, lens, Hq, Hkv, d)
    kp, vp, bt = paged_layout(k, v, lens, 8, 16, rng)
    sl = np.array(lens, np.int32)
    gqa = paref.attention_paged(q, kp, vp, bt, sl, 0.2)
    # query head h reads kv head h // G: replicate each kv head G times
    k_rep = [np.repeat(x, G, axis=1) for x in k]
    v_rep = [np.repeat(x, G, axis=1) for x in v]
    kp2, vp2, bt2 = paged_layout(k_rep, v_rep, lens, 8, 16, rng)
    mha = paref.attention_paged(q, kp2, vp2, bt2, sl, 0.2)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-13)
    # and a different mapping (h % Hkv) would give something else
    k_bad = [np.tile(x, (1, G, 1)) for x in k]
    v_bad = [np.tile(x, (1, G, 1)) for x in v]
    kp3, vp3, bt3 = paged_layout(k_bad, v_bad, lens, 8, 16, rng)
    bad = paref.attention_paged(q, kp3, vp3, bt3, sl, 0.2)
    assert np.abs(bad - gqa).max() > 1e-3


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
def test_paged_equals_contiguous(bs):
    rng = np.random.default_rng(6 + bs)
    lens, Hq, Hkv, d = [1, 15, 16, 17, 100, 33], 4, 2, 32
    q, k, v = rand_case(rng, lens, Hq, Hkv, d)
    nb = sum(-(-L // bs) for L in lens) + 5
    kp, vp, bt = paged_layout(k, v, lens, bs, nb, rng)
    out = paref.attention_paged(q, kp, vp, bt, np.array(lens, np.int32), 0.177)
    for s, L in enumerate(lens):
        ref = paref.attention_contiguous(q[s], k[s], v[s], 0.177)
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-13)


def test_row_subset_matches_full():
    rng = np.random.default_rng(8)
    lens = [30, 5, 64]
    q, k, v = rand_case(rng, lens, 4, 4, 16)
    kp, vp, bt = paged_layout(k, v, lens, 16, 10, rng)
    sl = np.array(lens, np.int32)
    full = paref.attention_paged(q, kp, vp, bt, sl, 0.25)
    rows = np.array([[2, 3], [0, 0], [1, 2]], np.int32)
    sub = paref.attention_paged(q, kp, vp, bt, sl, 0.25, rows=rows)
    for i, (s, h) in enumerate(rows):
        assert np.array_equal(sub[i], full[s, h])


def test_invariant_to_key_order_and_block_placement():
    # Attention is a sum over keys: reordering the (key, value) pairs or
    # moving blocks to other physical ids leaves the output unchanged.
    rng = np.random.default_rng(9)
    L = 45
    q, k, v = rand_case(rng, [L], 2, 2, 16)
    base = paref.attention_contiguous(q[0], k[0], v[0], 0.3)
    perm = rng.permutation(L)
    shuffled = paref.attention_contiguous(q[0], k[0][perm].copy(), v[0][perm].copy(), 0.3)
    np.testing.assert_allclose(shuffled, base, rtol=0, atol=1e-13)
    for trial in range(3):
        kp, vp, bt = paged_layout(k, v, [L], 16, 20, np.random.default_rng(100 + trial))
        out = paref.attention_paged(q, kp, vp, bt, np.array([L], np.int32), 0.3)[0]
        np.testing.assert_allclose(out, base, rtol=0, atol=1e-13)


def test_linear_in_values_and_inside_their_hull():
    rng = np.random.default_rng(10)
    L, d = 25, 16
    q, k, v = rand_case(rng, [L], 1, 1, d)
    v2 = [bf16_bits(rng.standard_normal((L, 1, d)))]
    o1 = paref.attention_contiguous(q[0], k[0], v[0], 0.4)
    o2 = paref.attention_contiguous(q[0], k[0], v2[0], 0.4)
    # values with a dyadic sum that bf16 holds exactly
    vs = bf16_bits(bits_to_f64(v[0]) + bits_to_f64(v2[0]))
    exact = np.array_equal(bits_to_f64(vs), bits_to_f64(v[0]) + bits_to_f64(v2[0]))
    if exact:
        o12 = paref.attention_contiguous(q[0], k[0], vs, 0.4)
        np.testing.assert_allclose(o12, o1 + o2, atol=1e-12)
    vv = bits_to_f64(v[0])[:, 0, :]
    assert np.all(o1[0] <= vv.max(axis=0) + 1e-12)
    assert np.all(o1[0] >= vv.min(axis=0) - 1e-12)


def test_matches_library_softmax_on_tiny_inputs():
    # Brute force on tiny inputs with scipy's softmax as the weights.
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(11)
    for _ in range(20):
        L = int(rng.integers(1, 6))
        q, k, v = rand_case(rng, [L], 2, 1, 4)
        qf, kf, vf = bits_to_f64(q[0]), bits_to_f64(k[0]), bits_to_f64(v[0])
        for h in range(2):
            w = scipy_special.softmax(0.5 * (kf[:, 0, :] @ qf[h]))
            want = w @ vf[:, 0, :]
            got = paref.attention_contiguous(q[0], k[0], v[0], 0.5)[h]
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_bad_table_entry_is_an_error():
    rng = np.random.default_rng(12)
    q, k, v = rand_case(rng, [20], 1, 1, 8)
    kp, vp, bt = paged_layout(k, v, [20], 16, 3, rng)
    bt[0, 1] = 3  # outside the 3-block pool
    with pytest.raises(ValueError):
        paref.attention_paged(q, kp, vp, bt, np.array([20], np.int32), 1.0)
