"""Pins of the oracle's chunked-prefill attention: causal closed forms, a
one-hot key seen only from its own position on, and agreement with the
(separately pinned) decode routine at every chunk position."""
import numpy as np
import pytest

from oracle import paref
from tests.test_oracle_attention import bf16_bits, bits_to_f64, paged_layout


def chunk_case(rng, lens, chunks, Hq, Hkv, d, bs=16, equal_keys=False):
    k = [bf16_bits(rng.standard_normal((L, Hkv, d))) for L in lens]
    if equal_keys:
        k = [np.repeat(x[:1], len(x), axis=0) for x in k]
    v = [bf16_bits(rng.standard_normal((L, Hkv, d))) for L in lens]
    nb = sum(-(-L // bs) for L in lens) + 4
    kp, vp, bt = paged_layout(k, v, lens, bs, nb, rng)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = bf16_bits(rng.standard_normal((int(cu[-1]), Hq, d)))
    return q, k, v, kp, vp, bt, np.array(lens, np.int32), cu


def test_equal_keys_give_the_causal_running_mean_of_values():
    # all keys of a sequence equal -> uniform weights over positions 0..p
    rng = np.random.default_rng(0)
    lens, chunks, Hq, Hkv, d = [40, 9, 33], [12, 9, 1], 4, 2, 16
    q, k, v, kp, vp, bt, sl, cu = chunk_case(rng, lens, chunks, Hq, Hkv, d, equal_keys=True)
    out = paref.prefill_paged(q, kp, vp, bt, sl, cu, 0.3)
    for s, (L, c) in enumerate(zip(lens, chunks)):
        vals = bits_to_f64(v[s])  # [L, Hkv, d]
        for i in range(c):
            p = L - c + i
            for h in range(Hq):
                want = vals[:p + 1, h // (Hq // Hkv)].mean(axis=0)
                np.testing.assert_allclose(out[cu[s] + i, h], want, rtol=0, atol=1e-12)


def test_a_dominant_key_is_seen_only_from_its_position_on():
    rng = np.random.default_rng(1)
    L, c, d, j0 = 30, 30, 16, 11
    q, k, v, kp, vp, bt, sl, cu = chunk_case(rng, [L], [c], 1, 1, d)
    qv = bits_to_f64(q)
    # make key j0 align with every query and dwarf the rest
    big = bf16_bits(np.sign(qv[:, 0].sum(axis=0)) * 8.0)
    kp[bt[0, j0 // 16], 0, j0 % 16] = big
    for i in range(c):  # the queries all point the same way
        q[i, 0] = bf16_bits(np.abs(qv[0, 0]) * np.sign(qv[:, 0].sum(axis=0)))
    out = paref.prefill_paged(q, kp, vp, bt, sl, cu, 4.0)
    vj0 = bits_to_f64(vp[bt[0, j0 // 16], 0, j0 % 16])
    for i in range(c):
        if i >= j0:
            np.testing.assert_allclose(out[i, 0], vj0, atol=1e-6)
        else:
            assert np.abs(out[i, 0] - vj0).max() > 0.1  # key j0 is in its future


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_every_chunk_row_equals_decode_at_its_length(bs):
    rng = np.random.default_rng(bs)
    lens, chunks, Hq, Hkv, d = [50, 17, 64, 3], [7, 17, 1, 3], 8, 2, 32
    q, k, v, kp, vp, bt, sl, cu = chunk_case(rng, lens, chunks, Hq, Hkv, d, bs=bs)
    out = paref.prefill_paged(q, kp, vp, bt, sl, cu, 0.2)
    for s, (L, c) in enumerate(zip(lens, chunks)):
        for i in range(c):
            p = L - c + i
            dec = paref.attention_paged(q[cu[s] + i][None], kp, vp, bt[s][None],
                                        np.array([p + 1], np.int32), 0.2)
            np.testing.assert_allclose(out[cu[s] + i], dec[0], rtol=0, atol=1e-12)


def test_rows_subset_and_bad_chunk():
    rng = np.random.default_rng(3)
    q, k, v, kp, vp, bt, sl, cu = chunk_case(rng, [20, 5], [4, 5], 4, 4, 16)
    full = paref.prefill_paged(q, kp, vp, bt, sl, cu, 0.25)
    rows = np.array([[0, 3], [8, 0], [5, 2]], np.int32)
    sub = paref.prefill_paged(q, kp, vp, bt, sl, cu, 0.25, rows=rows)
    for r, (row, h) in enumerate(rows):
        assert np.array_equal(sub[r], full[row, h])
    with pytest.raises(ValueError):  # a chunk longer than the sequence
        paref.prefill_paged(q, kp, vp, bt, np.array([20, 4], np.int32), cu, 0.25)
