"""Pins of the oracle's FP8 (E4M3) codec, fp8 cache write and fp8 attention."""
import math

import numpy as np
import pytest

from oracle import paref
from tests.test_oracle_attention import bf16_bits, bits_to_f64, paged_layout, rand_case

FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_known_codes():
    # OCP E4M3: bias 7, subnormals m * 2^-9, max 1.75 * 2^8, S.1111.111 is NaN
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for c, v in table.items():
        assert paref.e4m3_decode(c) == v, hex(c)
    assert math.isnan(paref.e4m3_decode(0x7F)) and math.isnan(paref.e4m3_decode(0xFF))
    assert math.copysign(1.0, paref.e4m3_decode(0x80)) < 0


def test_encode_inverts_decode_on_every_code():
    for c in FINITE:
        assert paref.e4m3_encode(paref.e4m3_decode(c)) == c, hex(c)


def test_encode_is_nearest_with_ties_to_even():
    # brute force: the nearest of all finite codes, even mantissa on a tie
    vals = np.array([paref.e4m3_decode(c) for c in FINITE])
    codes = np.array(FINITE)
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-460, 460, 3000), rng.normal(0, 1, 3000),
                         rng.normal(0, 2.0 ** -7, 1000)])
    for x in xs:
        d = np.abs(vals - x)
        best = codes[d == d.min()]
        if len(best) > 1:  # a tie (or +-0): prefer the even code of the right sign
            best = [b for b in best if (b & 1) == 0 and (b >> 7) == (x < 0)] or best
        want = best[0] if abs(x) < 448 else (0xFE if x < 0 else 0x7E)
        assert paref.e4m3_encode(x) == want or paref.e4m3_decode(paref.e4m3_encode(x)) == \
            paref.e4m3_decode(want), x
    assert paref.e4m3_encode(1.0625) == 0x38          # tie: 1.0 (even) not 1.125
    assert paref.e4m3_encode(1.1875) == 0x3A          # tie: 1.25 (even) not 1.125
    assert paref.e4m3_encode(2.0 ** -10) == 0x00      # tie between 0 and 2^-9
    assert paref.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie between 2^-9 and 2*2^-9
    assert paref.e4m3_encode(1e6) == 0x7E and paref.e4m3_encode(-1e6) == 0xFE
    assert paref.e4m3_encode(float("nan")) == 0x7F


def test_fp8_attention_equals_bf16_attention_on_the_same_values():
    # Codes times a power-of-two scale are exact in bf16, so fp8 attention must
    # equal the (already pinned) bf16 attention on those values.
    rng = np.random.default_rng(1)
    lens, Hq, Hkv, d, bs = [1, 17, 40, 5], 8, 2, 32, 16
    q, _, _ = rand_case(rng, lens, Hq, Hkv, d)
    codes = np.array(FINITE, np.uint8)
    nb = sum(-(-L // bs) for L in lens) + 3
    kc = rng.choice(codes[np.abs([paref.e4m3_decode(c) for c in codes]) < 8],
                    size=(nb, Hkv, bs, d)).astype(np.uint8)
    vc = rng.choice(codes, size=(nb, Hkv, bs, d)).astype(np.uint8)
    k_scale, v_scale = 0.5, 2.0 ** -5
    dec = np.vectorize(paref.e4m3_decode)
    kb = bf16_bits(dec(kc) * k_scale)
    vb = bf16_bits(dec(vc) * v_scale)
    assert np.array_equal(bits_to_f64(kb), dec(kc) * k_scale)
    bt = np.full((len(lens), 4), -1, np.int32)
    ids = rng.permutation(nb)
    nxt = 0
    for s, L in enumerate(lens):
        for j in range(-(-L // bs)):
            bt[s, j] = ids[nxt]
            nxt += 1
    sl = np.array(lens, np.int32)
    got = paref.attention_paged_fp8(q, kc, vc, bt, sl, 0.3, k_scale, v_scale)
    want = paref.attention_paged(q, kb, vb, bt, sl, 0.3)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_fp8_cache_write_codes():
    rng = np.random.default_rng(2)
    T, Hkv, d, bs, nb = 6, 2, 16, 8, 5
    k = bf16_bits(rng.normal(0, 3, (T, Hkv, d)))
    v = bf16_bits(rng.normal(0, 3, (T, Hkv, d)))
    kp = rng.integers(0, 256, (nb, Hkv, bs, d), dtype=np.uint8)
    vp = kp.copy()
    kp0 = kp.copy()
    slots = np.array([0, 9, -1, 39, 17, 40 * 9], np.int32)
    k_scale, v_scale = np.float32(0.037), np.float32(1.7)
    assert paref.reshape_and_cache_fp8(k, v, kp, vp, slots, k_scale, v_scale) == 1
    kf = bits_to_f64(k).astype(np.float32)
    for t, slot in enumerate(slots):
        if slot < 0 or slot >= nb * bs:
            continue
        b, o = divmod(int(slot), bs)
        want = [paref.e4m3_encode(float(np.float32(x) / k_scale)) for x in kf[t].ravel()]
        assert list(kp[b, :, o].ravel()) == want
    untouched = np.ones((nb, bs), bool)
    for s in slots:
        if 0 <= s < nb * bs:
            untouched[s // bs, s % bs] = False
    assert np.array_equal(kp.transpose(0, 2, 1, 3)[untouched], kp0.transpose(0, 2, 1, 3)[untouched])


def test_encode_matches_torch_float8_in_range():
    # An independent implementation of the same format: torch's float8_e4m3fn
    # cast (round to nearest even). Outside +-448 torch gives NaN where the
    # cache write saturates, so only in-range values are compared.
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(-447, 447, 20000), rng.normal(0, 1, 20000),
                         rng.normal(0, 2.0 ** -8, 5000)]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([paref.e4m3_encode(float(x)) for x in xs], np.uint8)
    same = (got == want) | ((got & 0x7F) == 0) & ((want & 0x7F) == 0)
    assert same.all(), xs[~same][:5]
    codes = np.arange(256, dtype=np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([paref.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(np.isnan(dec), np.isnan(mine))
    assert np.array_equal(dec[~np.isnan(dec)], mine[~np.isnan(mine)])
