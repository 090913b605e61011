"""Pins for the oracle's BFP encode/decode (no GPU).

The pages print no worked BFP values, so the encoder is pinned by:
  * an independent exact-rational statement of round-to-nearest over the set
    of values a block can hold (Python ``fractions``), on random and
    adversarial blocks (ties at exactly half a step, overflow into
    saturation, zeros, signed zeros, subnormals, powers of two);
  * hand-worked blocks written out below;
  * the invariants the pages state or imply: every stored value is exactly
    representable, so re-encoding reproduces it bit for bit (Qwen3.8-27B
    gptq-ctx2 card, "What changed in this release"), and the block maximum
    keeps its exponent;
  * the storage costs printed on the pages (tests/golden/storage_sizes.json).
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


def bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


def brute_block(fmt, vals):
    """Nearest representable value by exhaustive search over magnitudes (exact rationals).

    The block exponent is the largest fp32 exponent field among the values
    (zero and subnormal inputs count as 0); the block can hold
    +-m * 2^(E-127-(mb-1)), m = 0 .. 2^mb - 1. Each value goes to the nearest
    one; on an exact tie the even m wins. Returns (E, [code]).
    """
    mb = {4: 3, 8: 7}[fmt]
    fields = [(bits(v) >> 23) & 0xFF for v in vals]
    E = max(fields)
    step = Fraction(2) ** (E - 127 - (mb - 1))
    codes = []
    for v, e in zip(vals, fields):
        if e == 0:
            codes.append(0)
            continue
        x = Fraction(v)
        mag = abs(x)
        best = None
        for m in range(2 ** mb):
            d = abs(mag - m * step)
            if best is None or d < best[0] or (d == best[0] and m % 2 == 0):
                best = (d, m)
        m = best[1]
        s = 1 if (x < 0 and m != 0) else 0
        codes.append((s << mb) | m)
    return E, codes


def enc(fmt, vals):
    e, c = oracle.encode(fmt, np.array([vals], dtype=np.float32))
    return int(e[0, 0]), [int(v) for v in c[0]]


@pytest.mark.parametrize("fmt", [4, 8])
def test_encode_matches_brute_force_random(fmt):
    rng = np.random.default_rng(1234 + fmt)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-30, 30)
        vals = (rng.standard_normal(16) * scale).astype(np.float32)
        if trial % 5 == 0:
            vals[rng.integers(0, 16, 4)] = 0.0
        if trial % 7 == 0:  # wide dynamic range inside one block
            vals *= (10.0 ** rng.uniform(-8, 0, 16)).astype(np.float32)
        assert enc(fmt, list(vals)) == brute_block(fmt, [float(v) for v in vals]), vals


@pytest.mark.parametrize("fmt", [4, 8])
def test_encode_exact_ties_round_to_even(fmt):
    mb = {4: 3, 8: 7}[fmt]
    # Block maximum 2^(mb-1) * 2 = leading value 1.0 * 2^0 ... use E = 127 (max value in [1, 2)).
    step = 2.0 ** (0 - (mb - 1))
    for m in range(0, 2 ** mb - 1):
        tie = (m + 0.5) * step  # exactly halfway between m and m+1 steps
        vals = [1.5] + [tie, -tie] + [0.0] * 13
        E, codes = enc(fmt, vals)
        assert E == 127
        want = m if m % 2 == 0 else m + 1
        assert codes[1] == want, (m, codes[1])
        assert codes[2] == ((1 << mb) | want if want else 0)
        assert (E, codes) == brute_block(fmt, vals)


@pytest.mark.parametrize("fmt", [4, 8])
def test_encode_saturates_instead_of_bumping_exponent(fmt):
    mb = {4: 3, 8: 7}[fmt]
    # 1.9999999 has exponent field 127 and would round to 2^mb steps: saturate to 2^mb - 1.
    v = f32(0x3FFFFFFF)
    E, codes = enc(fmt, [v, -v] + [0.25] * 14)
    assert E == 127
    assert codes[0] == (1 << mb) - 1
    assert codes[1] == (1 << mb) | ((1 << mb) - 1)
    assert (E, codes) == brute_block(fmt, [v, -v] + [0.25] * 14)


@pytest.mark.parametrize("fmt", [4, 8])
def test_encode_zero_signed_zero_subnormal_and_powers_of_two(fmt):
    mb = {4: 3, 8: 7}[fmt]
    assert enc(fmt, [0.0] * 16) == (0, [0] * 16)
    assert enc(fmt, [-0.0] * 16) == (0, [0] * 16)
    sub = f32(0x00000001)
    assert enc(fmt, [sub, -sub] + [0.0] * 14) == (0, [0] * 16)
    # powers of two with the block max 1.0: 2^-j is m = 2^(mb-1-j) steps, exact until it underflows
    vals = [2.0 ** -j for j in range(16)]
    E, codes = enc(fmt, vals)
    assert E == 127
    for j, c in enumerate(codes):
        # 2^-mb is exactly half a step: the tie goes to the even magnitude 0
        assert c == (2 ** (mb - 1 - j) if j <= mb - 1 else 0), (j, c)
    assert (E, codes) == brute_block(fmt, vals)


def test_encode_hand_worked_bfp4_block():
    # Block max 3.0 -> E = 128, step = 2^(128-127-2) = 0.5. Magnitudes in steps:
    #   3.0 -> 6; 1.25 -> 2.5 -> tie -> even 2; 1.75 -> 3.5 -> tie -> even 4;
    #   -0.3 -> 0.6 -> 1 (negative: 0b1001 = 9); 0.2 -> 0.4 -> 0; 3.6 would be 7.2 but E is from 3.0's field
    #   (3.6 also has field 128) -> 7.2 -> 7; -3.9 -> 7.8 -> 8 -> saturates to 7 -> 0b1111 = 15.
    vals = [3.0, 1.25, 1.75, -0.3, 0.2, 3.6, -3.9] + [0.0] * 9
    E, codes = enc(4, vals)
    assert E == 128
    assert codes[:7] == [6, 2, 4, 9, 0, 7, 15]


def test_encode_hand_worked_bfp8_block():
    # Block max 0.02 -> field 121 (0.02 in [2^-6, 2^-5)), step = 2^(121-127-6) = 2^-12.
    #   0.02 / 2^-12 = 81.92 -> 82;  -0.001 / 2^-12 = 4.096 -> 4 -> sign bit: 128 + 4 = 132;
    #   2^-13 = half a step -> tie -> even 0.
    vals = [0.02, -0.001, 2.0 ** -13] + [0.0] * 13
    E, codes = enc(8, vals)
    assert E == 121
    assert codes[:3] == [82, 132, 0]


def test_encode_rejects_non_finite():
    for bad in (float("inf"), float("-inf"), float("nan")):
        with pytest.raises(ValueError):
            oracle.encode(4, np.array([[bad] + [0.0] * 15], dtype=np.float32))


@pytest.mark.parametrize("fmt", [4, 8])
def test_decoded_values_representable_idempotent_and_max_exponent_kept(fmt):
    mb = {4: 3, 8: 7}[fmt]
    w = synth.normal(7, 99 + fmt, (64, 256), std=0.02)
    e, c = oracle.encode(fmt, w)
    d = oracle.decode(fmt, e, c)
    # every decoded value is a whole number of steps of its block
    for r in range(0, 64, 7):
        for b in range(16):
            step = Fraction(2) ** (int(e[r, b]) - 127 - (mb - 1))
            for j in range(16):
                q = Fraction(float(d[r, 16 * b + j])) / step
                assert q.denominator == 1 and abs(q) < 2 ** mb
    # re-encoding the decoded matrix reproduces it bit for bit
    e2, c2 = oracle.encode(fmt, d)
    assert np.array_equal(e, e2) and np.array_equal(c, c2)
    # the block maximum keeps its fp32 exponent field
    fields = (d.view(np.uint32) >> 23) & 0xFF
    assert np.array_equal(fields.reshape(64, 16, 16).max(axis=2), e)
    # and each value is within half a step of its source (or saturated at the top)
    step = np.ldexp(1.0, e.astype(np.int32) - 127 - (mb - 1)).repeat(16, axis=1)
    err = np.abs(d.astype(np.float64) - w.astype(np.float64))
    saturated = np.abs(w.astype(np.float64)) >= (2 ** mb - 0.5) * step
    assert np.all(err[~saturated] <= 0.5 * step[~saturated])
    assert np.all(err[saturated] <= step[saturated])
    assert np.all(np.abs(d[saturated]) == (2 ** mb - 1) * step[saturated])


@pytest.mark.parametrize("fmt", [4, 8])
def test_storage_cost_matches_the_pages(fmt):
    g = json.load(open(os.path.join(GOLDEN, "storage_sizes.json")))
    assert g["block_size"]["values_per_block"] == 16
    bfp8 = oracle.storage_bytes_per_value(8)
    bfp4 = oracle.storage_bytes_per_value(4)
    kv = g["bfp8_kv_cache"]
    # bf16 is 2 bytes/value: the BFP8 cache is 20.0 * 1.0625 / 2 KiB, printed to one decimal
    assert round(kv["bf16_kib_per_token"] * bfp8 / 2.0, kv["printed_decimals"]) == kv["bfp8_kib_per_token_printed"]
    v = g["bfp4_v_cache"]
    s = v["bytes_per_token_k_bfp8_v_bfp8"] / (2 * bfp8)  # values per token for each of K and V
    assert s == int(s) == 16384
    assert s * bfp8 + s * bfp4 == v["bytes_per_token_k_bfp8_v_bfp4"]
    assert oracle.storage_bytes_per_value(fmt) == {4: 0.5625, 8: 1.0625}[fmt]


def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and l[0] != "#"]
    for r in rows:
        v = [int(t, 16) for t in r]
        out = synth.philox4x32_10(v[0:4], v[4:6])
        assert [int(o) for o in out] == v[6:10]
