"""Pins of the oracle's BFP KV-cache codec and decode attention.

  * the fast transform equals the Sylvester Hadamard matrix (scipy.linalg.hadamard) on integer
    inputs, where fp32 is exact, and applying it twice gives d times the input;
  * the cache fields are the plain encoder's fields of the (rotated) rows, and rotated rows decode
    back to the bf16 input within the BFP error;
  * attention reduces to closed forms: one cached token gives its V row, identical keys or a zero
    query give the mean of the V rows, a dominant key gives its row, and each query head reads the
    KV head of its group; on random inputs it equals a direct softmax (scipy.special.softmax).
"""
import numpy as np
import pytest
from scipy.linalg import hadamard
from scipy.special import softmax

import oracle
import synth


def bf16(a):
    return synth.to_bf16_bits(np.asarray(a, dtype=np.float32))


def f32(b):
    return synth.bf16_bits_to_f32(b)


@pytest.mark.parametrize("d", [16, 64, 256])
def test_fwht_is_the_sylvester_hadamard_matrix(d):
    x = np.random.default_rng(d).integers(-50, 50, (5, d)).astype(np.float32)
    assert np.array_equal(oracle.fwht_f32(x), (x.astype(np.float64) @ hadamard(d)).astype(np.float32))
    assert np.array_equal(oracle.fwht_f32(oracle.fwht_f32(x)), d * x)


@pytest.mark.parametrize("fmt,rotate", [(8, False), (4, True), (8, True), (4, False)])
def test_cache_fields_are_the_encoder_fields(fmt, rotate):
    d = 128
    rows = bf16(synth.normal(3, 1, (2, 7, d)))
    e, c = oracle.kv_encode(fmt, rows, rotate)
    src = f32(rows).reshape(-1, d)
    e2, c2 = oracle.encode(fmt, oracle.fwht_f32(src) if rotate else src)
    assert np.array_equal(e.reshape(-1, d // 16), e2) and np.array_equal(c.reshape(-1, d), c2)
    back = oracle.kv_decode(fmt, e, c, rotate)
    rel = np.max(np.abs(back - f32(rows))) / np.max(np.abs(f32(rows)))
    assert rel < (0.2 if fmt == 4 else 0.02)


def cache(seed, kvh, n, d, k_fmt=8, v_fmt=8, rot=False, k=None, v=None):
    k = bf16(synth.normal(seed, 1, (kvh, n, d))) if k is None else k
    v = bf16(synth.normal(seed, 2, (kvh, n, d))) if v is None else v
    return oracle.kv_encode(k_fmt, k, False), oracle.kv_encode(v_fmt, v, rot), k, v


@pytest.mark.parametrize("v_fmt,rot", [(8, False), (4, True)])
def test_single_token_gives_its_value_row(v_fmt, rot):
    d, kvh = 64, 2
    kf, vf, _, _ = cache(11, kvh, 1, d, v_fmt=v_fmt, rot=rot)
    q = bf16(synth.normal(11, 3, (4, d)))
    out = oracle.attn_decode(q, kf, vf, 1, 0.125, 8, v_fmt, rot)
    vrow = oracle.kv_decode(v_fmt, vf[0], vf[1], rot)
    for j in range(4):
        assert np.allclose(out[j], vrow[j // 2, 0], rtol=0, atol=1e-12)


def test_equal_keys_and_zero_query_average_the_values():
    d, kvh, n = 32, 1, 9
    k = np.repeat(bf16(synth.normal(21, 1, (kvh, 1, d))), n, axis=1)
    kf, vf, _, v = cache(21, kvh, n, d, k=k)
    vd = oracle.kv_decode(8, vf[0], vf[1], False)
    q = bf16(synth.normal(21, 3, (2, d)))
    out = oracle.attn_decode(q, kf, vf, n, 0.3, 8, 8, False)
    assert np.allclose(out, vd[0].mean(axis=0)[None, :], rtol=0, atol=1e-12)
    kf2, vf2, _, _ = cache(22, kvh, n, d, v=v)
    out0 = oracle.attn_decode(np.zeros((2, d), np.uint16), kf2, vf2, n, 0.3, 8, 8, False)
    assert np.allclose(out0, vd[0].mean(axis=0)[None, :], rtol=0, atol=1e-12)


def test_dominant_key_and_head_groups():
    d, kvh, n, g = 32, 2, 12, 3
    k = np.zeros((kvh, n, d), np.float32)
    k[0, 5, :] = 4.0   # head 0: token 5 dominates any query along +1
    k[1, 8, :] = 4.0   # head 1: token 8
    kf, vf, _, _ = cache(31, kvh, n, d, k=bf16(k))
    vd = oracle.kv_decode(8, vf[0], vf[1], False)
    q = bf16(np.ones((kvh * g, d)))
    out = oracle.attn_decode(q, kf, vf, n, 1.0, 8, 8, False)  # score gap 128: weights 1 and e^-128
    for j in range(kvh * g):
        assert np.allclose(out[j], vd[j // g, 5 if j < g else 8], rtol=0, atol=1e-12)


@pytest.mark.parametrize("v_fmt,rot", [(8, False), (4, True)])
def test_matches_a_direct_softmax(v_fmt, rot):
    d, kvh, n, g = 64, 2, 50, 4
    kf, vf, _, _ = cache(41, kvh, n, d, v_fmt=v_fmt, rot=rot)
    q = bf16(synth.normal(41, 3, (kvh * g, d)))
    out = oracle.attn_decode(q, kf, vf, n, 0.125, 8, v_fmt, rot)
    kd = oracle.decode(8, kf[0].reshape(-1, d // 16), kf[1].reshape(-1, d)).reshape(kvh, n, d).astype(np.float64)
    vd = oracle.kv_decode(v_fmt, vf[0], vf[1], rot)
    qf = f32(q).astype(np.float64)
    for j in range(kvh * g):
        p = softmax(0.125 * np.einsum("td,d->t", kd[j // g], qf[j]))
        assert np.allclose(out[j], np.einsum("t,td->d", p, vd[j // g]), rtol=1e-12, atol=1e-14)
    # only the first n_ctx tokens count
    out_short = oracle.attn_decode(q, kf, vf, 20, 0.125, 8, v_fmt, rot)
    p = softmax(0.125 * kd[0, :20] @ qf[0])
    assert np.allclose(out_short[0], p @ vd[0, :20], rtol=1e-12, atol=1e-14)
