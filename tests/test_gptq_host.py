"""The library's error-compensated (GPTQ-style) host encoder against the oracle's.

Each side forms its own factor of the inverse Hessian from the same seeded calibration inputs (the
library by a reversed Cholesky factorisation and a triangular inverse, the oracle by a matrix
inverse and a Cholesky factorisation), so the factors agree to rounding; the codes, decided in fp64
on both sides, must agree bit for bit.
"""
import numpy as np
import pytest

import block_floating_point_gb300 as bfp
import oracle
import synth


def calibration_inputs(seed, t, k, mix=3.0):
    """t samples of k correlated inputs: seeded N(0, 1) vectors through a seeded mixing matrix, with
    per-input scales (the input recipe; no part of the method)."""
    z = synth.normal(seed, 1, (t, k)).astype(np.float64)
    a = np.eye(k) + mix * synth.normal(seed, 2, (k, k)).astype(np.float64) / np.sqrt(k)
    scale = np.exp(0.5 * synth.normal(seed, 3, (k,)).astype(np.float64))
    return ((z @ a) * scale).astype(np.float32)


@pytest.mark.parametrize("k,t", [(16, 40), (64, 256), (256, 1024), (2048, 4096)])
def test_factor_matches_oracle(k, t):
    x = calibration_inputs(100 + k, t, k)
    u_lib = bfp.gptq_factor(x)
    u_or = oracle.gptq_factor(x)
    assert np.array_equal(np.tril(u_lib, -1), np.zeros((k, k)))
    assert np.max(np.abs(u_lib - u_or)) <= 1e-9 * np.max(np.abs(u_or))


@pytest.mark.parametrize("fmt", [4, 8])
@pytest.mark.parametrize("n,k,t", [(1, 16, 64), (37, 64, 300), (16, 512, 1024), (64, 2048, 4096)])
def test_encode_gptq_matches_oracle(fmt, n, k, t):
    x = calibration_inputs(200 + k, t, k)
    w = synth.normal(201 + n, 5, (n, k), std=0.02)
    if n > 5:
        w[1, :] = 0.0
        w[2, :16] = [1.5, 1.25, 1.75, 0.625, -0.375, 1.9999999, -1.9999999, 0.0625] * 2
        w[4, :] *= np.float32(1e3)
    packed = bfp.encode_gptq(fmt, w, bfp.gptq_factor(x))
    e_lib, c_lib = bfp.read_fields(fmt, n, k, packed)
    e_or, c_or = oracle.gptq_encode(fmt, w, oracle.gptq_factor(x))
    assert np.array_equal(e_lib, e_or) and np.array_equal(c_lib, c_or)
    # the stored blocks are what plain conversion gives for the decoded values
    assert np.array_equal(bfp.encode(fmt, bfp.decode_host(fmt, n, k, packed)), packed)


def test_gate_up_gptq_interleaves_row_groups():
    ffn, hidden = 48, 64
    x = calibration_inputs(301, 400, hidden)
    g = synth.normal(302, 1, (ffn, hidden), std=0.02)
    up = synth.normal(302, 2, (ffn, hidden), std=0.02)
    u = bfp.gptq_factor(x)
    e, c = bfp.read_fields(4, 2 * ffn, hidden, bfp.encode_gate_up_gptq(4, g, up, u))
    ge, gc = bfp.read_fields(4, ffn, hidden, bfp.encode_gptq(4, g, u))
    ue, uc = bfp.read_fields(4, ffn, hidden, bfp.encode_gptq(4, up, u))
    for i in range(ffn // 16):
        assert np.array_equal(c[32 * i:32 * i + 16], gc[16 * i:16 * i + 16])
        assert np.array_equal(c[32 * i + 16:32 * i + 32], uc[16 * i:16 * i + 16])
        assert np.array_equal(e[32 * i:32 * i + 16], ge[16 * i:16 * i + 16])
        assert np.array_equal(e[32 * i + 16:32 * i + 32], ue[16 * i:16 * i + 16])


@pytest.mark.parametrize("fmt", [4, 8])
def test_uncorrelated_inputs_give_round_to_nearest(fmt):
    k = 128
    x = np.diag(np.exp(synth.normal(401, 1, (k,)))).astype(np.float32)  # one input per sample: H diagonal
    w = synth.normal(402, 1, (40, k), std=0.02)
    assert np.array_equal(bfp.encode_gptq(fmt, w, bfp.gptq_factor(x)), bfp.encode(fmt, w))


def test_threads_do_not_change_bytes():
    k = 256
    x = calibration_inputs(501, 600, k)
    w = synth.normal(502, 1, (70, k), std=0.02)
    u1 = bfp.gptq_factor(x, threads=1)
    u7 = bfp.gptq_factor(x, threads=7)
    assert np.array_equal(u1, u7)
    assert np.array_equal(bfp.encode_gptq(4, w, u1, threads=1), bfp.encode_gptq(4, w, u1, threads=7))


def test_gptq_error_codes():
    x = calibration_inputs(601, 50, 32)
    u = bfp.gptq_factor(x)
    with pytest.raises(bfp.BFPError) as ei:
        bfp.gptq_factor(x, damp=0.0)
    assert ei.value.code == bfp.BFP_EINVAL
    with pytest.raises(bfp.BFPError) as ei:
        bfp.gptq_factor(np.zeros((10, 32), np.float32))
    assert ei.value.code == bfp.BFP_EINVAL
    bad = x.copy()
    bad[3, 4] = np.nan
    with pytest.raises(bfp.BFPError) as ei:
        bfp.gptq_factor(bad)
    assert ei.value.code == bfp.BFP_ENONFINITE
    w = synth.normal(602, 1, (16, 32), std=0.02)
    w[2, 5] = np.inf
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode_gptq(4, w, u)
    assert ei.value.code == bfp.BFP_ENONFINITE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode_gptq(4, synth.normal(603, 1, (16, 32)), np.zeros((32, 32)))
    assert ei.value.code == bfp.BFP_EINVAL
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode_gptq(4, synth.normal(604, 1, (16, 24)), np.eye(24))
    assert ei.value.code == bfp.BFP_ESHAPE


@pytest.mark.parametrize("fmt", [4, 8])
def test_dead_inputs_and_tiny_calibration_sets(fmt):
    # inputs that never fire (zero columns of x) leave H singular but for the damping; fewer samples
    # than inputs (t < k) likewise: both sides must still agree, and the dead columns move no error
    k = 64
    x = calibration_inputs(701, 40, k)
    x[:, [3, 17, 40, 41]] = 0.0
    w = synth.normal(702, 1, (20, k), std=0.02)
    packed = bfp.encode_gptq(fmt, w, bfp.gptq_factor(x))
    e_lib, c_lib = bfp.read_fields(fmt, 20, k, packed)
    u_or = oracle.gptq_factor(x)
    e_or, c_or = oracle.gptq_encode(fmt, w, u_or)
    assert np.array_equal(e_lib, e_or) and np.array_equal(c_lib, c_or)
    for j in (3, 17, 40, 41):
        assert np.all(u_or[j, j + 1:] == 0.0)


def test_layer_packing_with_error_compensated_experts():
    """pack_experts (the host half of MoELayer.from_source) lays out GPTQ-encoded experts at the same
    strides as plain ones, each expert's bytes those of its own encode calls."""
    hidden, ffn, ne = 64, 32, 3
    src = {e: (synth.normal(801, 3 * e, (ffn, hidden), std=0.02), synth.normal(801, 3 * e + 1, (ffn, hidden), std=0.02),
               synth.normal(801, 3 * e + 2, (hidden, ffn), std=0.02)) for e in range(ne)}
    fac = {e: (bfp.gptq_factor(calibration_inputs(810 + e, 200, hidden)),
               bfp.gptq_factor(calibration_inputs(820 + e, 200, ffn))) for e in range(ne)}
    gu, dn = bfp.pack_experts(hidden, ne, ffn, 4, lambda e: src[e], gptq_factors=lambda e: fac[e])
    gu0, dn0 = bfp.pack_experts(hidden, ne, ffn, 4, lambda e: src[e])
    gub, dnb = bfp.packed_size(4, 2 * ffn, hidden), bfp.packed_size(4, hidden, ffn)
    assert gu.nbytes == gu0.nbytes == ne * gub and dn.nbytes == dn0.nbytes == ne * dnb
    for e in range(ne):
        g, u, d = src[e]
        assert np.array_equal(gu[e * gub:(e + 1) * gub], bfp.encode_gate_up_gptq(4, g, u, fac[e][0]))
        assert np.array_equal(dn[e * dnb:(e + 1) * dnb], bfp.encode_gptq(4, d, fac[e][1]))
        assert np.array_equal(gu0[e * gub:(e + 1) * gub], bfp.encode_gate_up(4, g, u))
        assert np.array_equal(dn0[e * dnb:(e + 1) * dnb], bfp.encode(4, d))
