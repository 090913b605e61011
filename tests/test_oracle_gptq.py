"""Pins of the oracle's error-compensated (GPTQ-style) BFP encoding.

What fixes it, besides itself:
  * with a diagonal Hessian (uncorrelated calibration inputs) no error moves to another column, so
    the result must be plain round-to-nearest (``oracle.encode``, itself pinned by brute force);
  * GPTQ's Cholesky form equals the optimal-brain-quantiser form it was derived from (Frantar et
    al. 2022): after each column the remaining weights move by -(w_j - q_j) / [H_F^-1]_jj times
    row j of H_F^-1, and H_F^-1 loses column j by one step of Gaussian elimination. A scalar
    restatement of that form on tiny inputs must give the same codes;
  * every stored block is what round-to-nearest gives for its own decoded values (the Qwen3.8-27B
    gptq-ctx2 card: the runtime's conversion reproduces the GPTQ values bit for bit);
  * on correlated calibration inputs the layer-output error ||(W - Q) X^T|| is clearly smaller
    than round-to-nearest's, which is what the method is for.
"""
import math

import numpy as np
import pytest

import oracle


def correlated_inputs(seed, t, k, mix=0.9, sample_seed=0):
    """t samples of k correlated inputs: N(0, 1) vectors through a fixed mixing matrix (drawn from seed)
    and per-input scales; sample_seed picks the samples."""
    rng = np.random.default_rng(seed)
    a = np.eye(k) + mix * rng.standard_normal((k, k)) / math.sqrt(k)
    scale = np.exp(rng.standard_normal(k) * 0.5)
    z = np.random.default_rng([seed, sample_seed]).standard_normal((t, k))
    return ((z @ a) * scale).astype(np.float32)


def weights(seed, n, k, std=0.02):
    return (np.random.default_rng(seed).standard_normal((n, k)) * std).astype(np.float32)


@pytest.mark.parametrize("fmt", [4, 8])
@pytest.mark.parametrize("n,k", [(4, 16), (16, 64), (7, 160)])
def test_diagonal_hessian_is_round_to_nearest(fmt, n, k):
    w = weights(10 + n + k, n, k)
    w[0, :16] = [1.5, 1.25, 1.75, 0.625, -0.375, 1.9999999, -1.9999999, 0.0625] * 2  # ties, saturation
    d = np.exp(np.random.default_rng(3).standard_normal(k)).astype(np.float32)
    x = np.diag(d)  # k calibration inputs, one per column: H diagonal
    for xx in (x, np.eye(k, dtype=np.float32)):
        e, c = oracle.gptq_encode(fmt, w, oracle.gptq_factor(xx))
        e_r, c_r = oracle.encode(fmt, w)
        assert np.array_equal(e, e_r) and np.array_equal(c, c_r)


def _quantise_scalar(v, E, mb):
    """One value on a block's grid, from Python floats: magnitude and value."""
    if E == 0 or v == 0.0 or abs(v) < 2.0 ** -126:
        return 0, 0.0
    s = E - 127 - (mb - 1)
    mag = min(round(abs(v) * 2.0 ** -s), 2 ** mb - 1)  # round(): ties to even
    return mag, math.copysign(mag * 2.0 ** s, v) if mag else 0.0


def _obq_encode(fmt, w, h):
    """Scalar optimal-brain-quantiser form of the same procedure (explicit inverse-Hessian updates)."""
    mb = 3 if fmt == 4 else 7
    n, k = w.shape
    exps = np.zeros((n, k // 16), np.uint8)
    codes = np.zeros((n, k), np.uint8)
    for r in range(n):
        v = [float(a) for a in w[r]]
        hinv = np.linalg.inv(h).tolist()
        for b in range(k // 16):
            j0 = 16 * b
            E = 0
            for j in range(j0, j0 + 16):
                if abs(v[j]) >= 2.0 ** -126:
                    E = max(E, math.frexp(abs(v[j]))[1] + 126)
            mags = []
            for j in range(j0, j0 + 16):
                mag, q = _quantise_scalar(v[j], E, mb)
                mags.append(mag)
                codes[r, j] = ((1 << mb) if (mag and v[j] < 0) else 0) | mag
                d = hinv[j][j]
                for l in range(j + 1, k):
                    v[l] -= (v[j] - q) * hinv[j][l] / d
                # eliminate column j from the inverse Hessian of the columns still free
                for a in range(j + 1, k):
                    fa = hinv[a][j] / d
                    for c in range(j + 1, k):
                        hinv[a][c] -= fa * hinv[j][c]
            if max(mags) == 0:
                E = 0
            while E > 1 and 0 < max(mags) < 2 ** (mb - 1):
                E -= 1
                mags = [2 * m for m in mags]
            for i, j in enumerate(range(j0, j0 + 16)):
                codes[r, j] = (codes[r, j] & (1 << mb)) | mags[i]
            exps[r, b] = E
    return exps, codes


@pytest.mark.parametrize("fmt", [4, 8])
def test_cholesky_form_matches_obq_form(fmt):
    k, n = 32, 6
    x = correlated_inputs(21, 256, k)
    w = weights(22, n, k, std=0.05)
    h = oracle.gptq_hessian(x)
    e, c = oracle.gptq_encode(fmt, w, oracle.gptq_factor(x))
    e_b, c_b = _obq_encode(fmt, w, h)
    assert np.array_equal(e, e_b) and np.array_equal(c, c_b)
    assert not np.array_equal(c, oracle.encode(fmt, w)[1])  # compensation did move some codes


@pytest.mark.parametrize("fmt", [4, 8])
def test_stored_blocks_are_round_to_nearest_fixed_points(fmt):
    k = 128
    x = correlated_inputs(31, 512, k)
    w = weights(32, 24, k)
    w[3, 16:32] = 0.0  # an all-zero block stays zero unless errors flow into it
    e, c = oracle.gptq_encode(fmt, w, oracle.gptq_factor(x))
    vals = oracle.decode(fmt, e, c)
    e2, c2 = oracle.encode(fmt, vals)
    assert np.array_equal(e, e2) and np.array_equal(c, c2)


@pytest.mark.parametrize("fmt", [4, 8])
def test_compensation_lowers_the_layer_output_error(fmt):
    # strongly correlated inputs: the error ratio is about 0.75 for both formats
    k = 256
    x = correlated_inputs(41, 2048, k, mix=3.0)
    w = weights(42, 64, k)
    x_eval = correlated_inputs(41, 2048, k, mix=3.0, sample_seed=1)  # same distribution, other samples
    u = oracle.gptq_factor(x)
    q_g = oracle.decode(fmt, *oracle.gptq_encode(fmt, w, u)).astype(np.float64)
    q_r = oracle.decode(fmt, *oracle.encode(fmt, w)).astype(np.float64)
    wd = w.astype(np.float64)
    err_g = np.linalg.norm((wd - q_g) @ x_eval.T.astype(np.float64))
    err_r = np.linalg.norm((wd - q_r) @ x_eval.T.astype(np.float64))
    assert err_g < 0.85 * err_r, (err_g, err_r)


def test_rows_are_independent():
    k = 64
    x = correlated_inputs(51, 300, k)
    w = weights(52, 10, k)
    u = oracle.gptq_factor(x)
    e, c = oracle.gptq_encode(4, w, u)
    e3, c3 = oracle.gptq_encode(4, w[3:6], u)
    assert np.array_equal(e[3:6], e3) and np.array_equal(c[3:6], c3)


def test_factor_is_the_inverse_hessian_cholesky():
    k = 48
    x = correlated_inputs(61, 200, k)
    u = oracle.gptq_factor(x, damp=0.05)
    h = x.astype(np.float64).T @ x.astype(np.float64) / 200
    h += 0.05 * np.mean(np.diag(h)) * np.eye(k)
    assert np.allclose(np.triu(u), u) and np.all(np.diag(u) > 0)
    assert np.allclose(u.T @ u @ h, np.eye(k), atol=1e-9)


@pytest.mark.parametrize("fmt", [4, 8])
def test_block_whose_maximum_shrinks_is_renormalised(fmt):
    # One block, inputs that are nearly one shared signal (errors flow strongly to the next columns),
    # the block's largest value last and exactly a power of two: compensation pulls it below that
    # power in some rows, whose exponent must then come down (what plain conversion of the values gives).
    rng = np.random.default_rng(5)
    k, n, t = 16, 256, 512
    x = (rng.standard_normal((t, 1)) + 0.3 * rng.standard_normal((t, k))).astype(np.float32)
    w = (rng.uniform(-0.8, 0.8, (n, k)) * 2.0 ** -5).astype(np.float32)
    w[:, 15] = 2.0 ** -5
    e, c = oracle.gptq_encode(fmt, w, oracle.gptq_factor(x))
    e_raw, _ = oracle.encode(fmt, w)
    assert np.sum(e[:, 0] < e_raw[:, 0]) >= 5 and np.all(e[:, 0] <= e_raw[:, 0])
    e2, c2 = oracle.encode(fmt, oracle.decode(fmt, e, c))
    assert np.array_equal(e, e2) and np.array_equal(c, c2)
