"""Pins for the oracle's linear, routing, MoE layer and stack pieces (no GPU).

What pins each piece (none of them reuses the oracle's own loops):
  * linear / router logits: fp64 NumPy matmul on the decoded weights;
  * routing: brute-force sort of (-logit, index) pairs, softmax in NumPy,
    renormalised weights summing to one;
  * MoE layer: a dense NumPy evaluation on tiny shapes, plus identities that
    a dropped term, a wrong sign or a transposed operand would break:
      - top-k = all experts with identical experts equals one expert (plus shared),
      - an all-zero expert contributes nothing,
      - a zero shared gate vector scales the shared expert by sigmoid(0) = 1/2,
      - M rows together equal M single-row calls;
  * RMSNorm / residual: NumPy fp32 statement of the same formula.
"""
import numpy as np
import pytest

import oracle
import synth


def bf16(a):
    return synth.to_bf16_bits(np.asarray(a, dtype=np.float32))


def f32_of(b):
    return synth.bf16_bits_to_f32(b)


def rand_bf16(seed, shape, std=1.0):
    return bf16(np.random.default_rng(seed).standard_normal(shape) * std)


@pytest.mark.parametrize("fmt", [4, 8])
@pytest.mark.parametrize("m,n,k", [(1, 16, 16), (3, 40, 96), (16, 128, 512)])
def test_linear_matches_numpy_fp64(fmt, m, n, k):
    w = synth.normal(3, 1000 + n, (n, k), std=0.02)
    e, c = oracle.encode(fmt, w)
    wd = oracle.decode(fmt, e, c).astype(np.float64)
    x = rand_bf16(n + k, (m, k))
    y, yb = oracle.linear(fmt, e, c, x)
    ref = f32_of(x).astype(np.float64) @ wd.T
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - ref) <= ulp)  # one rounding to fp32 from an exact-ish sum
    assert np.array_equal(yb, bf16(y))  # bf16 output is the RNE of the fp32 value


def test_linear_identity_block_is_exact():
    # W = I (16x16): every row has one 1.0 -> E = 127, code 2^(mb-1); y = x exactly.
    for fmt in (4, 8):
        e, c = oracle.encode(fmt, np.eye(16, dtype=np.float32))
        x = rand_bf16(5, (4, 16))
        y, yb = oracle.linear(fmt, e, c, x)
        assert np.array_equal(y, f32_of(x))
        assert np.array_equal(yb, x)


def test_router_logits_match_numpy():
    wr = rand_bf16(11, (37, 64), 0.02)
    x = rand_bf16(12, (5, 64))
    bias = np.random.default_rng(13).standard_normal(37).astype(np.float32)
    l = oracle.router_logits(wr, x)
    ref = (f32_of(x).astype(np.float64) @ f32_of(wr).astype(np.float64).T).astype(np.float32)
    assert np.array_equal(l, ref)
    lb = oracle.router_logits(wr, x, bias)
    assert np.array_equal(lb, (ref + bias).astype(np.float32))


def test_routing_brute_force():
    rng = np.random.default_rng(21)
    for trial in range(200):
        e = int(rng.integers(2, 300))
        k = int(rng.integers(1, min(e, 9) + 1))
        l = rng.standard_normal(e).astype(np.float32)
        if trial % 4 == 0:  # force ties
            l = np.round(l * 2) / 2
        idx, w = oracle.route_row(l, k)
        order = sorted(range(e), key=lambda i: (-float(l[i]), i))[:k]
        assert list(idx) == order
        p = np.exp(l.astype(np.float64) - l.max())
        p /= p.sum()
        assert np.allclose(w, p[order] / p[order].sum(), rtol=1e-12, atol=0)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(np.diff(w) <= 1e-15)  # slots come in descending weight


def make_layer(seed, spec, identical=False, zero_expert=None, zero_gate=False, fmt=4):
    lw = synth.LayerWeights(spec, seed)

    def source(e):
        key = synth.SHARED_EXPERT if e == "shared" else (0 if identical else e)
        g, u, d = lw.gate(key), lw.up(key), lw.down(key)
        if zero_expert is not None and e == zero_expert:
            g, u, d = g * 0, u * 0, d * 0
        return g, u, d

    router = lw.router_bf16()
    sg = lw.shared_gate_bf16()
    if zero_gate:
        sg = np.zeros_like(sg)
    return dict(router_bf16=router, shared_gate_bf16=sg, experts=oracle.ExpertCache(fmt, source), top_k=spec.top_k)


def dense_numpy_layer(x_bf16, args, n_experts, fmt=4):
    """Independent NumPy statement of the MoE layer on decoded weights (tiny shapes)."""
    x = f32_of(x_bf16).astype(np.float64)
    wr = f32_of(args["router_bf16"]).astype(np.float64)
    logits = (x @ wr.T).astype(np.float32)
    k = args["top_k"]
    cache = args["experts"]

    def ffn(key, xr):
        ex = cache(key)
        G = oracle.decode(fmt, *ex.g).astype(np.float64)
        U = oracle.decode(fmt, *ex.u).astype(np.float64)
        D = oracle.decode(fmt, *ex.d).astype(np.float64)
        a, b = G @ xr, U @ xr
        return D @ (a / (1.0 + np.exp(-a)) * b)

    y = np.zeros_like(x)
    for r in range(x.shape[0]):
        order = sorted(range(n_experts), key=lambda i: (-float(logits[r, i]), i))[:k]
        p = np.exp(logits[r].astype(np.float64) - logits[r].max())
        p /= p.sum()
        w = p[order] / p[order].sum()
        for s, ei in enumerate(order):
            y[r] += w[s] * ffn(ei, x[r])
        gs = 1.0 / (1.0 + np.exp(-(f32_of(args["shared_gate_bf16"]).astype(np.float64) @ x[r])))
        y[r] += gs * ffn("shared", x[r])
    return y


TINY = synth.TINY


def tol_ok(got, ref, rel=1e-9):
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    return np.all(np.abs(np.asarray(got, dtype=np.float64) - ref) <= rel * (np.abs(ref) + rms) + 1e-30)


def test_moe_layer_matches_dense_numpy():
    args = make_layer(31, TINY)
    x = rand_bf16(32, (3, TINY.hidden))
    y, idx, w = oracle.moe_layer(x, **args)
    ref = dense_numpy_layer(x, args, TINY.n_experts)
    assert tol_ok(y, ref, 1e-6)  # y is fp32-rounded; ref fp64
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_moe_topk_all_identical_experts_equals_one_expert():
    spec = synth.MoESpec(64, 6, 32, 6, 32)
    args = make_layer(41, spec, identical=True)
    x = rand_bf16(42, (2, spec.hidden))
    y, idx, w = oracle.moe_layer(x, **args)
    ex = args["experts"]
    for r in range(2):
        one = ex(0).ffn_row(x[r])
        gs = oracle.shared_gate(args["shared_gate_bf16"], x[r])
        ref = one + gs * ex("shared").ffn_row(x[r])
        assert tol_ok(y[r], ref, 1e-6)
        assert sorted(idx[r]) == list(range(6))


def test_moe_zero_expert_contributes_nothing():
    args = make_layer(51, TINY)
    x = rand_bf16(52, (1, TINY.hidden))
    y, idx, w = oracle.moe_layer(x, **args)
    victim = int(idx[0, 0])
    args0 = make_layer(51, TINY, zero_expert=victim)
    y0, idx0, w0 = oracle.moe_layer(x, **args0)
    assert np.array_equal(idx, idx0) and np.array_equal(w, w0)
    ex = args["experts"]
    assert tol_ok(y0[0], y[0].astype(np.float64) - w[0, 0] * ex(victim).ffn_row(x[0]), 1e-5)


def test_moe_zero_gate_halves_shared_expert():
    args = make_layer(61, TINY, zero_gate=True)
    x = rand_bf16(62, (1, TINY.hidden))
    assert oracle.shared_gate(args["shared_gate_bf16"], x[0]) == 0.5
    y, idx, w = oracle.moe_layer(x, **args)
    ex = args["experts"]
    routed = sum(w[0, s] * ex(int(idx[0, s])).ffn_row(x[0]) for s in range(TINY.top_k))
    assert tol_ok(y[0], routed + 0.5 * ex("shared").ffn_row(x[0]), 1e-6)


def test_moe_rows_are_independent():
    args = make_layer(71, TINY)
    x = rand_bf16(72, (4, TINY.hidden))
    y, idx, w = oracle.moe_layer(x, **args)
    for r in range(4):
        y1, idx1, w1 = oracle.moe_layer(x[r:r + 1], **args)
        assert np.array_equal(y1[0], y[r]) and np.array_equal(idx1[0], idx[r])


def test_rmsnorm_and_residual():
    h = rand_bf16(81, (3, 256), 3.0)
    t = oracle.rmsnorm_bf16(h)
    hf = f32_of(h)
    inv = (np.float32(1.0) / np.sqrt((np.sum(hf.astype(np.float64) ** 2, axis=1) / 256).astype(np.float32)
                                     + np.float32(1e-6))).astype(np.float32)
    assert np.array_equal(t, bf16((hf * inv[:, None]).astype(np.float32)))
    y = np.random.default_rng(82).standard_normal((3, 256)).astype(np.float32)
    assert np.array_equal(oracle.residual_bf16(h, y), bf16((hf + y).astype(np.float32)))


def test_rmsnorm_and_residual_closed_forms():
    """Values fixed by hand, independent of the formula's code: a constant row normalises to 1; a
    one-hot row of width 16 gives sqrt(16) = 4 (the mean divides by the width, not width - 1, which
    would give 3.875); a row of 2^-12 shows eps inside the square root (2^-12 / sqrt(2^-24 + 1e-6)
    = 0.23717 -> bf16 0.237305; eps outside would give 0.99609, no eps 1.0); the residual rounds
    h + y to nearest bf16 with ties to even."""
    h = bf16(np.full((1, 256), 3.0, np.float32))
    assert np.all(f32_of(oracle.rmsnorm_bf16(h)) == 1.0)
    h = bf16(np.eye(1, 16, dtype=np.float32))
    t = f32_of(oracle.rmsnorm_bf16(h))
    assert t[0, 0] == 4.0 and np.all(t[0, 1:] == 0.0)
    h = bf16(np.full((1, 64), 2.0 ** -12, np.float32))
    assert np.all(f32_of(oracle.rmsnorm_bf16(h)) == np.float32(0.2373046875))
    one = bf16(np.array([[1.0, 1.0078125, 1.0, -1.0]], np.float32))
    y = np.array([[2.0 ** -8, 2.0 ** -8, 2.0 ** -8 + 2.0 ** -20, 0.5]], np.float32)
    assert list(f32_of(oracle.residual_bf16(one, y))[0]) == [1.0, 1.015625, 1.0078125, -0.5]


def test_greedy_tokens_brute_force_and_special_cases():
    # Brute force: the first index whose value no other non-NaN value exceeds.
    rng = np.random.default_rng(91)
    for trial in range(300):
        n = int(rng.integers(1, 70))
        l = rng.standard_normal(n).astype(np.float32)
        if trial % 3 == 0:  # ties
            l = np.round(l)
        if trial % 5 == 0:  # NaNs sprinkled in
            l[rng.random(n) < 0.3] = np.nan
        vals = [float(v) for v in l]
        ok = [i for i in range(n) if vals[i] == vals[i]]
        want = 0 if not ok else min(i for i in ok if all(vals[i] >= vals[j] for j in ok))
        assert oracle.greedy_tokens(l)[0] == want
    # Closed cases: a one-hot row, equal values, signed zeros, infinities, NaN alone.
    one_hot = np.full(1000, -1.0, np.float32)
    one_hot[637] = 2.0
    assert oracle.greedy_tokens(one_hot)[0] == 637
    assert oracle.greedy_tokens(np.full(9, 3.5, np.float32))[0] == 0
    assert oracle.greedy_tokens(np.array([-0.0, 0.0, -1.0], np.float32))[0] == 0
    assert oracle.greedy_tokens(np.array([-1.0, -0.0, 0.0], np.float32))[0] == 1
    assert oracle.greedy_tokens(np.array([np.nan, -np.inf, 1e30, np.inf, np.inf], np.float32))[0] == 3
    assert oracle.greedy_tokens(np.array([np.nan, np.nan], np.float32))[0] == 0
    assert oracle.greedy_tokens(np.array([np.nan, -np.inf], np.float32))[0] == 1
    # Rows are independent; the last index can win.
    m = np.zeros((3, 5), np.float32)
    m[0, 4], m[1, 2], m[2, 0] = 1, 1, 1
    assert list(oracle.greedy_tokens(m)) == [4, 2, 0]
