"""ORACLE — test infrastructure only.

Plain CPU reference for the BFP MoE decode path. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
the library (``block_floating_point_gb300``) never does, and the two share no
code. The arithmetic of the decode step lives in ``bfp_oracle.c`` (plain C,
fp64); this module loads it with ctypes and strings its pieces together in the
order the decode step defines: router -> softmax -> top-k -> renormalise ->
experts -> combine. The error-compensated encoding and the KV-cache attention
are plain NumPy further down (fp64, except where the method fixes fp32).

Every function cites the passage of the block_floating_point pages it follows
(page titles abbreviated as in ``bfp_oracle.c``). Readings of points the pages
leave open are stated in ``bfp_oracle.c``'s header.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(brute-force rational rounding, closed-form sizes, fp64 NumPy matmul,
brute-force sorting, special-case MoE identities; for the greedy token brute
force; for error-compensated encoding the diagonal-Hessian, optimal-brain-
quantiser, fixed-point and output-error cases; for the KV cache the Hadamard
matrix, closed forms of attention and a direct softmax).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

BFP4, BFP8 = 4, 8
RMS_EPS = 1e-6

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``bfp_oracle.c`` with gcc into ``_build/liboracle.so`` (no -ffast-math: IEEE fp64 as written)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    src = os.path.join(_HERE, "bfp_oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", src, "-o", tmp,
                               "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            sig = {
                "oracle_encode": [_I, _P, _I64, _I64, _P, _P],
                "oracle_decode": [_I, _P, _P, _I64, _I64, _P],
                "oracle_linear": [_I, _P, _P, _I64, _I64, _P, _I, _P, _P],
                "oracle_router_logits": [_P, _I, _I, _P, _I, _P, _P],
                "oracle_route_row": [_P, _I, _I, _P, _P],
                "oracle_expert_ffn": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P],
                "oracle_rmsnorm_bf16": [_P, _I, _I, ctypes.c_float, _P],
                "oracle_residual_bf16": [_P, _P, _I64],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.oracle_greedy_row.argtypes = [_P, _I64]
            lib.oracle_greedy_row.restype = ctypes.c_int64
            lib.oracle_shared_gate.argtypes = [_P, _P, _I]
            lib.oracle_shared_gate.restype = ctypes.c_double
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------------------------------------------------------------------
# Format: encode / decode / storage size
# ---------------------------------------------------------------------------
def mant_bits(fmt: int) -> int:
    """Magnitude bits of a code: 3 for BFP4, 7 for BFP8 (sign-magnitude, one sign bit)."""
    return {BFP4: 3, BFP8: 7}[fmt]


def storage_bytes_per_value(fmt: int) -> float:
    """Bytes per value: code bits/8 plus one exponent byte per 16 values.

    BFP8: 1 + 1/16 = 1.0625 (the pages' BFP8 KV cache: 20.0 KiB -> 10.6 KiB per
    token, qwen3.6-a3b-blackhole page, QWEN36_KV_DTYPE row). BFP4: 0.5 + 1/16 =
    0.5625 (Qwen3.8-27B card, "Changes in s27": K BFP8 + V BFP4 = 26,624 B per
    token vs 34,816 B in BFP8 + BFP8).
    """
    return (mant_bits(fmt) + 1) / 8.0 + 1.0 / 16.0


def encode(fmt: int, w: np.ndarray):
    """fp32 [n, k] -> (exps u8 [n, k/16], codes u8 [n, k]); round to nearest (ties to even) in 16-value blocks.

    Blocks of 16 along k: Qwen3.8-27B gptq-ctx2 card, "What changed in this
    release"; round-to-nearest: Qwen3.6-35B-A3B card, "Verification" (RTN parent).
    """
    w, wp = _c(w, np.float32)
    n, k = w.shape
    exps = np.zeros((n, k // 16), dtype=np.uint8)
    codes = np.zeros((n, k), dtype=np.uint8)
    rc = _load().oracle_encode(fmt, wp, n, k, exps.ctypes.data, codes.ctypes.data)
    if rc == -4:
        raise ValueError("non-finite input")
    if rc != 0:
        raise ValueError(f"oracle_encode failed ({rc})")
    return exps, codes


def decode(fmt: int, exps: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """(exps, codes) -> fp32 [n, k]: value = (-1)^s * m * 2^(E - 127 - (mb - 1))."""
    exps, ep = _c(exps, np.uint8)
    codes, cp = _c(codes, np.uint8)
    n, k = codes.shape
    out = np.zeros((n, k), dtype=np.float32)
    rc = _load().oracle_decode(fmt, ep, cp, n, k, out.ctypes.data)
    assert rc == 0
    return out


# ---------------------------------------------------------------------------
# Dense BFP projection (dense projections and the LM head are BFP8:
# Qwen3.6-35B-A3B card, "Precision as served").
# ---------------------------------------------------------------------------
def linear(fmt: int, exps, codes, x_bf16: np.ndarray):
    """y = x W^T with bf16 x [m, k]; returns (y fp32 [m, n], y bf16 bits [m, n])."""
    exps, ep = _c(exps, np.uint8)
    codes, cp = _c(codes, np.uint8)
    x, xp = _c(x_bf16, np.uint16)
    n, k = codes.shape
    m = x.shape[0]
    assert x.shape[1] == k
    y = np.zeros((m, n), dtype=np.float32)
    yb = np.zeros((m, n), dtype=np.uint16)
    rc = _load().oracle_linear(fmt, ep, cp, n, k, xp, m, y.ctypes.data, yb.ctypes.data)
    assert rc == 0
    return y, yb


# ---------------------------------------------------------------------------
# MoE decode layer: device top-k routing + batched expert streams
# (Qwen3.6-35B-A3B card, "Fused decode kernels"; 256 experts, top-8 plus a
# shared expert: qwen3.6-a3b-blackhole page, opening paragraph).
# ---------------------------------------------------------------------------
def router_logits(router_bf16, x_bf16, bias=None) -> np.ndarray:
    r, rp = _c(router_bf16, np.uint16)
    x, xp = _c(x_bf16, np.uint16)
    e, h = r.shape
    m = x.shape[0]
    out = np.zeros((m, e), dtype=np.float32)
    bp = None
    if bias is not None:
        b, bp = _c(bias, np.float32)
    rc = _load().oracle_router_logits(rp, e, h, xp, m, bp, out.ctypes.data)
    assert rc == 0
    return out


def route_row(logits_row, k: int):
    """Softmax (fp64 from fp32 logits) -> top-k on fp32 logits (ties: lower index) -> renormalise."""
    l, lp = _c(logits_row, np.float32)
    idx = np.zeros(k, dtype=np.int32)
    w = np.zeros(k, dtype=np.float64)
    rc = _load().oracle_route_row(lp, l.shape[0], k, idx.ctypes.data, w.ctypes.data)
    assert rc == 0
    return idx, w


def topk_margin(logits_row, k: int) -> float:
    """Gap between the k-th and (k+1)-th largest fp32 logit (inf when k == number of experts)."""
    s = np.sort(np.asarray(logits_row, dtype=np.float64))[::-1]
    return float(s[k - 1] - s[k]) if k < s.shape[0] else float("inf")


def shared_gate(g_bf16, x_row_bf16) -> float:
    g, gp = _c(g_bf16, np.uint16)
    x, xp = _c(x_row_bf16, np.uint16)
    return float(_load().oracle_shared_gate(gp, xp, g.shape[0]))


class EncodedExpert:
    """An expert's three matrices as the oracle's own logical encoding."""

    def __init__(self, fmt, gate_f32, up_f32, down_f32):
        self.fmt = fmt
        self.ffn, self.hidden = gate_f32.shape
        self.g = encode(fmt, gate_f32)
        self.u = encode(fmt, up_f32)
        self.d = encode(fmt, down_f32)

    def ffn_row(self, x_row_bf16) -> np.ndarray:
        """o = D (silu(G x) * (U x)) in fp64."""
        x, xp = _c(x_row_bf16, np.uint16)
        o = np.zeros(self.hidden, dtype=np.float64)
        ge, gc = self.g
        ue, uc = self.u
        de, dc = self.d
        rc = _load().oracle_expert_ffn(self.fmt, self.hidden, self.ffn, ge.ctypes.data, gc.ctypes.data,
                                       ue.ctypes.data, uc.ctypes.data, de.ctypes.data, dc.ctypes.data, xp,
                                       o.ctypes.data)
        assert rc == 0
        return o


class ExpertCache:
    """Encodes experts on first use; ``source(e)`` returns fp32 (gate, up, down) of expert e (e = 'shared' too)."""

    def __init__(self, fmt, source):
        self.fmt, self.source, self._c = fmt, source, {}

    def __call__(self, e) -> EncodedExpert:
        if e not in self._c:
            g, u, d = self.source(e)
            self._c[e] = EncodedExpert(self.fmt, g, u, d)
        return self._c[e]


def moe_layer(x_bf16, router_bf16, shared_gate_bf16, experts: ExpertCache, top_k: int, router_bias=None,
              shared_key="shared"):
    """One MoE decode layer on M bf16 rows.

    Per row r:  l = Wr x (fp32),  p = softmax(l),  S = top-k(l),
    w_s = p_s / sum_S p,  y = sum_s w_s * D_s(silu(G_s x) * U_s x) + sigmoid(g . x) * shared(x).
    Returns (y fp32 [M, H], idx int32 [M, k], w fp64 [M, k]).
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    m, hidden = x.shape
    logits = router_logits(router_bf16, x, router_bias)
    y = np.zeros((m, hidden), dtype=np.float32)
    idx_all = np.zeros((m, top_k), dtype=np.int32)
    w_all = np.zeros((m, top_k), dtype=np.float64)
    for r in range(m):
        idx, w = route_row(logits[r], top_k)
        acc = np.zeros(hidden, dtype=np.float64)
        for s in range(top_k):
            acc += w[s] * experts(int(idx[s])).ffn_row(x[r])
        acc += shared_gate(shared_gate_bf16, x[r]) * experts(shared_key).ffn_row(x[r])
        y[r] = acc.astype(np.float32)
        idx_all[r], w_all[r] = idx, w
    return y, idx_all, w_all


def rmsnorm_bf16(h_bf16, eps: float = RMS_EPS) -> np.ndarray:
    """bf16(h / sqrt(mean(h^2) + eps)), unit weight (the one-launch decode RMSNorm of the
    Qwen3.6-35B-A3B card, "Fused decode kernels", as a plain function)."""
    h, hp = _c(h_bf16, np.uint16)
    m, hidden = h.shape
    out = np.zeros_like(h)
    rc = _load().oracle_rmsnorm_bf16(hp, m, hidden, np.float32(eps), out.ctypes.data)
    assert rc == 0
    return out


def residual_bf16(h_bf16, y_f32) -> np.ndarray:
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16).copy()
    y, yp = _c(y_f32, np.float32)
    rc = _load().oracle_residual_bf16(h.ctypes.data, yp, h.size)
    assert rc == 0
    return h


def stack_layer(h_bf16, layer_args: dict):
    """h <- bf16(h + MoE(bf16(RMSNorm(h)))). Returns (new h, MoE input t, y, idx, w)."""
    t = rmsnorm_bf16(h_bf16)
    y, idx, w = moe_layer(t, **layer_args)
    return residual_bf16(h_bf16, y), t, y, idx, w


def lm_head_rows(h_bf16, lm_rows_f32: np.ndarray, fmt: int = BFP8):
    """Logits of a subset of vocabulary rows: fp32( W_rows . bf16(RMSNorm(h)) ), W encoded by the oracle."""
    t = rmsnorm_bf16(h_bf16)
    e, c = encode(fmt, lm_rows_f32)
    y, _ = linear(fmt, e, c, t)
    return y


def greedy_tokens(logits_f32) -> np.ndarray:
    """Greedy next token per row of fp32 logits [M, V]: index of the largest value, ties to the lower
    index, NaN never chosen (a NaN-only row gives 0). The step after the LM head in greedy decoding
    (Qwen3.6-35B-A3B card, "Fused decode kernels")."""
    lg = np.ascontiguousarray(logits_f32, dtype=np.float32)
    if lg.ndim == 1:
        lg = lg[None, :]
    lib = _load()
    out = np.zeros(lg.shape[0], dtype=np.int32)
    for r in range(lg.shape[0]):
        out[r] = lib.oracle_greedy_row(lg[r].ctypes.data, lg.shape[1])
    return out


# ---------------------------------------------------------------------------
# Error-compensated (GPTQ-style) BFP encoding. The Qwen3.8-27B gptq-ctx2 card,
# "What changed in this release": BFP4 weights computed by a GPTQ variant for
# block floating point, with error compensation inside the 16-value blocks,
# every value exactly representable so that the plain conversion reproduces it.
# GPTQ itself is the published method of Frantar et al., "GPTQ: Accurate
# Post-Training Quantization for Generative Pre-trained Transformers" (2022):
# columns are quantised one at a time and each rounding error is moved onto the
# columns not yet quantised through the inverse of the layer's Hessian
# H = X^T X of its calibration inputs X.
# Readings (the pages give no more): H = X^T X / t plus damp * mean(diag) on the
# diagonal; columns in their natural order; a block's exponent is taken from its
# current (already compensated) values when its first column comes up; after its
# 16 columns the block is brought to canonical form (exponent lowered while every
# magnitude fits one bit less), which is what plain round-to-nearest would give
# for the same values.
# ---------------------------------------------------------------------------
def gptq_hessian(x_f32, damp: float = 0.01) -> np.ndarray:
    """H = X^T X / t + damp * mean(diag(X^T X / t)) * I in fp64; x is [t, k] (t calibration inputs)."""
    x = np.asarray(x_f32, dtype=np.float64)
    h = x.T @ x / x.shape[0]
    h[np.diag_indices_from(h)] += damp * float(np.mean(np.diag(h)))
    return h


def gptq_factor(x_f32, damp: float = 0.01) -> np.ndarray:
    """Upper-triangular U with H^-1 = U^T U (GPTQ's Cholesky form of the inverse Hessian)."""
    hinv = np.linalg.inv(gptq_hessian(x_f32, damp))
    return np.linalg.cholesky(hinv).T


def _exp_field(v: np.ndarray) -> np.ndarray:
    """fp32-style biased exponent of fp64 values: floor(log2|v|) + 127, 0 below 2^-126 (and for 0)."""
    _, p = np.frexp(np.abs(v))
    e = p.astype(np.int64) + 126
    return np.where(np.abs(v) < 2.0 ** -126, 0, e)


def gptq_quantise_column(v: np.ndarray, E: np.ndarray, mb: int):
    """Magnitude codes and values of one column on the blocks' grids (ties to even, saturating)."""
    s = E - 127 - (mb - 1)
    mag = np.rint(np.ldexp(np.abs(v), -s))
    mag = np.minimum(mag, 2 ** mb - 1)
    mag = np.where((E == 0) | (_exp_field(v) == 0), 0, mag).astype(np.int64)
    q = np.where(mag > 0, np.sign(v) * np.ldexp(mag.astype(np.float64), s), 0.0)
    return mag, q


def gptq_encode(fmt: int, w_f32, u: np.ndarray):
    """Error-compensated encoding of w [n, k] with the factor u [k, k]: returns (exps [n, k/16] u8,
    codes [n, k] u8) in the same logical form as ``encode``. Rows are independent; within a row the
    columns go left to right and column j's error (v - q) / u[j, j] is taken off the later columns
    in proportion to u[j, j+1:]."""
    mb = mant_bits(fmt)
    w = np.array(w_f32, dtype=np.float64)
    n, k = w.shape
    if k % 16 or u.shape != (k, k):
        raise ValueError("k must be a multiple of 16 and u [k, k]")
    exps = np.zeros((n, k // 16), dtype=np.uint8)
    mags = np.zeros((n, k), dtype=np.int64)
    neg = np.zeros((n, k), dtype=bool)
    for b in range(k // 16):
        j0 = 16 * b
        E = _exp_field(w[:, j0:j0 + 16]).max(axis=1)
        if np.any(E >= 255):
            raise ValueError("compensated values left the fp32 range")
        for j in range(j0, j0 + 16):
            mag, q = gptq_quantise_column(w[:, j], E, mb)
            mags[:, j], neg[:, j] = mag, (mag > 0) & (w[:, j] < 0)
            err = (w[:, j] - q) / u[j, j]
            if j + 1 < k:
                w[:, j + 1:] -= np.outer(err, u[j, j + 1:])
        # canonical form: lower the exponent while every magnitude of the block fits mb - 1 bits
        blk = mags[:, j0:j0 + 16]
        for r in range(n):
            if blk[r].max() == 0:
                E[r] = 0
                continue
            while E[r] > 1 and blk[r].max() < 2 ** (mb - 1):
                E[r] -= 1
                blk[r] *= 2
        exps[:, b] = E.astype(np.uint8)
    codes = (neg.astype(np.int64) << mb) | mags
    return exps, codes.astype(np.uint8)


# ---------------------------------------------------------------------------
# BFP KV cache and decode attention. The qwen3.6-a3b-blackhole page
# (QWEN36_KV_DTYPE row): the attention KV cache stored as BFP8, 20.0 -> 10.6
# KiB per token, decode attention re-reading the whole cache each step. The
# Qwen3.8-27B s27v6 card ("Changes in s27", bfp8_v4r): K in BFP8 and V
# Hadamard-rotated, then stored as BFP4 (26,624 instead of 34,816 bytes per
# token).
# Readings: the rotation is the Sylvester-ordered Hadamard matrix H_d (entries
# +-1, d a power of two), applied to each head's V vector before encoding; it
# is computed in fp32 by the fast transform, stage h = 1, 2, 4, ... pairing
# (i, i + h) into (a + b, a - b), which is the precision and order in which the
# encoder decides the codes. Attention undoes it on the weighted sum of the
# decoded rows: out = H_d (sum_t p_t v'_t) / d (H_d H_d = d I).
# Attention per query head: s_t = scale * q . k_t, p = softmax(s), out =
# sum_t p_t v_t, with query head j reading KV head j // (q_heads / kv_heads).
# ---------------------------------------------------------------------------
def fwht_f32(x) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform over the last axis, in fp32, stage by stage."""
    y = np.array(x, dtype=np.float32)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("length must be a power of two")
    h = 1
    while h < d:
        v = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a, b = v[..., 0, :].copy(), v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        h *= 2
    return y


def kv_encode(fmt: int, rows_bf16, rotate: bool):
    """Cache fields of bf16 rows [..., d]: (exps [..., d/16], codes [..., d]) of the rows (Hadamard-
    rotated in fp32 first when ``rotate``), by the plain round-to-nearest encoder."""
    r = np.asarray(rows_bf16, dtype=np.uint16)
    shape = r.shape
    f = (r.astype(np.uint32) << 16).view(np.float32).reshape(-1, shape[-1])
    if rotate:
        f = fwht_f32(f)
    e, c = encode(fmt, f)
    return e.reshape(shape[:-1] + (shape[-1] // 16,)), c.reshape(shape)


def kv_decode(fmt: int, exps, codes, rotated: bool) -> np.ndarray:
    """Decoded cache rows in fp64 (rotated back when stored rotated)."""
    e = np.asarray(exps)
    c = np.asarray(codes)
    d = c.shape[-1]
    v = decode(fmt, e.reshape(-1, d // 16), c.reshape(-1, d)).astype(np.float64)
    if rotated:
        v = _hadamard_f64(v) / d
    return v.reshape(c.shape)


def _hadamard_f64(v: np.ndarray) -> np.ndarray:
    d = v.shape[-1]
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return v @ h  # H is symmetric


def attn_decode(q_bf16, k_fields, v_fields, n_ctx: int, scale: float, k_fmt: int, v_fmt: int,
                v_rotated: bool) -> np.ndarray:
    """Decode attention of one query token over n_ctx cached tokens, fp64.

    q_bf16 [q_heads, d]; k_fields / v_fields = (exps [kv_heads, n, d/16], codes [kv_heads, n, d]).
    Returns out [q_heads, d]: softmax(scale * q K^T) V per query head (V rotated back if stored rotated).
    """
    q = (np.asarray(q_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qh, d = q.shape
    ke, kc = (np.asarray(a)[:, :n_ctx] for a in k_fields)
    ve, vc = (np.asarray(a)[:, :n_ctx] for a in v_fields)
    kvh = kc.shape[0]
    if qh % kvh:
        raise ValueError("q_heads must be a multiple of kv_heads")
    g = qh // kvh
    kd = kv_decode(k_fmt, ke, kc, False)
    vd = decode(v_fmt, ve.reshape(-1, d // 16), vc.reshape(-1, d)).astype(np.float64).reshape(kvh, n_ctx, d)
    out = np.zeros((qh, d))
    for j in range(qh):
        h = j // g
        s = scale * (kd[h] @ q[j])
        p = np.exp(s - s.max())
        p /= p.sum()
        o = p @ vd[h]
        out[j] = _hadamard_f64(o[None, :])[0] / d if v_rotated else o
    return out
