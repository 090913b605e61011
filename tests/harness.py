"""Test harness: seeded inputs for both sides, the oracle's answers, and the
element-wise tolerance.

Inputs come from ``synth`` only; the oracle encodes its own copy of every
weight from the same fp32 values, so no oracle input comes from the CUDA path.

Tolerance (stated for the decode step's fp32 outputs):
    |gpu - oracle| <= 1e-3 * (|oracle| + rms(oracle))   per element, rms per row.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL = 1e-3
MARGIN = 1e-3  # rows whose k-th / (k+1)-th router-logit gap is below this are redrawn


def within_tol(got, ref, tol=TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    bound = tol * (np.abs(ref) + rms)
    err = np.abs(got - ref)
    ok = np.all(err <= bound)
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if ref.size else 0.0
    return bool(ok), worst


def assert_close(got, ref, what="", tol=TOL):
    ok, worst = within_tol(got, ref, tol)
    assert ok, f"{what}: max |err| / bound = {worst:.3f} (> 1)"


class LayerCase:
    """One synthetic MoE decode layer: fp32 sources (synth), oracle encodings, inputs."""

    def __init__(self, spec: synth.MoESpec, seed: int, layer: int = 0, instance: int = 0, hot: bool = False,
                 fmt: int = 4):
        self.spec, self.seed, self.fmt = spec, seed, fmt
        self.w = synth.LayerWeights(spec, seed, layer, instance)
        self.router = self.w.router_bf16()
        self.sgate = self.w.shared_gate_bf16()
        self.bias = synth.hot_bias(spec.n_experts, seed) if hot else None

        def source(e):
            key = synth.SHARED_EXPERT if e == "shared" else e
            return self.w.gate(key), self.w.up(key), self.w.down(key)

        self.source = source
        self.experts = oracle.ExpertCache(fmt, source)

    def inputs(self, m: int, rms_normalise: bool, row_seed0: int = 0):
        """m bf16 rows; a row is redrawn (next row seed) while its top-k margin is below MARGIN."""
        rows, seeds = [], []
        rs = row_seed0
        for _ in range(m):
            while True:
                x = synth.activation_row(self.seed, rs, self.spec.hidden, rms_normalise)
                l = oracle.router_logits(self.router, x[None, :], self.bias)[0]
                rs += 1
                if oracle.topk_margin(l, self.spec.top_k) >= MARGIN:
                    break
            rows.append(x)
            seeds.append(rs - 1)
        return np.stack(rows), seeds

    def oracle_layer(self, x):
        return oracle.moe_layer(x, self.router, self.sgate, self.experts, self.spec.top_k, self.bias)

    def device_layer(self, device="cuda"):
        import block_floating_point_gb300 as bfp
        s = self.spec
        return bfp.MoELayer.from_source(s.hidden, s.n_experts, s.ffn, s.top_k, s.shared_ffn, self.fmt, self.router,
                                        self.sgate, lambda e: self.source(e), lambda: self.source("shared"),
                                        router_bias=self.bias, device=device)


def bf16_tensor(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(device)


# ---------------------------------------------------------------- KV-cache tile layout (include/bfpmoe.h)
def _p(code):
    return (int(code) & 0x7F) | ((int(code) >> 7) << 15)


def tile_bytes(codes16, which, fmt):
    """One 16-token x 16-column tile of codes in the cache layout (the layout text of include/bfpmoe.h)."""
    t = np.zeros(256 if fmt == 8 else 128, np.uint8)
    for r in range(16):
        for c in range(16):
            code = int(codes16[r, c])
            if which == "k" and fmt == 8 and c % 4 == 0:
                cs = codes16[r, c:c + 4]
                p01, p23 = _p(cs[0]) | (_p(cs[1]) << 16), _p(cs[2]) | (_p(cs[3]) << 16)
                w = p01 | (((p23 << 8) | (p23 >> 24)) & 0xFFFFFFFF)
                off = (4 * (r % 8) + c // 4) * 8 + (r // 8) * 4
                t[off:off + 4] = np.frombuffer(np.uint32(w).tobytes(), np.uint8)
            elif which == "k" and fmt == 4:
                off = (4 * (r % 8) + c // 4) * 4 + (r // 8) * 2 + (c % 4) // 2
                t[off] |= code << (4 * (c % 2))
            elif which == "v" and fmt == 8:
                t[(4 * (c % 8) + r // 4) * 8 + (c // 8) * 4 + r % 4] = code
            elif which == "v" and fmt == 4:
                t[(4 * (c % 8) + r // 4) * 4 + r % 4] |= code << (4 * (c // 8))
    return t


def expected_codes(codes, which, fmt, cap):
    """Cache code bytes [kvh, cap / 16, NB, TB] of oracle codes [kvh, n, d] (slots past n left as zero)."""
    kvh, n, d = codes.shape
    nb, tb = d // 16, (256 if fmt == 8 else 128)
    out = np.zeros((kvh, cap // 16, nb, tb), np.uint8)
    full = np.zeros((kvh, cap, d), np.uint8)
    full[:, :n] = codes
    for h in range(kvh):
        for g in range((n + 15) // 16):
            for b in range(nb):
                out[h, g, b] = tile_bytes(full[h, 16 * g:16 * g + 16, 16 * b:16 * b + 16], which, fmt)
    return out
