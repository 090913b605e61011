"""Seeded synthetic inputs, shared by the oracle side and the CUDA side.

This package draws numbers and nothing else: it contains none of the block
floating point arithmetic (no exponents, rounding to codes or packing). The
generator is Philox4x32-10 (Salmon et al., SC'11) with Box-Muller normals,
written in ``gen.c``; every value is a pure function of (seed, stream, index),
so any matrix of any layer can be regenerated on its own.

Workload recipes follow the decode-layer configurations the benchmark and the
tests use (weights N(0, 0.02) in fp32 before encoding, bf16 activations
N(0, 1), optionally RMS-normalised per row, bf16 router and shared gate
N(0, 0.02)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_build/libsynth.so`` with gcc (host code, any arch)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                             ctypes.c_double, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.synth_normal_f32.restype = ctypes.c_int
            lib.synth_bits_u32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_int]
            lib.synth_bits_u32.restype = ctypes.c_int
            lib.synth_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_philox4x32_10.restype = None
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox4x32-10 block (for known-answer checks)."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def normal(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0, offset: int = 0,
           threads: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """fp32 array of N(mean, std) deviates drawn from (seed, stream), starting at value ``offset``."""
    n = int(np.prod(shape)) if not isinstance(shape, int) else int(shape)
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    rc = _load().synth_normal_f32(seed & (2**64 - 1), stream & (2**64 - 1), offset, n, float(mean), float(std),
                                  out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise RuntimeError("synth_normal_f32 failed")
    return out


def bits(seed: int, stream: int, n: int, offset: int = 0, threads: int | None = None) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    rc = _load().synth_bits_u32(seed & (2**64 - 1), stream & (2**64 - 1), offset, n, out.ctypes.data,
                                threads or default_threads())
    if rc != 0:
        raise RuntimeError("synth_bits_u32 failed")
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the 16-bit patterns.

    Input preparation only: activations and router weights are bf16 inputs of
    the decode step, so the generator hands out bf16 bit patterns.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Stream ids: one independent stream per (instance, layer, expert, matrix).
# ---------------------------------------------------------------------------
KIND_GATE, KIND_UP, KIND_DOWN = 1, 2, 3
KIND_ROUTER, KIND_SHGATE, KIND_X, KIND_DENSE, KIND_LMHEAD, KIND_STACK_H = 4, 5, 6, 7, 8, 9
SHARED_EXPERT = 0xFFFF


def stream_id(kind: int, layer: int = 0, expert: int = 0, instance: int = 0, row: int = 0) -> int:
    return ((instance & 0xFF) << 56) | ((kind & 0xFF) << 48) | ((layer & 0xFFF) << 36) | \
           ((expert & 0xFFFF) << 20) | (row & 0xFFFFF)


class MoESpec:
    """Shapes of one synthetic MoE decode layer."""

    def __init__(self, hidden: int, n_experts: int, ffn: int, top_k: int, shared_ffn: int):
        self.hidden, self.n_experts, self.ffn, self.top_k, self.shared_ffn = hidden, n_experts, ffn, top_k, shared_ffn

    def __repr__(self):
        return (f"MoESpec(hidden={self.hidden}, n_experts={self.n_experts}, ffn={self.ffn}, "
                f"top_k={self.top_k}, shared_ffn={self.shared_ffn})")


TINY = MoESpec(256, 16, 128, 2, 128)          # tiny decode layer: H=256, 16 experts, F=128, top-2, shared 128
FULL = MoESpec(2048, 256, 512, 8, 512)        # full-size decode layer: H=2048, 256 experts, F=512, top-8, shared 512

W_STD = 0.02


class LayerWeights:
    """fp32 source weights of one synthetic layer, generated lazily per expert."""

    def __init__(self, spec: MoESpec, seed: int, layer: int = 0, instance: int = 0):
        self.spec, self.seed, self.layer, self.instance = spec, seed, layer, instance

    def _mat(self, kind, expert, rows, cols):
        return normal(self.seed, stream_id(kind, self.layer, expert, self.instance), (rows, cols), std=W_STD)

    def gate(self, e):
        f = self.spec.shared_ffn if e == SHARED_EXPERT else self.spec.ffn
        return self._mat(KIND_GATE, e, f, self.spec.hidden)

    def up(self, e):
        f = self.spec.shared_ffn if e == SHARED_EXPERT else self.spec.ffn
        return self._mat(KIND_UP, e, f, self.spec.hidden)

    def down(self, e):
        f = self.spec.shared_ffn if e == SHARED_EXPERT else self.spec.ffn
        return self._mat(KIND_DOWN, e, self.spec.hidden, f)

    def router_bf16(self):
        r = normal(self.seed, stream_id(KIND_ROUTER, self.layer, 0, self.instance),
                   (self.spec.n_experts, self.spec.hidden), std=W_STD)
        return to_bf16_bits(r)

    def shared_gate_bf16(self):
        g = normal(self.seed, stream_id(KIND_SHGATE, self.layer, 0, self.instance), (self.spec.hidden,), std=W_STD)
        return to_bf16_bits(g)


def activation_row(seed: int, row_seed: int, hidden: int, rms_normalise: bool, instance: int = 0) -> np.ndarray:
    """One bf16 activation row: N(0,1) fp32, optionally scaled to RMS 1 in fp32, then rounded to bf16."""
    x = normal(seed, stream_id(KIND_X, 0, 0, instance, row_seed), (hidden,), std=1.0)
    if rms_normalise:
        rms = np.float32(np.sqrt(np.mean(x.astype(np.float32) ** 2, dtype=np.float32)))
        x = (x / rms).astype(np.float32)
    return to_bf16_bits(x)


def hot_bias(n_experts: int, seed: int, n_hot: int = 8, value: float = 2.0) -> np.ndarray:
    """Router-logit bias of +value on n_hot experts picked by a seeded draw (the highly overlapped routing case)."""
    w = bits(seed, stream_id(KIND_ROUTER, 0xFFF, 0xFFFF), n_experts)
    hot = np.argsort(w, kind="stable")[:n_hot]
    b = np.zeros(n_experts, dtype=np.float32)
    b[hot] = value
    return b
