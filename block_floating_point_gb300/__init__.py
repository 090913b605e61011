"""Python binding of the GB300 BFP MoE decode library (``include/bfpmoe.h``).

Argument marshalling only: every step of the decode path runs in the native
library ``_build/libbfpmoe.so`` (CUDA for sm_103a plus the host packer). There
is no Python or CPU fallback; if the library is missing or cannot be loaded,
every call raises.

PyTorch supplies device memory and streams: device arguments are CUDA torch
tensors (their ``data_ptr()`` is passed), the stream is the current torch
stream unless one is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

BFP_OK, BFP_EINVAL, BFP_ESHAPE, BFP_EALIGN, BFP_ENONFINITE, BFP_EWORKSPACE, BFP_ECUDA, BFP_ETIMEOUT = \
    0, -1, -2, -3, -4, -5, -6, -7
BFP4, BFP8 = 4, 8
STATUS_NAMES = {0: "BFP_OK", -1: "BFP_EINVAL", -2: "BFP_ESHAPE", -3: "BFP_EALIGN", -4: "BFP_ENONFINITE",
                -5: "BFP_EWORKSPACE", -6: "BFP_ECUDA", -7: "BFP_ETIMEOUT"}


class BFPError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class BfpMatrixC(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64), ("data", ctypes.c_void_p), ("bytes", ctypes.c_int64)]


class MoeLayerC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("shared_ffn", ctypes.c_int32), ("expert_fmt", ctypes.c_int32),
                ("router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("shared_gate", ctypes.c_void_p),
                ("experts_gate_up", ctypes.c_void_p), ("experts_down", ctypes.c_void_p),
                ("gate_up_stride", ctypes.c_int64), ("down_stride", ctypes.c_int64),
                ("shared_gate_up", ctypes.c_void_p), ("shared_down", ctypes.c_void_p)]


class KvCacheC(ctypes.Structure):
    _fields_ = [("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("k_fmt", ctypes.c_int32),
                ("v_fmt", ctypes.c_int32), ("v_rotated", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("capacity", ctypes.c_int64), ("k_codes", ctypes.c_void_p), ("k_exps", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_exps", ctypes.c_void_p)]


# Every entry point declared in include/bfpmoe.h, with its ctypes signature.
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_MP = ctypes.POINTER(BfpMatrixC)
_LP = ctypes.POINTER(MoeLayerC)
SIGNATURES = {
    "bfp_packed_size": [_I, _I64, _I64, ctypes.POINTER(_I64)],
    "bfp_encode": [_I, _P, _I64, _I64, _P, _I64, _I],
    "bfp_encode_gate_up": [_I, _P, _P, _I64, _I64, _P, _I64, _I],
    "bfp_gptq_factor": [_P, _I64, _I64, ctypes.c_double, _P, _I],
    "bfp_encode_gptq": [_I, _P, _I64, _I64, _P, _P, _I64, _I],
    "bfp_encode_gate_up_gptq": [_I, _P, _P, _I64, _I64, _P, _P, _I64, _I],
    "bfp_read_fields": [_MP, _P, _P],
    "bfp_decode_host": [_MP, _P],
    "bfp_unpack_device": [_MP, _P, _P],
    "bfp_linear_workspace_size": [_MP, _I, ctypes.POINTER(_SZ)],
    "bfp_linear": [_MP, _P, _I, _I64, _P, _P, _I64, _P, _SZ, _P],
    "bfp_linear_greedy": [_MP, _P, _I, _I64, _P, _I64, _P, _P, _SZ, _P],
    "moe_workspace_size": [_LP, _I, ctypes.POINTER(_SZ)],
    "bfp_workspace_init": [_P, _SZ, _P],
    "moe_decode_layer": [_LP, _P, _I, _P, _P, _P, _P, _SZ, _P],
    "moe_decode_layer_static": [_LP, _P, _I, _P, _P, _P, _P],
    "moe_stack_workspace_size": [_LP, _I, _MP, _I, ctypes.POINTER(_SZ)],
    "moe_stack_decode": [_LP, _I, _MP, _P, _I, _P, _P, _P, _SZ, _P],
    "moe_stack_decode_greedy": [_LP, _I, _MP, _P, _I, _P, _P, _P, _P, _SZ, _P],
    "bfp_greedy_workspace_size": [_I, _I64, ctypes.POINTER(_SZ)],
    "bfp_greedy_tokens": [_P, _I, _I64, _I64, _P, _P, _SZ, _P],
    "bfp_kv_cache_size": [_I, _I, _I, _I64, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)],
    "bfp_kv_encode_host": [ctypes.POINTER(KvCacheC), _P, _P, _I64, _I, _I],
    "bfp_kv_read_fields": [ctypes.POINTER(KvCacheC), _I, _I64, _I64, _P, _P],
    "bfp_kv_append": [ctypes.POINTER(KvCacheC), _P, _P, _I64, _I, _P],
    "bfp_attn_workspace_size": [ctypes.POINTER(KvCacheC), _I, _I64, ctypes.POINTER(_SZ)],
    "bfp_attn_decode": [ctypes.POINTER(KvCacheC), _P, _I, _I64, ctypes.c_float, _P, _P, _SZ, _P],
    "bfp_workspace_status": [_P, ctypes.POINTER(_I), _P],
    "bfp_set_wait_limit": [_I64],
    "bfp_set_launch_mode": [_I],
    "bfp_set_row_path": [_I],
    "bfp_set_linear_path": [_I],
    "bfp_last_error": [],
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load (building first if needed) the native library; raises if it cannot."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            for name, args in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name == "bfp_last_error" else ctypes.c_int
            _lib = lib
    return _lib


def _check(rc: int, fn: str):
    if rc != BFP_OK:
        raise BFPError(rc, fn, load().bfp_last_error().decode())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------------------------- format
def packed_size(fmt: int, n: int, k: int) -> int:
    out = ctypes.c_int64()
    _check(load().bfp_packed_size(fmt, n, k, ctypes.byref(out)), "bfp_packed_size")
    return out.value


def encode(fmt: int, w: np.ndarray, threads: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """Host packer: fp32 [n, k] -> packed uint8 buffer (tile-record layout)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    size = packed_size(fmt, n, k)
    if out is None:
        out = np.empty(size, dtype=np.uint8)
    assert out.nbytes >= size and out.flags.c_contiguous
    _check(load().bfp_encode(fmt, w.ctypes.data, n, k, out.ctypes.data, out.nbytes, threads), "bfp_encode")
    return out


def encode_gate_up(fmt: int, gate: np.ndarray, up: np.ndarray, threads: int = 0,
                   out: np.ndarray | None = None) -> np.ndarray:
    """Host packer for an expert's gate and up [ffn, hidden] -> packed [2*ffn, hidden] (row groups interleaved)."""
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    up = np.ascontiguousarray(up, dtype=np.float32)
    ffn, hidden = gate.shape
    assert up.shape == gate.shape
    size = packed_size(fmt, 2 * ffn, hidden)
    if out is None:
        out = np.empty(size, dtype=np.uint8)
    assert out.nbytes >= size
    _check(load().bfp_encode_gate_up(fmt, gate.ctypes.data, up.ctypes.data, ffn, hidden, out.ctypes.data,
                                     out.nbytes, threads), "bfp_encode_gate_up")
    return out


def gptq_factor(x: np.ndarray, damp: float = 0.01, threads: int = 0) -> np.ndarray:
    """Upper factor u [k, k] (fp64) with H^-1 = u^T u, H = x^T x / t + damp * mean(diag) * I (x: [t, k] fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    t, k = x.shape
    u = np.empty((k, k), dtype=np.float64)
    _check(load().bfp_gptq_factor(x.ctypes.data, t, k, float(damp), u.ctypes.data, threads), "bfp_gptq_factor")
    return u


def encode_gptq(fmt: int, w: np.ndarray, u: np.ndarray, threads: int = 0) -> np.ndarray:
    """Error-compensated host encoding of fp32 w [n, k] with the factor u [k, k]; packed bytes."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float64)
    n, k = w.shape
    if u.shape != (k, k):
        raise ValueError("u must be [k, k]")
    out = np.empty(packed_size(fmt, n, k), dtype=np.uint8)
    _check(load().bfp_encode_gptq(fmt, w.ctypes.data, n, k, u.ctypes.data, out.ctypes.data, out.nbytes, threads),
           "bfp_encode_gptq")
    return out


def encode_gate_up_gptq(fmt: int, gate: np.ndarray, up: np.ndarray, u: np.ndarray, threads: int = 0) -> np.ndarray:
    """bfp_encode_gate_up's layout with both halves error-compensated through the same factor u."""
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    up = np.ascontiguousarray(up, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float64)
    ffn, hidden = gate.shape
    if up.shape != gate.shape or u.shape != (hidden, hidden):
        raise ValueError("gate and up must match; u must be [hidden, hidden]")
    out = np.empty(packed_size(fmt, 2 * ffn, hidden), dtype=np.uint8)
    _check(load().bfp_encode_gate_up_gptq(fmt, gate.ctypes.data, up.ctypes.data, ffn, hidden, u.ctypes.data,
                                          out.ctypes.data, out.nbytes, threads), "bfp_encode_gate_up_gptq")
    return out


def _host_matrix(fmt, n, k, packed: np.ndarray) -> BfpMatrixC:
    return BfpMatrixC(fmt, 0, n, k, packed.ctypes.data, packed_size(fmt, n, k))


def read_fields(fmt: int, n: int, k: int, packed: np.ndarray):
    """Logical (exps [n, k/16], codes [n, k]) of a packed host buffer."""
    m = _host_matrix(fmt, n, k, packed)
    exps = np.zeros((n, k // 16), dtype=np.uint8)
    codes = np.zeros((n, k), dtype=np.uint8)
    _check(load().bfp_read_fields(ctypes.byref(m), exps.ctypes.data, codes.ctypes.data), "bfp_read_fields")
    return exps, codes


def decode_host(fmt: int, n: int, k: int, packed: np.ndarray) -> np.ndarray:
    m = _host_matrix(fmt, n, k, packed)
    out = np.zeros((n, k), dtype=np.float32)
    _check(load().bfp_decode_host(ctypes.byref(m), out.ctypes.data), "bfp_decode_host")
    return out


class DeviceMatrix:
    """A packed BFP matrix resident in device memory (a torch uint8 CUDA tensor)."""

    def __init__(self, fmt: int, n: int, k: int, data):
        self.fmt, self.n, self.k, self.data = fmt, n, k, data
        self.nbytes = packed_size(fmt, n, k)
        assert data.numel() >= self.nbytes

    @classmethod
    def from_host(cls, fmt, n, k, packed: np.ndarray, device="cuda"):
        import torch
        t = torch.from_numpy(np.ascontiguousarray(packed)).to(device)
        return cls(fmt, n, k, t)

    def c(self) -> BfpMatrixC:
        return BfpMatrixC(self.fmt, 0, self.n, self.k, self.data.data_ptr(), self.nbytes)


def unpack_device(mat: DeviceMatrix, stream=None):
    import torch
    out = torch.empty((mat.n, mat.k), dtype=torch.float32, device=mat.data.device)
    m = mat.c()
    _check(load().bfp_unpack_device(ctypes.byref(m), _ptr(out), _stream(stream)), "bfp_unpack_device")
    return out


# ----------------------------------------------------------------------------- workspaces
def workspace_init(ws, stream=None):
    _check(load().bfp_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "bfp_workspace_init")


def workspace_status(ws, stream=None) -> int:
    st = ctypes.c_int()
    _check(load().bfp_workspace_status(_ptr(ws), ctypes.byref(st), _stream(stream)), "bfp_workspace_status")
    return st.value


def set_wait_limit(iterations: int):
    _check(load().bfp_set_wait_limit(iterations), "bfp_set_wait_limit")


LAUNCH_DEPENDENT, LAUNCH_COOPERATIVE = 0, 1


def set_launch_mode(mode: int):
    """How the MoE layer kernel is launched (include/bfpmoe.h, bfp_set_launch_mode)."""
    _check(load().bfp_set_launch_mode(mode), "bfp_set_launch_mode")


def set_row_path(enabled: bool):
    """Which kernel runs one-row MoE layers: the one-row kernel (True, default) or the general one
    (include/bfpmoe.h, bfp_set_row_path)."""
    _check(load().bfp_set_row_path(1 if enabled else 0), "bfp_set_row_path")


def set_linear_path(mode: int):
    """Which kernel bfp_linear runs: 0 (default) or 1 the mma.sync kernel, 2 the tcgen05 kernel wherever the
    shape fits it (include/bfpmoe.h, bfp_set_linear_path)."""
    _check(load().bfp_set_linear_path(int(mode)), "bfp_set_linear_path")


def _alloc_ws(nbytes: int, device, stream=None):
    import torch
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


# ----------------------------------------------------------------------------- dense linear
def linear_workspace_size(mat: DeviceMatrix, m: int) -> int:
    out = ctypes.c_size_t()
    c = mat.c()
    _check(load().bfp_linear_workspace_size(ctypes.byref(c), m, ctypes.byref(out)), "bfp_linear_workspace_size")
    return out.value


def linear_workspace(mat: DeviceMatrix, m: int, stream=None):
    return _alloc_ws(linear_workspace_size(mat, m), mat.data.device, stream)


def linear(mat: DeviceMatrix, x, ws, y=None, y_bf16=None, stream=None):
    """y = x W^T for bf16 x [m, k] (CUDA tensor); fills y (fp32 [m, n]) and/or y_bf16 (bf16 [m, n])."""
    import torch
    m = x.shape[0]
    if y is None and y_bf16 is None:
        y = torch.empty((m, mat.n), dtype=torch.float32, device=x.device)
    ldy = (y if y is not None else y_bf16).stride(0)
    c = mat.c()
    _check(load().bfp_linear(ctypes.byref(c), _ptr(x), m, x.stride(0), _ptr(y), _ptr(y_bf16), ldy, _ptr(ws),
                             ws.numel(), _stream(stream)), "bfp_linear")
    return y if y is not None else y_bf16


def linear_greedy(mat: DeviceMatrix, x, ws, tokens=None, y=None, stream=None):
    """Greedy next token per row of y = x W^T, taken in the projection's epilogue (bfp_linear_greedy): int32 [m];
    y (optional fp32 [m, n] CUDA tensor) also receives the outputs."""
    import torch
    m = x.shape[0]
    if tokens is None:
        tokens = torch.empty(m, dtype=torch.int32, device=x.device)
    ldy = y.stride(0) if y is not None else mat.n
    c = mat.c()
    _check(load().bfp_linear_greedy(ctypes.byref(c), _ptr(x), m, x.stride(0), _ptr(y), ldy, _ptr(tokens), _ptr(ws),
                                    ws.numel(), _stream(stream)), "bfp_linear_greedy")
    return tokens


# ----------------------------------------------------------------------------- MoE layer
class MoELayer:
    """Device-resident weights of one MoE decode layer (all BFP experts packed, bf16 router/gate)."""

    def __init__(self, hidden, n_experts, ffn, top_k, shared_ffn, expert_fmt, router, shared_gate,
                 experts_gate_up, experts_down, shared_gate_up, shared_down, router_bias=None):
        self.hidden, self.n_experts, self.ffn, self.top_k, self.shared_ffn = hidden, n_experts, ffn, top_k, shared_ffn
        self.expert_fmt = expert_fmt
        self.router, self.shared_gate, self.router_bias = router, shared_gate, router_bias
        self.experts_gate_up, self.experts_down = experts_gate_up, experts_down
        self.shared_gate_up, self.shared_down = shared_gate_up, shared_down
        self.gate_up_bytes = packed_size(expert_fmt, 2 * ffn, hidden)
        self.down_bytes = packed_size(expert_fmt, hidden, ffn)

    def c(self) -> MoeLayerC:
        return MoeLayerC(self.hidden, self.n_experts, self.ffn, self.top_k, self.shared_ffn, self.expert_fmt,
                         self.router.data_ptr(), None if self.router_bias is None else self.router_bias.data_ptr(),
                         self.shared_gate.data_ptr(), self.experts_gate_up.data_ptr(), self.experts_down.data_ptr(),
                         self.gate_up_bytes, self.down_bytes, self.shared_gate_up.data_ptr(),
                         self.shared_down.data_ptr())

    def weight_bytes(self, n_routed: int) -> int:
        """BFP bytes one step streams for n_routed distinct routed experts plus the shared expert."""
        sh = packed_size(self.expert_fmt, 2 * self.shared_ffn, self.hidden) + \
            packed_size(self.expert_fmt, self.hidden, self.shared_ffn)
        return n_routed * (self.gate_up_bytes + self.down_bytes) + sh

    @classmethod
    def from_source(cls, hidden, n_experts, ffn, top_k, shared_ffn, expert_fmt, router_bf16: np.ndarray,
                    shared_gate_bf16: np.ndarray, expert_source, shared_source, router_bias=None, device="cuda",
                    threads: int = 0, gptq_factors=None, shared_gptq_factors=None):
        """Pack fp32 weights on the host (pack_experts) and upload them.

        expert_source(e) -> (gate [ffn, hidden], up [ffn, hidden], down [hidden, ffn]) fp32;
        shared_source() -> the same for the shared expert. gptq_factors(e) / shared_gptq_factors()
        (optional) -> (u_in [hidden, hidden], u_mid [ffn, ffn]) fp64 factors from gptq_factor
        of the expert's calibration inputs (x for gate/up, h for down): error-compensated encoding.
        """
        import torch
        host_gu, host_dn = pack_experts(hidden, n_experts, ffn, expert_fmt, expert_source, threads, gptq_factors)
        sgu, sdn = pack_experts(hidden, 1, shared_ffn, expert_fmt, lambda e: shared_source(), threads,
                                None if shared_gptq_factors is None else (lambda e: shared_gptq_factors()))
        dev = torch.device(device)

        def up_(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        rb = None if router_bias is None else up_(np.asarray(router_bias, dtype=np.float32))
        return cls(hidden, n_experts, ffn, top_k, shared_ffn, expert_fmt,
                   up_(np.asarray(router_bf16, dtype=np.uint16).view(np.int16)),
                   up_(np.asarray(shared_gate_bf16, dtype=np.uint16).view(np.int16)),
                   up_(host_gu), up_(host_dn), up_(sgu), up_(sdn), router_bias=rb)


def pack_experts(hidden, n_experts, ffn, expert_fmt, expert_source, threads: int = 0, gptq_factors=None):
    """Host packing of a layer's experts: (gate/up bytes of all experts, down bytes of all experts), each
    expert at a stride of its packed size (the layout moe_decode_layer reads). expert_source(e) -> fp32
    (gate, up, down); gptq_factors(e) -> (u_in, u_mid) selects error-compensated encoding (bfp_encode_gate_up_gptq
    with u_in, bfp_encode_gptq of down with u_mid), else round to nearest."""
    gub = packed_size(expert_fmt, 2 * ffn, hidden)
    dnb = packed_size(expert_fmt, hidden, ffn)
    host_gu = np.empty(n_experts * gub, dtype=np.uint8)
    host_dn = np.empty(n_experts * dnb, dtype=np.uint8)

    def pack(e):
        g, u, d = expert_source(e)
        if gptq_factors is None:
            encode_gate_up(expert_fmt, g, u, threads, out=host_gu[e * gub:(e + 1) * gub])
            encode(expert_fmt, d, threads, out=host_dn[e * dnb:(e + 1) * dnb])
        else:
            u_in, u_mid = gptq_factors(e)
            host_gu[e * gub:(e + 1) * gub] = encode_gate_up_gptq(expert_fmt, g, u, u_in, threads)
            host_dn[e * dnb:(e + 1) * dnb] = encode_gptq(expert_fmt, d, u_mid, threads)

    # experts are independent: pack several at once (the C calls release the GIL)
    import concurrent.futures as cf
    workers = max(1, min(8, (os.cpu_count() or 1) // 2, n_experts))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(pack, range(n_experts)))
    return host_gu, host_dn


def moe_workspace_size(layer: MoELayer, m: int) -> int:
    out = ctypes.c_size_t()
    c = layer.c()
    _check(load().moe_workspace_size(ctypes.byref(c), m, ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_workspace(layer: MoELayer, m: int, stream=None):
    return _alloc_ws(moe_workspace_size(layer, m), layer.router.device, stream)


def moe_decode_layer(layer: MoELayer, x, ws, y=None, topk_idx=None, topk_w=None, stream=None):
    """One MoE decode layer on bf16 x [m, hidden]; returns y fp32 [m, hidden] (and fills topk_idx/topk_w)."""
    import torch
    m = x.shape[0]
    if y is None:
        y = torch.empty((m, layer.hidden), dtype=torch.float32, device=x.device)
    c = layer.c()
    _check(load().moe_decode_layer(ctypes.byref(c), _ptr(x), m, _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                                   ws.numel(), _stream(stream)), "moe_decode_layer")
    return y


def moe_decode_layer_static(layer: MoELayer, x, y=None, topk_idx=None, topk_w=None, stream=None):
    """moe_decode_layer without a workspace, for callers that cannot allocate device memory.

    Uses the library's built-in 1.5 MiB device scratch array (shared by every
    call on a device; overlapping calls race). The first call on a device
    sets the array up synchronously, so make it before any stream capture.
    """
    import torch
    m = x.shape[0]
    if y is None:
        y = torch.empty((m, layer.hidden), dtype=torch.float32, device=x.device)
    c = layer.c()
    _check(load().moe_decode_layer_static(ctypes.byref(c), _ptr(x), m, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                                          _stream(stream)), "moe_decode_layer_static")
    return y


def _layers_array(layers):
    arr = (MoeLayerC * len(layers))()
    for i, l in enumerate(layers):
        arr[i] = l.c()
    return arr


def moe_stack_workspace_size(layers, lm_head: DeviceMatrix, m: int) -> int:
    out = ctypes.c_size_t()
    arr = _layers_array(layers)
    c = lm_head.c()
    _check(load().moe_stack_workspace_size(arr, len(layers), ctypes.byref(c), m, ctypes.byref(out)),
           "moe_stack_workspace_size")
    return out.value


def moe_stack_workspace(layers, lm_head: DeviceMatrix, m: int, stream=None):
    return _alloc_ws(moe_stack_workspace_size(layers, lm_head, m), lm_head.data.device, stream)


def moe_stack_decode(layers, lm_head: DeviceMatrix, h, ws, logits=None, topk_idx=None, stream=None):
    """Decode stack: h (bf16 [m, hidden], updated in place) through every layer, then LM-head logits fp32.
    topk_idx (optional int32 CUDA tensor, [n_layers, m, top_k] when the layers share top_k) receives every
    layer's selection."""
    import torch
    m = h.shape[0]
    if logits is None:
        logits = torch.empty((m, lm_head.n), dtype=torch.float32, device=h.device)
    arr = _layers_array(layers)
    c = lm_head.c()
    if topk_idx is not None and topk_idx.numel() < m * sum(L.top_k for L in layers):
        raise ValueError("topk_idx holds fewer than m * sum(top_k) entries")
    _check(load().moe_stack_decode(arr, len(layers), ctypes.byref(c), _ptr(h), m, _ptr(logits), _ptr(topk_idx),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_stack_decode")
    return logits


def moe_stack_decode_greedy(layers, lm_head: DeviceMatrix, h, ws, tokens=None, logits=None, topk_idx=None,
                            stream=None):
    """The decode stack with the greedy next token taken in the LM head's epilogue: int32 [m] tokens; logits
    (optional fp32 [m, vocab] CUDA tensor) are written only when given."""
    import torch
    m = h.shape[0]
    if tokens is None:
        tokens = torch.empty(m, dtype=torch.int32, device=h.device)
    arr = _layers_array(layers)
    c = lm_head.c()
    if topk_idx is not None and topk_idx.numel() < m * sum(L.top_k for L in layers):
        raise ValueError("topk_idx holds fewer than m * sum(top_k) entries")
    _check(load().moe_stack_decode_greedy(arr, len(layers), ctypes.byref(c), _ptr(h), m, _ptr(logits),
                                          _ptr(tokens), _ptr(topk_idx), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_stack_decode_greedy")
    return tokens


# ----------------------------------------------------------------------------- greedy next token
def greedy_workspace_size(m: int, n: int) -> int:
    out = ctypes.c_size_t()
    _check(load().bfp_greedy_workspace_size(m, n, ctypes.byref(out)), "bfp_greedy_workspace_size")
    return out.value


def greedy_workspace(m: int, n: int, device, stream=None):
    return _alloc_ws(greedy_workspace_size(m, n), device, stream)


def greedy_tokens(logits, ws, tokens=None, stream=None):
    """Greedy next token per row of fp32 logits [m, n] (CUDA tensor): int32 [m] arg max, ties to the lower index."""
    import torch
    m, n = logits.shape
    if tokens is None:
        tokens = torch.empty(m, dtype=torch.int32, device=logits.device)
    _check(load().bfp_greedy_tokens(_ptr(logits), m, n, logits.stride(0), _ptr(tokens), _ptr(ws), ws.numel(),
                                    _stream(stream)), "bfp_greedy_tokens")
    return tokens


# ----------------------------------------------------------------------------- BFP KV cache + decode attention
class KvCache:
    """Device arrays of one layer's BFP KV cache (include/bfpmoe.h, bfp_kv_cache)."""

    def __init__(self, kv_heads, head_dim, capacity, k_fmt=BFP8, v_fmt=BFP8, v_rotated=False, device="cuda"):
        import torch
        self.kv_heads, self.head_dim, self.capacity = kv_heads, head_dim, capacity
        self.k_fmt, self.v_fmt, self.v_rotated = k_fmt, v_fmt, bool(v_rotated)
        self.k_codes, self.k_exps = (torch.zeros(n, dtype=torch.uint8, device=device)
                                     for n in kv_cache_size(k_fmt, kv_heads, head_dim, capacity))
        self.v_codes, self.v_exps = (torch.zeros(n, dtype=torch.uint8, device=device)
                                     for n in kv_cache_size(v_fmt, kv_heads, head_dim, capacity))

    def c(self) -> KvCacheC:
        return KvCacheC(self.kv_heads, self.head_dim, self.k_fmt, self.v_fmt, int(self.v_rotated), 0, self.capacity,
                        self.k_codes.data_ptr(), self.k_exps.data_ptr(), self.v_codes.data_ptr(),
                        self.v_exps.data_ptr())

    def bytes_per_token(self) -> int:
        d, h = self.head_dim, self.kv_heads
        code = {BFP8: d, BFP4: d // 2}
        return h * (code[self.k_fmt] + code[self.v_fmt] + 2 * (d // 16))


def kv_cache_size(fmt: int, kv_heads: int, head_dim: int, capacity: int):
    cb, eb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().bfp_kv_cache_size(fmt, kv_heads, head_dim, capacity, ctypes.byref(cb), ctypes.byref(eb)),
           "bfp_kv_cache_size")
    return cb.value, eb.value


def kv_read_fields(cache: KvCache, which: str, t0: int, n: int):
    """Logical fields of tokens t0 .. t0 + n - 1 of K ("k") or V ("v"), read from a host copy of the cache:
    (exps [kv_heads, n, head_dim/16], codes [kv_heads, n, head_dim]) uint8."""
    arrs = [a.cpu().numpy() for a in (cache.k_codes, cache.k_exps, cache.v_codes, cache.v_exps)]
    return kv_read_host_fields(cache.kv_heads, cache.head_dim, cache.capacity, cache.k_fmt, cache.v_fmt,
                               cache.v_rotated, arrs, which, t0, n)


def kv_encode_host(kv_heads, head_dim, capacity, k_fmt, v_fmt, v_rotated, arrays, k, v, pos: int, threads: int = 0):
    """bfp_kv_encode_host into host arrays (k_codes, k_exps, v_codes, v_exps; uint8 numpy, written in place) from
    bf16 bit patterns k, v [n_new, kv_heads, head_dim] (uint16 numpy)."""
    for a in arrays:
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    c = KvCacheC(kv_heads, head_dim, k_fmt, v_fmt, int(v_rotated), 0, capacity, *[a.ctypes.data for a in arrays])
    _check(load().bfp_kv_encode_host(ctypes.byref(c), k.ctypes.data, v.ctypes.data, pos, k.shape[0], threads),
           "bfp_kv_encode_host")


def kv_read_host_fields(kv_heads, head_dim, capacity, k_fmt, v_fmt, v_rotated, arrays, which: str, t0: int, n: int):
    """bfp_kv_read_fields over host arrays (k_codes, k_exps, v_codes, v_exps) of a cache's layout."""
    arrays = [np.ascontiguousarray(a, dtype=np.uint8) for a in arrays]
    c = KvCacheC(kv_heads, head_dim, k_fmt, v_fmt, int(v_rotated), 0, capacity, *[a.ctypes.data for a in arrays])
    exps = np.empty((kv_heads, n, head_dim // 16), np.uint8)
    codes = np.empty((kv_heads, n, head_dim), np.uint8)
    _check(load().bfp_kv_read_fields(ctypes.byref(c), {"k": 0, "v": 1}[which], t0, n, exps.ctypes.data,
                                     codes.ctypes.data), "bfp_kv_read_fields")
    return exps, codes


def kv_append(cache: KvCache, k, v, pos: int, stream=None):
    """Encode bf16 k, v [n_new, kv_heads, head_dim] (CUDA tensors) into slots pos .. pos + n_new - 1."""
    c = cache.c()
    _check(load().bfp_kv_append(ctypes.byref(c), _ptr(k), _ptr(v), pos, k.shape[0], _stream(stream)), "bfp_kv_append")


def attn_workspace_size(cache: KvCache, q_heads: int, n_ctx: int) -> int:
    out = ctypes.c_size_t()
    c = cache.c()
    _check(load().bfp_attn_workspace_size(ctypes.byref(c), q_heads, n_ctx, ctypes.byref(out)),
           "bfp_attn_workspace_size")
    return out.value


def attn_workspace(cache: KvCache, q_heads: int, n_ctx: int, stream=None):
    return _alloc_ws(attn_workspace_size(cache, q_heads, n_ctx), cache.k_codes.device, stream)


def attn_decode(cache: KvCache, q, n_ctx: int, scale: float, ws, out=None, stream=None):
    """Decode attention of bf16 q [q_heads, head_dim] over the first n_ctx cached tokens; fp32 out."""
    import torch
    qh = q.shape[0]
    if out is None:
        out = torch.empty((qh, cache.head_dim), dtype=torch.float32, device=q.device)
    c = cache.c()
    _check(load().bfp_attn_decode(ctypes.byref(c), _ptr(q), qh, n_ctx, float(scale), _ptr(out), _ptr(ws), ws.numel(),
                                  _stream(stream)), "bfp_attn_decode")
    return out
