"""C-ABI library on the CPU: loads, exports every symbol of include/bfpmoe.h, and
its host packer agrees bit for bit with the oracle's encoding.

The packed layout is read back two independent ways: by the library's own
``bfp_read_fields`` and by a NumPy statement of the layout text in the header
(``layout_fields`` below), so a packer bug that the library's reader mirrored
would still show.
"""
import os
import re

import numpy as np
import pytest

import block_floating_point_gb300 as bfp
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    txt = open(os.path.join(ROOT, "include", "bfpmoe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char \*)\s*\*?\s*(\w+)\s*\(", txt, flags=re.M)))


def test_library_exports_every_header_symbol():
    lib = bfp.load()
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in bfp.SIGNATURES, n
    assert set(bfp.SIGNATURES) == set(names)


def layout_fields(fmt, n, k, packed):
    """NumPy reading of the tile-record layout exactly as include/bfpmoe.h states it."""
    cb = 4 if fmt == 4 else 2
    mb = 3 if fmt == 4 else 7
    rec = 512 + 16 * cb
    ng = (n + 15) // 16
    kb = k // 16
    kc = (kb + cb - 1) // cb
    codes = np.zeros((ng * 16, kc * cb * 16), dtype=np.uint8)
    exps = np.zeros((ng * 16, kc * cb), dtype=np.uint8)
    buf = np.asarray(packed, dtype=np.uint8)[: ng * kc * rec].reshape(ng, kc, rec)
    words = buf[:, :, :512].copy().view("<u4").reshape(ng, kc, 32, 4)
    ex = buf[:, :, 512:].reshape(ng, kc, 8, cb, 2)
    for g in range(8):
        for b in range(cb):
            for h in range(2):
                exps[np.arange(ng)[:, None] * 16 + g + 8 * h, np.arange(kc)[None, :] * cb + b] = ex[:, :, g, b, h]

    def bits(w, pos, cnt):
        pos %= 32
        return (w >> np.uint32(pos)) & np.uint32((1 << cnt) - 1) if pos + cnt <= 32 else None

    for lane in range(32):
        g, t = lane >> 2, lane & 3
        for b in range(cb):
            blk = np.arange(kc)[None, :] * cb + b
            rows0 = np.arange(ng)[:, None] * 16 + g
            if fmt == 4:
                w = words[:, :, lane, b]
                pairs = [(rows0, 2 * t), (rows0 + 8, 2 * t), (rows0, 2 * t + 8), (rows0 + 8, 2 * t + 8)]
                for p, (rr, col) in enumerate(pairs):
                    for second in (0, 1):
                        mpos = (16 * second + 4 * p) % 32
                        spos = (15 + 16 * second + 4 * p) % 32
                        m = bits(w, mpos, 3)
                        s = bits(w, spos, 1)
                        codes[rr, blk * 16 + col + second] = (s << np.uint32(mb)) | m
            else:
                for half in range(2):
                    w = words[:, :, lane, 2 * b + half]
                    for q, rr in enumerate((rows0, rows0 + 8)):
                        col = 2 * t + 8 * half
                        for second in (0, 1):
                            mpos = (16 * second + 8 * q) % 32
                            spos = (15 + 16 * second + 8 * q) % 32
                            m = bits(w, mpos, 7)
                            s = bits(w, spos, 1)
                            codes[rr, blk * 16 + col + second] = (s << np.uint32(mb)) | m
    return exps[:n, :kb], codes[:n, :k]


SHAPES = [(16, 64), (16, 16), (37, 96), (5, 208), (64, 512), (130, 2048)]


@pytest.mark.parametrize("fmt", [4, 8])
@pytest.mark.parametrize("n,k", SHAPES)
def test_host_packer_matches_oracle(fmt, n, k):
    w = synth.normal(11, 7000 + n * 31 + k, (n, k), std=0.02)
    if n > 5:  # adversarial rows: zeros, a huge dynamic range, exact ties, saturation
        w[1, :] = 0.0
        w[2, :16] = np.float32(2.0) ** -np.arange(16, dtype=np.float32)
        w[3, :16] = [1.5, 1.25, 1.75, 0.625, -0.375, 1.9999999, -1.9999999, 0.0625] * 2
    packed = bfp.encode(fmt, w)
    assert packed.nbytes == bfp.packed_size(fmt, n, k)
    e_or, c_or = oracle.encode(fmt, w)
    e_lib, c_lib = bfp.read_fields(fmt, n, k, packed)
    assert np.array_equal(e_lib, e_or) and np.array_equal(c_lib, c_or)
    e_lay, c_lay = layout_fields(fmt, n, k, packed)
    assert np.array_equal(e_lay, e_or) and np.array_equal(c_lay, c_or)
    assert np.array_equal(bfp.decode_host(fmt, n, k, packed), oracle.decode(fmt, e_or, c_or))


@pytest.mark.parametrize("fmt", [4, 8])
def test_packed_size_is_the_storage_cost(fmt):
    per_value = oracle.storage_bytes_per_value(fmt)
    for n, k in [(16, 64), (8192, 2048), (512, 2048), (2048, 512), (151936, 2048)]:
        assert bfp.packed_size(fmt, n, k) == int(per_value * n * k)
    # ragged shapes pad to whole records
    assert bfp.packed_size(fmt, 17, 16) == 2 * (512 + 16 * (4 if fmt == 4 else 2))


def test_gate_up_interleaves_row_groups():
    ffn, hidden = 48, 64
    g = synth.normal(5, 1, (ffn, hidden), std=0.02)
    u = synth.normal(5, 2, (ffn, hidden), std=0.02)
    packed = bfp.encode_gate_up(4, g, u)
    e, c = bfp.read_fields(4, 2 * ffn, hidden, packed)
    ge, gc = oracle.encode(4, g)
    ue, uc = oracle.encode(4, u)
    for i in range(ffn // 16):
        assert np.array_equal(c[32 * i:32 * i + 16], gc[16 * i:16 * i + 16])
        assert np.array_equal(c[32 * i + 16:32 * i + 32], uc[16 * i:16 * i + 16])
        assert np.array_equal(e[32 * i:32 * i + 16], ge[16 * i:16 * i + 16])
        assert np.array_equal(e[32 * i + 16:32 * i + 32], ue[16 * i:16 * i + 16])


def test_error_codes():
    with pytest.raises(bfp.BFPError) as ei:
        bfp.packed_size(4, 16, 24)
    assert ei.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.packed_size(5, 16, 32)
    assert ei.value.code == bfp.BFP_EINVAL
    w = np.zeros((16, 32), dtype=np.float32)
    w[3, 7] = np.nan
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode(8, w)
    assert ei.value.code == bfp.BFP_ENONFINITE
    w[3, 7] = np.inf
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode(4, w)
    assert ei.value.code == bfp.BFP_ENONFINITE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.encode_gate_up(4, np.zeros((8, 32), np.float32), np.zeros((8, 32), np.float32))
    assert ei.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.set_wait_limit(-1)
    assert ei.value.code == bfp.BFP_EINVAL
    bfp.set_wait_limit(0)


def test_packer_threads_do_not_change_bytes():
    w = synth.normal(3, 3, (256, 512), std=0.02)
    a = bfp.encode(4, w, threads=1)
    b = bfp.encode(4, w, threads=7)
    assert np.array_equal(a, b)


def test_kv_cache_sizes_match_the_pages():
    """bfp_kv_cache_size against the per-token cache sizes the pages print (tests/golden/storage_sizes.json):
    the 35B bundle's 10 attention layers of 2 KV heads x 256 in BFP8 (20.0 -> 10.6 KiB per token) and the
    27B card's 16,384 K and 16,384 V values per token (K BFP8 with V BFP4: 26,624 instead of 34,816 B)."""
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "storage_sizes.json")))
    cap = 64

    def per_token(fmt, heads, d):
        c, e = bfp.kv_cache_size(fmt, heads, d, cap)
        return (c + e) / cap

    kv = g["bfp8_kv_cache"]
    bfp8_35b = 10 * 2 * per_token(8, 2, 256)  # K and V, 10 layers
    assert 10 * 2 * 2 * 256 * 2 / 1024 == kv["bf16_kib_per_token"]
    assert round(bfp8_35b / 1024, kv["printed_decimals"]) == kv["bfp8_kib_per_token_printed"]
    v = g["bfp4_v_cache"]
    heads = 16384 // 256  # KV heads x layers
    assert heads * (per_token(8, 1, 256) + per_token(8, 1, 256)) == v["bytes_per_token_k_bfp8_v_bfp8"]
    assert heads * (per_token(8, 1, 256) + per_token(4, 1, 256)) == v["bytes_per_token_k_bfp8_v_bfp4"]


def test_greedy_and_kv_argument_checks_on_the_host():
    """Argument validation of the greedy-token and KV-cache entry points happens before any CUDA call."""
    import ctypes
    lib = bfp.load()
    fake = ctypes.c_void_p(4096)  # never dereferenced: every call below is rejected first
    sz = ctypes.c_size_t()
    assert lib.bfp_greedy_tokens(fake, 0, 10, 10, fake, fake, 64, None) == bfp.BFP_ESHAPE
    assert lib.bfp_greedy_tokens(fake, 17, 10, 10, fake, fake, 64, None) == bfp.BFP_ESHAPE
    assert lib.bfp_greedy_tokens(fake, 2, 10, 5, fake, fake, 64, None) == bfp.BFP_EINVAL
    assert lib.bfp_greedy_workspace_size(1, 0, ctypes.byref(sz)) == bfp.BFP_ESHAPE
    c1, c2 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.bfp_kv_cache_size(5, 2, 256, 64, ctypes.byref(c1), ctypes.byref(c2)) == bfp.BFP_EINVAL
    assert lib.bfp_kv_cache_size(8, 2, 96, 64, ctypes.byref(c1), ctypes.byref(c2)) == bfp.BFP_ESHAPE
    assert lib.bfp_kv_cache_size(8, 2, 256, 100, ctypes.byref(c1), ctypes.byref(c2)) == bfp.BFP_ESHAPE
    assert lib.bfp_kv_cache_size(4, 3, 128, 128, ctypes.byref(c1), ctypes.byref(c2)) == bfp.BFP_OK
    assert (c1.value, c2.value) == (3 * 128 * 64, 3 * 128 * 8)

    def cache(**kw):
        f = dict(kv_heads=2, head_dim=128, k_fmt=8, v_fmt=8, v_rotated=0, reserved=0, capacity=128,
                 k_codes=4096, k_exps=8192, v_codes=12288, v_exps=16384)
        f.update(kw)
        return bfp.KvCacheC(*[f[n] for n, _ in bfp.KvCacheC._fields_])

    k = ctypes.c_void_p(4096)
    for kw, code in ((dict(head_dim=96), bfp.BFP_ESHAPE), (dict(reserved=1), bfp.BFP_EINVAL),
                     (dict(v_rotated=2), bfp.BFP_EINVAL), (dict(k_fmt=3), bfp.BFP_EINVAL),
                     (dict(capacity=96), bfp.BFP_ESHAPE), (dict(v_exps=16385), bfp.BFP_EALIGN),
                     (dict(k_codes=0), bfp.BFP_EINVAL)):
        c = cache(**kw)
        assert lib.bfp_kv_append(ctypes.byref(c), k, k, 0, 1, None) == code, kw
    c = cache()
    assert lib.bfp_kv_append(ctypes.byref(c), k, k, 120, 9, None) == bfp.BFP_ESHAPE   # past the capacity
    assert lib.bfp_kv_append(ctypes.byref(c), k, ctypes.c_void_p(4100), 0, 1, None) == bfp.BFP_EALIGN
    assert lib.bfp_attn_workspace_size(ctypes.byref(c), 18, 10, ctypes.byref(sz)) == bfp.BFP_ESHAPE  # group 9
    assert lib.bfp_attn_workspace_size(ctypes.byref(c), 3, 10, ctypes.byref(sz)) == bfp.BFP_ESHAPE
    assert lib.bfp_attn_workspace_size(ctypes.byref(c), 16, 129, ctypes.byref(sz)) == bfp.BFP_ESHAPE
    assert lib.bfp_attn_decode(ctypes.byref(c), k, 16, 0, ctypes.c_float(0.1), k, k, 1 << 20, None) == bfp.BFP_ESHAPE


@pytest.mark.parametrize("kvh,d,k_fmt,v_fmt,rot", [(2, 256, 8, 8, False), (4, 256, 8, 4, True), (3, 64, 4, 8, False)])
def test_kv_read_fields_inverts_the_cache_layout(kvh, d, k_fmt, v_fmt, rot):
    """bfp_kv_read_fields on host arrays packed by the layout text of include/bfpmoe.h (tests/harness.py)
    returns the oracle's fields of the same seeded rows."""
    from harness import expected_codes
    n, cap = 45, 64
    k = synth.to_bf16_bits(synth.normal(901 + d, 1, (kvh, n, d)))
    v = synth.to_bf16_bits(synth.normal(901 + d, 2, (kvh, n, d)))
    ke, kc = oracle.kv_encode(k_fmt, k, False)
    ve, vc = oracle.kv_encode(v_fmt, v, rot)
    nb = d // 16
    arrays = []
    for which, fmt, e, c in (("k", k_fmt, ke, kc), ("v", v_fmt, ve, vc)):
        arrays.append(expected_codes(np.asarray(c, np.uint8), which, fmt, cap).reshape(-1))
        ex = np.zeros((kvh, cap, nb), np.uint8)
        ex[:, :n] = e
        arrays.append(ex.reshape(-1))
    for which, (e, c) in (("k", (ke, kc)), ("v", (ve, vc))):
        got_e, got_c = bfp.kv_read_host_fields(kvh, d, cap, k_fmt, v_fmt, rot, arrays, which, 0, n)
        assert np.array_equal(got_e, e) and np.array_equal(got_c, c)
        got_e, got_c = bfp.kv_read_host_fields(kvh, d, cap, k_fmt, v_fmt, rot, arrays, which, 17, 20)
        assert np.array_equal(got_e, e[:, 17:37]) and np.array_equal(got_c, c[:, 17:37])


@pytest.mark.parametrize("kvh,d,k_fmt,v_fmt,rot", [(2, 256, 8, 8, False), (4, 256, 8, 4, True), (3, 128, 4, 8, True),
                                                   (1, 64, 4, 4, True)])
def test_kv_encode_host_matches_the_oracle(kvh, d, k_fmt, v_fmt, rot):
    """bfp_kv_encode_host: the cache bytes of the oracle's fields (layout text of include/bfpmoe.h), written
    in two appends; slots never written keep their bytes."""
    from harness import expected_codes
    n, cap = 45, 64
    k = synth.to_bf16_bits(synth.normal(951 + d, 1, (n, kvh, d)))
    v = synth.to_bf16_bits(synth.normal(951 + d, 2, (n, kvh, d)))
    sizes = [bfp.kv_cache_size(f, kvh, d, cap) for f in (k_fmt, v_fmt)]
    arrays = [np.zeros(sizes[0][0], np.uint8), np.zeros(sizes[0][1], np.uint8),
              np.zeros(sizes[1][0], np.uint8), np.zeros(sizes[1][1], np.uint8)]
    bfp.kv_encode_host(kvh, d, cap, k_fmt, v_fmt, rot, arrays, k[:20], v[:20], 0, threads=3)
    bfp.kv_encode_host(kvh, d, cap, k_fmt, v_fmt, rot, arrays, k[20:], v[20:], 20)
    nb = d // 16
    for i, (which, fmt, src, r) in enumerate((("k", k_fmt, k, False), ("v", v_fmt, v, rot))):
        e, c = oracle.kv_encode(fmt, src.transpose(1, 0, 2), r)
        assert np.array_equal(arrays[2 * i].reshape(kvh, cap // 16, nb, -1),
                              expected_codes(np.asarray(c, np.uint8), which, fmt, cap))
        ex = arrays[2 * i + 1].reshape(kvh, cap, nb)
        assert np.array_equal(ex[:, :n], e) and not ex[:, n:].any()
