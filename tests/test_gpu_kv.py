"""GPU parity of the BFP KV cache (append: bit-exact cache bytes) and decode attention (within
1e-3 * (|oracle| + rms(oracle)) per element) against the oracle, through the C-ABI.

Inputs: seeded N(0, 1) bf16 K, V and q (K scaled up in one case so that scores span tens of units and
the running softmax has to rescale across chunks); shapes of the pages' two caches (2 KV heads x 256,
BFP8 K and V, 16 query heads; 4 KV heads x 256, BFP8 K and rotated BFP4 V, 24 query heads) plus other
head sizes, group sizes and formats; contexts from 1 token to 32,768, with ragged last chunks; cache
slots past the context filled with random bytes, which must not matter.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from harness import expected_codes, tile_bytes, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

bfp = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global bfp
    import block_floating_point_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    bfp = m
    yield


def bf16_rows(seed, stream, shape, std=1.0):
    return synth.to_bf16_bits(synth.normal(seed, stream, shape, std=std))


def build_cache(seed, kvh, d, cap, n, k_fmt, v_fmt, rot, k_std=1.0, chunks=(None,)):
    """Append n tokens (in the given pieces), return the device cache and the bf16 K, V [n, kvh, d]."""
    cache = bfp.KvCache(kvh, d, cap, k_fmt, v_fmt, rot)
    g = torch.Generator(device="cpu").manual_seed(seed)
    for t in (cache.k_codes, cache.k_exps, cache.v_codes, cache.v_exps):  # garbage in every slot
        t.copy_(torch.randint(0, 256, t.shape, generator=g, dtype=torch.uint8))
    k = bf16_rows(seed, 1, (n, kvh, d), std=k_std)
    v = bf16_rows(seed, 2, (n, kvh, d))
    pos = 0
    pieces = [n] if chunks == (None,) else list(chunks)
    assert sum(pieces) == n
    for p in pieces:
        kt = torch.from_numpy(k[pos:pos + p].view(np.int16)).cuda()
        vt = torch.from_numpy(v[pos:pos + p].view(np.int16)).cuda()
        bfp.kv_append(cache, kt, vt, pos)
        pos += p
    torch.cuda.synchronize()
    return cache, k, v


@pytest.mark.parametrize("kvh,d,k_fmt,v_fmt,rot", [(2, 256, 8, 8, False), (4, 256, 8, 4, True), (3, 128, 4, 8, True),
                                                   (2, 64, 8, 4, False), (1, 64, 4, 4, True)])
def test_append_is_bit_exact(kvh, d, k_fmt, v_fmt, rot):
    n, cap = 150, 256
    cache, k, v = build_cache(10 + d + kvh, kvh, d, cap, n, k_fmt, v_fmt, rot, chunks=(100, 1, 1, 48))
    ke, kc = oracle.kv_encode(k_fmt, k.transpose(1, 0, 2), False)
    ve, vc = oracle.kv_encode(v_fmt, v.transpose(1, 0, 2), rot)
    nb = d // 16
    for which, fmt, (e, c), (tc, te) in (("k", k_fmt, (ke, kc), (cache.k_codes, cache.k_exps)),
                                         ("v", v_fmt, (ve, vc), (cache.v_codes, cache.v_exps))):
        assert np.array_equal(te.cpu().numpy().reshape(kvh, cap, nb)[:, :n], e)
        got = tc.cpu().numpy().reshape(kvh, cap // 16, nb, -1)
        want = expected_codes(np.asarray(c, np.uint8), which, fmt, cap)
        full_groups = n // 16  # whole tiles; the last, partial tile is checked on its written rows below
        assert np.array_equal(got[:, :full_groups], want[:, :full_groups])
        if n % 16:
            # rows past n in the last tile hold the random fill: compare the bytes of written rows only
            g = full_groups
            for h in range(kvh):
                for b in range(nb):
                    mask = tile_bytes(np.where(np.arange(16)[:, None] < n % 16, 0xFF if fmt == 8 else 0xF, 0)
                                      * np.ones((16, 16), np.int64), which, fmt)
                    assert np.array_equal(got[h, g, b] & mask, want[h, g, b] & mask)


CASES = [  # kvh, G, d, k_fmt, v_fmt, rot, n_ctx, cap, k_std
    (2, 8, 256, 8, 8, False, 1, 64, 1.0),
    (2, 8, 256, 8, 8, False, 65, 128, 1.0),
    (2, 8, 256, 8, 8, False, 1000, 1024, 1.0),
    (2, 8, 256, 8, 8, False, 32768, 32768, 1.0),     # the BFP8 cache of the 35B card's attention layers
    (4, 6, 256, 8, 4, True, 4097, 4160, 1.0),        # bfp8_v4r of the 27B card
    (4, 6, 256, 8, 4, True, 32768, 32768, 1.0),
    (2, 8, 256, 8, 8, False, 3000, 3008, 6.0),       # large scores: the running max moves between chunks
    (4, 4, 128, 8, 8, False, 777, 832, 1.0),
    (8, 1, 64, 8, 4, True, 300, 320, 1.0),
    (2, 2, 64, 4, 4, False, 129, 192, 1.0),
]


@pytest.mark.parametrize("kvh,G,d,k_fmt,v_fmt,rot,n_ctx,cap,k_std", CASES)
def test_attention_matches_oracle(kvh, G, d, k_fmt, v_fmt, rot, n_ctx, cap, k_std):
    seed = 100 + n_ctx + d + kvh
    cache, k, v = build_cache(seed, kvh, d, cap, n_ctx, k_fmt, v_fmt, rot, k_std=k_std)
    q = bf16_rows(seed, 3, (kvh * G, d))
    scale = 1.0 / math.sqrt(d)
    ws = bfp.attn_workspace(cache, kvh * G, n_ctx)
    out = bfp.attn_decode(cache, torch.from_numpy(q.view(np.int16)).cuda(), n_ctx, scale, ws)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    got = out.cpu().numpy().astype(np.float64)
    kf = oracle.kv_encode(k_fmt, k.transpose(1, 0, 2), False)
    vf = oracle.kv_encode(v_fmt, v.transpose(1, 0, 2), rot)
    want = oracle.attn_decode(q, kf, vf, n_ctx, scale, k_fmt, v_fmt, rot)
    # the stated tolerance, rms per output row (one query head)
    assert_close(got, want, "attention output")
    # a shorter context over the same cache only sees its own tokens
    n2 = max(1, n_ctx // 3)
    ws2 = bfp.attn_workspace(cache, kvh * G, n2)
    out2 = bfp.attn_decode(cache, torch.from_numpy(q.view(np.int16)).cuda(), n2, scale, ws2)
    want2 = oracle.attn_decode(q, kf, vf, n2, scale, k_fmt, v_fmt, rot)
    assert_close(out2.cpu().numpy(), want2, "attention output, shorter context")


def test_attention_rejects_bad_arguments():
    cache = bfp.KvCache(2, 128, 128)
    ws = bfp.attn_workspace(cache, 16, 100)
    q = torch.zeros((18, 128), dtype=torch.int16, device="cuda")
    for qh, n, code in ((18, 100, bfp.BFP_ESHAPE), (3, 100, bfp.BFP_ESHAPE), (16, 129, bfp.BFP_ESHAPE),
                        (16, 0, bfp.BFP_ESHAPE)):
        with pytest.raises(bfp.BFPError) as e:
            bfp.attn_decode(cache, q[:qh], n, 0.1, ws)
        assert e.value.code == code
    with pytest.raises(bfp.BFPError) as e:
        bfp.attn_decode(cache, q[:16], 100, 0.1, ws[:64])
    assert e.value.code == bfp.BFP_EWORKSPACE
    with pytest.raises(bfp.BFPError) as e:
        bfp.KvCache(2, 96, 128)
    assert e.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as e:
        bfp.KvCache(2, 128, 100)
    assert e.value.code == bfp.BFP_ESHAPE
    kt = torch.zeros((4, 2, 128), dtype=torch.int16, device="cuda")
    with pytest.raises(bfp.BFPError) as e:
        bfp.kv_append(cache, kt, kt, 126)  # past the capacity
    assert e.value.code == bfp.BFP_ESHAPE
