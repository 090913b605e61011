"""GPU parity of the greedy next-token step (bfp_greedy_tokens) against the oracle: bit-exact indices.

Inputs are seeded normal logits (the LM head's output range) with planted cases: a tie for the row
maximum at two indices, signed zeros, infinities, NaNs, a NaN-only row, and the maximum at the first
and last index. Sizes span one CTA, many CTAs with a ragged last slice, the 151,936-entry vocabulary
and a row stride larger than the row.
"""
import numpy as np
import pytest

import oracle
import synth

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


def planted_logits(seed, m, n, ldl):
    full = synth.normal(seed, 7, (m, ldl), std=3.0)
    full[:, n:] = np.float32(1e38)  # beyond the row: must never be read as a candidate
    lg = full[:, :n]
    for r in range(m):
        kind = r % 8
        if kind == 1 and n > 3:  # a tie for the maximum: the lower index wins
            a, b = (r * 7919) % n, (r * 104729 + n // 2) % n
            lo, hi = min(a, b), max(a, b)
            if lo != hi:
                lg[r, lo] = lg[r, hi] = np.float32(50.0)
        elif kind == 2:  # maximum at the last index
            lg[r, n - 1] = np.float32(60.0)
        elif kind == 3:  # maximum at index 0
            lg[r, 0] = np.float32(60.0)
        elif kind == 4:  # NaNs everywhere but a few values
            lg[r, :] = np.nan
            lg[r, ::max(1, n // 5)] = -np.float32(2.0)
        elif kind == 5:  # a NaN-only row
            lg[r, :] = np.nan
        elif kind == 6:  # all values equal to zero of either sign
            lg[r, :] = 0.0
            lg[r, ::2] = -0.0
        elif kind == 7 and n > 2:  # infinities
            lg[r, n // 3] = np.inf
            lg[r, (2 * n) // 3] = np.inf
            lg[r, n - 1] = -np.inf
    return full


@pytest.mark.parametrize("m,n,pad", [(1, 1, 0), (3, 7, 1), (8, 2049, 3), (16, 4096, 0), (5, 20000, 4),
                                     (16, 151936, 0), (8, 151936, 16), (1, 248320, 0), (16, 1 << 20, 0)])
def test_greedy_matches_oracle(m, n, pad):
    full = planted_logits(900 + n + m, m, n, n + pad)
    want = oracle.greedy_tokens(full[:, :n])
    dev = torch.from_numpy(full).cuda()
    ws = bfp.greedy_workspace(m, n, dev.device)
    tok = bfp.greedy_tokens(dev[:, :n], ws)
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), want)
    # the same call again (workspace reused, no re-initialisation needed)
    tok2 = bfp.greedy_tokens(dev[:, :n], ws)
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2)


def test_greedy_rejects_bad_arguments():
    dev = torch.zeros((17, 64), dtype=torch.float32, device="cuda")
    ws = bfp.greedy_workspace(16, 64, dev.device)
    tok = torch.zeros(17, dtype=torch.int32, device="cuda")
    with pytest.raises(bfp.BFPError) as e:
        bfp.greedy_tokens(dev, ws, tok)  # 17 rows
    assert e.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as e:
        bfp.greedy_tokens(dev[:, :0], ws, tok)  # empty rows
    assert e.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as e:
        bfp.greedy_tokens(dev[:4], ws[:8], tok)  # workspace too small for 4 rows
    assert e.value.code == bfp.BFP_EWORKSPACE
    with pytest.raises(bfp.BFPError) as e:
        bfp.greedy_tokens(dev[:4, 1:], ws, tok)  # logits not 16-byte aligned
    assert e.value.code == bfp.BFP_EALIGN
