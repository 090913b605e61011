"""GPU parity of the BFP unpack and the dense BFP linear against the oracle (C-ABI calls)."""
import numpy as np
import pytest

import oracle
import synth
from harness import assert_close, bf16_tensor

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


def adversarial(w):
    n = w.shape[0]
    if n > 6:
        w[1, :] = 0.0
        w[2, :] = np.float32(1e-37) * np.sign(w[2, :])     # block exponents near the bottom: subnormal decodes
        w[3, :16] = [1.5, 1.25, 1.75, 0.625, -0.375, 1.9999999, -1.9999999, 0.0625] * 2  # ties, saturation
        w[4, :] *= np.float32(1e30)                          # large exponents
        w[5, ::17] = 0.0
    return w


@pytest.mark.parametrize("fmt", [4, 8])
@pytest.mark.parametrize("n,k", [(16, 64), (37, 96), (5, 208), (130, 2048), (512, 2048)])
def test_unpack_device_bit_exact(fmt, n, k):
    w = adversarial(synth.normal(21, 100 + n + k, (n, k), std=0.02))
    e, c = oracle.encode(fmt, w)
    ref = oracle.decode(fmt, e, c)
    mat = bfp.DeviceMatrix.from_host(fmt, n, k, bfp.encode(fmt, w))
    got = bfp.unpack_device(mat).cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


LINEAR_CASES = [
    (8, 8192, 2048, 1), (8, 8192, 2048, 8), (8, 8192, 2048, 16),   # dense BFP8 projection y[M x 8192] = x W^T
    (4, 512, 2048, 1), (4, 512, 2048, 16),
    (8, 37, 96, 3), (4, 37, 96, 9), (8, 130, 2048, 16), (4, 16, 16, 1), (8, 2000, 1024, 5),
    # up to 32 rows in one weight pass (four activation groups, fragments built in place)
    (8, 8192, 2048, 17), (8, 8192, 2048, 24), (8, 8192, 2048, 32), (4, 512, 2048, 32), (8, 37, 96, 29),
    (8, 130, 2048, 32), (4, 2000, 1024, 20),
    # k below the records' padded width (staged rows then take the padded width plus 8 elements)
    (8, 2000, 2000, 32), (4, 96, 1008, 31),
]


@pytest.mark.parametrize("fmt,n,k,m", LINEAR_CASES)
def test_linear_matches_oracle(fmt, n, k, m):
    w = adversarial(synth.normal(31, 200 + n + k, (n, k), std=0.02))
    if n > 6:
        w[2, :] = synth.normal(31, 9, (k,), std=0.02)  # keep rows' outputs in a normal range
        w[4, :] = synth.normal(31, 10, (k,), std=0.02)
    x = np.stack([synth.activation_row(31, 1000 + r, k, False) for r in range(m)])
    e, c = oracle.encode(fmt, w)
    y_ref, yb_ref = oracle.linear(fmt, e, c, x)
    mat = bfp.DeviceMatrix.from_host(fmt, n, k, bfp.encode(fmt, w))
    ws = bfp.linear_workspace(mat, m)
    xt = bf16_tensor(x)
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    yb = torch.empty((m, n), dtype=torch.int16, device="cuda")
    bfp.linear(mat, xt, ws, y=y, y_bf16=yb)
    got = y.cpu().numpy()
    gotb = yb.cpu().numpy().view(np.uint16)
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert_close(got, y_ref, f"linear fmt={fmt} {n}x{k} m={m}")
    assert np.array_equal(gotb, synth.to_bf16_bits(got))  # bf16 output is the RNE of the kernel's own fp32
    # and, away from cancellation (|y| >= rms/10), within one bf16 step of the oracle's bf16 output
    rms = np.sqrt(np.mean(y_ref.astype(np.float64) ** 2, axis=1, keepdims=True))
    big = np.abs(y_ref) >= 0.1 * rms
    diff = np.abs(gotb.astype(np.int32) - yb_ref.astype(np.int32))
    assert np.all(diff[big] <= 1)
    # repeated calls are bit-identical (fixed-order reduction, workspace left clean)
    y2 = bfp.linear(mat, xt, ws)
    assert torch.equal(y, y2)


def test_linear_rejects_bad_arguments():
    mat = bfp.DeviceMatrix.from_host(8, 64, 64, bfp.encode(8, synth.normal(1, 1, (64, 64), std=0.02)))
    ws = bfp.linear_workspace(mat, 1)
    x = torch.zeros((33, 64), dtype=torch.int16, device="cuda")
    with pytest.raises(bfp.BFPError) as ei:
        bfp.linear(mat, x, ws)
    assert ei.value.code == bfp.BFP_ESHAPE
    # more than 16 rows keeps every fragment in registers while they are built: k <= 2048
    wide = bfp.DeviceMatrix.from_host(8, 16, 2064, bfp.encode(8, synth.normal(1, 2, (16, 2064), std=0.02)))
    with pytest.raises(bfp.BFPError) as ei:
        bfp.linear_workspace(wide, 17)
    assert ei.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.linear(mat, x[:2], ws[:64])
    assert ei.value.code == bfp.BFP_EWORKSPACE


def greedy_of(y):
    """First index of each row's largest non-NaN value (-0 equal to +0), 0 for a row of NaN only."""
    out = []
    for row in np.asarray(y, dtype=np.float32):
        ok = ~np.isnan(row)
        out.append(int(np.flatnonzero(ok & (row == row[ok].max()))[0]) if ok.any() else 0)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("fmt,n,k,m", [(8, 8192, 2048, 1), (8, 8192, 2048, 16), (8, 8192, 2048, 32),
                                       (8, 151936, 2048, 8), (4, 37, 96, 9), (8, 2000, 1024, 5), (4, 16, 16, 1)])
def test_linear_greedy_token_in_the_epilogue(fmt, n, k, m):
    """bfp_linear_greedy: the projection's outputs are those of bfp_linear, and the tokens are the greedy
    rule applied to them (exact: comparisons only); away from near-ties (the two largest oracle outputs
    apart by more than the tolerance) they are also the oracle's arg max. Two rows of W are made equal
    and largest, so the lower index must win the tie."""
    w = synth.normal(41, 300 + n + k, (n, k), std=0.02)
    x = np.stack([synth.activation_row(41, 2000 + r, k, False) for r in range(m)])
    if n > 40:
        xf = synth.bf16_bits_to_f32(x[0])
        w[23] = np.float32(0.05) * np.sign(xf)  # a clear maximum for row 0 ...
        w[37] = w[23]                           # ... twice: ties go to the lower index
    mat = bfp.DeviceMatrix.from_host(fmt, n, k, bfp.encode(fmt, w))
    ws = bfp.linear_workspace(mat, m)
    xt = bf16_tensor(x)
    y_plain = bfp.linear(mat, xt, ws)
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    for call in range(2):  # the counter in the workspace is left at zero: a second call works the same
        tok = bfp.linear_greedy(mat, xt, ws, y=y)
        torch.cuda.synchronize()
        assert bfp.workspace_status(ws) == bfp.BFP_OK
        assert torch.equal(y, y_plain)
        assert np.array_equal(tok.cpu().numpy(), greedy_of(y.cpu().numpy())), f"call {call}"
    tok_only = bfp.linear_greedy(mat, xt, ws)  # no outputs written at all
    assert torch.equal(tok_only, tok)
    if n > 40:
        assert int(tok[0]) == 23
    e, c = oracle.encode(fmt, w)
    y_ref, _ = oracle.linear(fmt, e, c, x)
    for r in range(m):
        top2 = np.sort(y_ref[r].astype(np.float64))[-2:]
        rms = np.sqrt(np.mean(y_ref[r].astype(np.float64) ** 2))
        if top2[1] - top2[0] > 2e-3 * (abs(top2[1]) + rms):
            assert int(tok[r]) == int(np.argmax(y_ref[r]))


@pytest.mark.parametrize("path,fmt,n,k,m", [
    (2, 8, 8192, 2048, 1), (2, 8, 8192, 2048, 8), (2, 8, 8192, 2048, 16), (2, 4, 512, 2048, 8),
    (2, 8, 130, 2048, 5), (2, 4, 2000, 1024, 16), (2, 8, 8192, 2048, 17), (2, 8, 8192, 2048, 24),
    (2, 8, 8192, 2048, 32), (2, 4, 512, 2048, 32), (2, 8, 130, 2048, 32), (2, 4, 2000, 1024, 20),
    (1, 8, 8192, 2048, 24), (1, 8, 8192, 2048, 32), (1, 4, 512, 2048, 32),
])
def test_linear_each_kernel_matches_oracle(path, fmt, n, k, m):
    """Both kernels behind bfp_linear against the oracle: the tcgen05 one (path 2, asked for) and the mma.sync
    one (path 1, the default's)."""
    bfp.set_linear_path(path)
    try:
        test_linear_matches_oracle(fmt, n, k, m)
    finally:
        bfp.set_linear_path(0)


def test_linear_tcgen05_block_exponent_spread():
    """The tcgen05 kernel scales each 16-value block relative to the largest exponent among a row's 64 inputs
    of a chunk: blocks 2^14 apart within a chunk stay exact, blocks 2^40 apart lose only what lies below 2^-16
    of the chunk's largest value; checked against the oracle within the stated tolerance."""
    fmt, n, k, m = 8, 256, 2048, 32
    w = synth.normal(41, 7, (n, k), std=0.02)
    w[:, 0:16] *= np.float32(2.0 ** 14)   # block 0 of every chunk-0 row far above its neighbours
    w[:128, 64:80] *= np.float32(2.0 ** -40)  # a tiny block in chunk 1 of the first half of the rows
    x = np.stack([synth.activation_row(41, 2000 + r, k, False) for r in range(m)])
    e, c = oracle.encode(fmt, w)
    y_ref, _ = oracle.linear(fmt, e, c, x)
    mat = bfp.DeviceMatrix.from_host(fmt, n, k, bfp.encode(fmt, w))
    ws = bfp.linear_workspace(mat, m)
    bfp.set_linear_path(2)
    try:
        y = bfp.linear(mat, bf16_tensor(x), ws)
    finally:
        bfp.set_linear_path(0)
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert_close(y.cpu().numpy(), y_ref, "tcgen05 linear, spread block exponents")
