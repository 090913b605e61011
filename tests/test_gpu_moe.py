"""GPU parity of the fused MoE decode layer against the oracle (C-ABI calls).

Expert selection (top-k indices, slot order) must match bit for bit; routing
weights and outputs within 1e-3 * (|oracle| + rms(oracle)). Inputs are redrawn
per row until the k-th / (k+1)-th router-logit gap is at least 1e-3.
"""
import numpy as np
import pytest

import synth
from harness import LayerCase, assert_close, bf16_tensor

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


def run_layer(layer, x, m):
    ws = bfp.moe_workspace(layer, m)
    xt = bf16_tensor(x)
    idx = torch.empty((m, layer.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((m, layer.top_k), dtype=torch.float32, device="cuda")
    y = bfp.moe_decode_layer(layer, xt, ws, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    return y, idx, w, ws, xt


def check(case, layer, m, rms_norm, row_seed0=0):
    x, _ = case.inputs(m, rms_norm, row_seed0)
    y, idx, w, ws, xt = run_layer(layer, x, m)
    y_ref, idx_ref, w_ref = case.oracle_layer(x)
    assert np.array_equal(idx.cpu().numpy(), idx_ref), "expert selection differs"
    assert_close(w.cpu().numpy(), w_ref, "routing weights")
    assert_close(y.cpu().numpy(), y_ref, "layer output")
    # a second launch on the same workspace gives the same bits (self-cleaning counters, fixed-order combine)
    idx2 = torch.empty_like(idx)
    y2 = bfp.moe_decode_layer(layer, xt, ws, topk_idx=idx2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(idx, idx2)
    return x


@pytest.fixture(scope="module")
def tiny():
    case = LayerCase(synth.TINY, seed=101)
    return case, case.device_layer()


@pytest.fixture(scope="module")
def full():
    case = LayerCase(synth.FULL, seed=202)
    return case, case.device_layer()


@pytest.mark.parametrize("m", [1, 2, 5, 16])
def test_tiny_layer(tiny, m):
    case, layer = tiny
    check(case, layer, m, rms_norm=False, row_seed0=10 * m)


def test_cooperative_launch_mode(tiny):
    """The layer launched cooperatively (for GPUs shared with other work) gives the same bits as the
    default dependent launch."""
    case, layer = tiny
    x, _ = case.inputs(4, False, 77)
    y0 = run_layer(layer, x, 4)[0]
    bfp.set_launch_mode(bfp.LAUNCH_COOPERATIVE)
    try:
        y1 = run_layer(layer, x, 4)[0]
    finally:
        bfp.set_launch_mode(bfp.LAUNCH_DEPENDENT)
    assert torch.equal(y0, y1)
    assert_close(y1.cpu().numpy(), case.oracle_layer(x)[0], "cooperative launch")


def test_tiny_layer_bfp8_experts():
    case = LayerCase(synth.TINY, seed=103, fmt=8)
    check(case, case.device_layer(), 3, rms_norm=False)


def test_full_layer_m1(full):
    case, layer = full
    check(case, layer, 1, rms_norm=True, row_seed0=0)


def test_full_layer_m16(full):
    case, layer = full
    check(case, layer, 16, rms_norm=True, row_seed0=100)


def test_full_layer_m8(full):
    case, layer = full
    check(case, layer, 8, rms_norm=True, row_seed0=300)


def test_contiguous_runs_one_activation_group():
    """Hidden 2048, 64 experts of width 1024, 8 rows: one activation group with at least 16 f-tile
    units per CTA, so phase 1 cuts each CTA's unit list into contiguous runs per warp (units split
    between neighbouring warps), and each down row group spans two chunks."""
    spec = synth.MoESpec(hidden=2048, n_experts=64, ffn=1024, top_k=8, shared_ffn=1024)
    case = LayerCase(spec, seed=414)
    check(case, case.device_layer(), 8, rms_norm=True, row_seed0=700)


def test_full_layer_hot_routing_m16():
    case = LayerCase(synth.FULL, seed=303, hot=True)
    layer = case.device_layer()
    x = check(case, layer, 16, rms_norm=True, row_seed0=500)
    # the bias concentrates the rows: far fewer distinct experts than random routing (~102 of 256
    # for 16 rows x top-8), and the 8 hot experts take a large share of the picks
    idx = case.oracle_layer(x)[1]
    hot = np.flatnonzero(case.bias)
    assert len(np.unique(idx)) < 80
    assert np.isin(idx, hot).mean() > 0.3


def test_odd_shapes():
    spec = synth.MoESpec(hidden=208, n_experts=37, ffn=48, top_k=3, shared_ffn=80)
    case = LayerCase(spec, seed=404)
    check(case, case.device_layer(), 7, rms_norm=False)


def test_bounded_wait_reports_timeout_and_recovers(tiny):
    """A cross-block wait that cannot be satisfied in one poll gives BFP_ETIMEOUT, not a hang;
    after re-initialising the workspace the layer runs correctly again."""
    case, layer = tiny
    x, _ = case.inputs(4, False, 900)
    ws = bfp.moe_workspace(layer, 4)
    xt = bf16_tensor(x)
    bfp.set_wait_limit(1)
    try:
        seen = set()
        for _ in range(5):
            bfp.moe_decode_layer(layer, xt, ws)
            seen.add(bfp.workspace_status(ws))
    finally:
        bfp.set_wait_limit(0)
    assert bfp.BFP_ETIMEOUT in seen
    bfp.workspace_init(ws)
    y = bfp.moe_decode_layer(layer, xt, ws)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert_close(y.cpu().numpy(), case.oracle_layer(x)[0], "after recovery")


def test_rejects_bad_arguments(tiny):
    case, layer = tiny
    ws = bfp.moe_workspace(layer, 1)
    x = torch.zeros((17, case.spec.hidden), dtype=torch.int16, device="cuda")
    with pytest.raises(bfp.BFPError) as ei:
        bfp.moe_decode_layer(layer, x, ws)
    assert ei.value.code == bfp.BFP_ESHAPE
    with pytest.raises(bfp.BFPError) as ei:
        bfp.moe_decode_layer(layer, x[:1], ws[:256])
    assert ei.value.code == bfp.BFP_EWORKSPACE


# ---------------------------------------------------------------- the one-row kernel (m = 1)
ROW_CASES = {
    "tiny": (synth.TINY, 121, 4, False),
    "tiny_bfp8_experts": (synth.TINY, 123, 8, False),
    "odd_shapes": (synth.MoESpec(hidden=208, n_experts=37, ffn=48, top_k=3, shared_ffn=80), 405, 4, False),
    "full": (synth.FULL, 222, 4, False),
    "full_hot_routing": (synth.FULL, 304, 4, True),
    # 64 experts of width 1024: a CTA's share exceeds shared memory, so the general kernel runs it
    "wide_experts": (synth.MoESpec(hidden=2048, n_experts=64, ffn=1024, top_k=8, shared_ffn=1024), 415, 4, False),
}


@pytest.mark.parametrize("name", list(ROW_CASES))
def test_one_row_kernel_against_oracle_and_general_kernel(name):
    """m = 1 runs on the one-row kernel (every CTA's share fixed at launch, each CTA summing whole output
    row groups): selection bit-exact and outputs within tolerance of the oracle, and the general kernel
    (bfp_set_row_path(0)) selects the same experts on the same row."""
    spec, seed, fmt, hot = ROW_CASES[name]
    case = LayerCase(spec, seed=seed, hot=hot, fmt=fmt)
    layer = case.device_layer()
    full = spec.hidden == 2048
    for row_seed0 in (0, 40):
        x = check(case, layer, 1, rms_norm=full, row_seed0=row_seed0)
        bfp.set_row_path(False)
        try:
            y_g, idx_g, w_g, _, _ = run_layer(layer, x, 1)
        finally:
            bfp.set_row_path(True)
        y_ref, idx_ref, w_ref = case.oracle_layer(x)
        assert np.array_equal(idx_g.cpu().numpy(), idx_ref)
        assert_close(y_g.cpu().numpy(), y_ref, "general kernel, one row")


def test_one_row_and_general_kernels_share_a_workspace(full):
    """The one-row and the general kernel keep separate counters in the workspace: calls with m = 1 and
    m = 16 alternating on one workspace stay correct."""
    case, layer = full
    x16, _ = case.inputs(16, True, 1300)
    x1 = x16[:1]
    ws = bfp.moe_workspace(layer, 16)
    y16_ref, y1_ref = case.oracle_layer(x16)[0], case.oracle_layer(x1)[0]
    for _ in range(2):
        y1 = bfp.moe_decode_layer(layer, bf16_tensor(x1), ws)
        y16 = bfp.moe_decode_layer(layer, bf16_tensor(x16), ws)
        torch.cuda.synchronize()
        assert bfp.workspace_status(ws) == bfp.BFP_OK
        assert_close(y1.cpu().numpy(), y1_ref, "m = 1 between m = 16 calls")
        assert_close(y16.cpu().numpy(), y16_ref, "m = 16 between m = 1 calls")


def test_one_row_bounded_wait_reports_timeout_and_recovers(tiny):
    case, layer = tiny
    x, _ = case.inputs(1, False, 950)
    ws = bfp.moe_workspace(layer, 1)
    xt = bf16_tensor(x)
    bfp.set_wait_limit(1)
    try:
        seen = set()
        for _ in range(5):
            bfp.moe_decode_layer(layer, xt, ws)
            seen.add(bfp.workspace_status(ws))
    finally:
        bfp.set_wait_limit(0)
    assert bfp.BFP_ETIMEOUT in seen
    bfp.workspace_init(ws)
    y = bfp.moe_decode_layer(layer, xt, ws)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert_close(y.cpu().numpy(), case.oracle_layer(x)[0], "one row, after recovery")


# ---------------------------------------------------------------- the benchmark's 40-layer decode stack
STACK_SEED = 20261202  # bench.py's default seed; its layer l is LayerWeights(FULL, STACK_SEED, layer=l)


@pytest.mark.parametrize("layer", [0, 17, 39])
def test_layers_of_the_benchmarked_stack(layer):
    """Three of the 40 independently seeded full-size layers the benchmark's decode stack runs, each on
    RMS-normalised bf16 rows (the input the stack feeds a layer), 8 rows (general kernel) and 1 row
    (one-row kernel): selection bit-exact, outputs within tolerance of the oracle."""
    case = LayerCase(synth.FULL, seed=STACK_SEED, layer=layer)
    dl = case.device_layer()
    check(case, dl, 8, rms_norm=True, row_seed0=3000 + 100 * layer)
    check(case, dl, 1, rms_norm=True, row_seed0=5000 + 100 * layer)


# ---------------------------------------------------------------- error-compensated (GPTQ-style) experts
def test_gptq_encoded_layer_matches_oracle():
    """A layer whose experts the library encoded with error compensation (bfp_encode_gate_up_gptq,
    bfp_encode_gptq) against the oracle's layer on the oracle's own gptq_encode fields of the same fp32
    weights and calibration inputs: selection bit-exact, outputs within tolerance, 1 and 6 rows."""
    import oracle
    spec = synth.MoESpec(hidden=512, n_experts=32, ffn=128, top_k=4, shared_ffn=128)
    lw = synth.LayerWeights(spec, 515)

    def calib(seed, t, k):  # correlated synthetic calibration inputs (the recipe of the host GPTQ tests)
        z = synth.normal(seed, 1, (t, k)).astype(np.float64)
        a = np.eye(k) + 3.0 * synth.normal(seed, 2, (k, k)).astype(np.float64) / np.sqrt(k)
        return ((z @ a) * np.exp(0.5 * synth.normal(seed, 3, (k,)).astype(np.float64))).astype(np.float32)

    x_cal, h_cal = calib(516, 2048, spec.hidden), calib(517, 1024, spec.ffn)
    u_in, u_mid = bfp.gptq_factor(x_cal), bfp.gptq_factor(h_cal)
    uo_in, uo_mid = oracle.gptq_factor(x_cal), oracle.gptq_factor(h_cal)

    def source(e):
        key = synth.SHARED_EXPERT if e == "shared" else e
        return lw.gate(key), lw.up(key), lw.down(key)

    class GptqExpert(oracle.EncodedExpert):  # the oracle's expert evaluation on its own GPTQ fields
        def __init__(self, fmt, g, u, d):
            self.fmt, (self.ffn, self.hidden) = fmt, g.shape
            self.g, self.u = oracle.gptq_encode(fmt, g, uo_in), oracle.gptq_encode(fmt, u, uo_in)
            self.d = oracle.gptq_encode(fmt, d, uo_mid)

    class GptqCache(oracle.ExpertCache):
        def __call__(self, e):
            if e not in self._c:
                self._c[e] = GptqExpert(self.fmt, *self.source(e))
            return self._c[e]

    router, sgate = lw.router_bf16(), lw.shared_gate_bf16()
    layer = bfp.MoELayer.from_source(spec.hidden, spec.n_experts, spec.ffn, spec.top_k, spec.shared_ffn, bfp.BFP4,
                                     router, sgate, source, lambda: source("shared"),
                                     gptq_factors=lambda e: (u_in, u_mid), shared_gptq_factors=lambda: (u_in, u_mid))
    plain = bfp.MoELayer.from_source(spec.hidden, spec.n_experts, spec.ffn, spec.top_k, spec.shared_ffn, bfp.BFP4,
                                     router, sgate, source, lambda: source("shared"))
    assert not torch.equal(layer.experts_gate_up, plain.experts_gate_up)  # compensation changed the codes
    experts = GptqCache(bfp.BFP4, source)
    for m, rs in ((1, 0), (6, 10)):
        rows = []
        while len(rows) < m:
            x = synth.activation_row(515, rs, spec.hidden, True)
            rs += 1
            if oracle.topk_margin(oracle.router_logits(router, x[None])[0], spec.top_k) >= 1e-3:
                rows.append(x)
        x = np.stack(rows)
        y, idx, w, _, _ = run_layer(layer, x, m)
        y_ref, idx_ref, w_ref = oracle.moe_layer(x, router, sgate, experts, spec.top_k)
        assert np.array_equal(idx.cpu().numpy(), idx_ref)
        assert_close(w.cpu().numpy(), w_ref, "routing weights")
        assert_close(y.cpu().numpy(), y_ref, f"GPTQ-encoded layer, {m} rows")
