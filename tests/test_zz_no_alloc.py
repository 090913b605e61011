"""moe_decode_layer_static: the MoE decode layer for callers that cannot allocate.

Some callers cannot call cudaMalloc: code embedded in a host runtime that owns
all device memory through its own allocator, or a latency-critical path where
an allocation could synchronise the device. moe_decode_layer_static takes no
workspace and uses the library's built-in 2 MiB device scratch array instead.
This test calls it through the C-ABI and checks its outputs against the
workspace entry point (moe_decode_layer) and against the oracle, on two calls
in a row, within the tolerance the other GPU tests use (16 rows and 1 row:
the general kernel and the one-row kernel). It lives in a file that pytest collects
last, and it is self-contained so it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import synth
from harness import LayerCase, assert_close, bf16_tensor

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("spec,m,seed", [(synth.TINY, 3, 611), (synth.FULL, 16, 612), (synth.FULL, 1, 613)])
def test_static_scratch_layer_matches_workspace_layer(spec, m, seed):
    import block_floating_point_gb300 as bfp
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    lib = bfp.load()
    case = LayerCase(spec, seed=seed)
    layer = case.device_layer()
    x, _ = case.inputs(m, rms_normalise=spec is synth.FULL)
    xt = bf16_tensor(x)
    ws = bfp.moe_workspace(layer, m)
    y_ref = bfp.moe_decode_layer(layer, xt, ws)
    idx_ref = torch.empty((m, spec.top_k), dtype=torch.int32, device="cuda")
    bfp.moe_decode_layer(layer, xt, ws, topk_idx=idx_ref)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    c = layer.c()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share the built-in scratch
        y = torch.full((m, spec.hidden), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.full((m, spec.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.empty((m, spec.top_k), dtype=torch.float32, device="cuda")
        rc = lib.moe_decode_layer_static(c, xt.data_ptr(), m, y.data_ptr(), idx.data_ptr(), w.data_ptr(), stream)
        assert rc == bfp.BFP_OK, lib.bfp_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), f"call {call}: expert selection differs"
        assert_close(y.cpu().numpy(), y_ref.cpu().numpy(), f"call {call}: static-scratch layer output")
        # and directly against the oracle (the tolerance of every other layer test)
        y_or, idx_or, _ = case.oracle_layer(x)
        assert np.array_equal(idx.cpu().numpy(), idx_or), f"call {call}: selection differs from the oracle's"
        assert_close(y.cpu().numpy(), y_or, f"call {call}: static-scratch layer against the oracle")


def test_static_scratch_rejects_layers_beyond_its_size():
    import block_floating_point_gb300 as bfp
    lib = bfp.load()
    # hidden 2048, ffn 1024, 16 rows: fits in shared memory but needs about 2.18 MB of scratch (> 2 MiB);
    # the size check comes before anything touches the (placeholder) pointers
    h, f = 2048, 1024
    c = bfp.MoeLayerC(h, 256, f, 8, f, bfp.BFP4, 16, None, 16, 16, 16,
                      bfp.packed_size(4, 2 * f, h), bfp.packed_size(4, h, f), 16, 16)
    rc = lib.moe_decode_layer_static(c, 16, 16, 16, None, None, None)
    assert rc == bfp.BFP_EWORKSPACE
    assert b"built-in scratch" in lib.bfp_last_error()
