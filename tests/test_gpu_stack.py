"""GPU parity of the decode stack (moe_stack_decode) against the oracle.

Per layer: h <- bf16(h + MoE(bf16(RMSNorm(h)))); then logits = LMhead(bf16(RMSNorm(h))).
Rows are redrawn until the oracle's top-k margin is at least 1e-3 at every
layer of their trajectory (the same rule as for one layer).

A residual add rounds to bf16; where the kernel's fp32 sum and the oracle's
straddle a rounding boundary the two pick neighbouring bf16 values, and later
layers carry that difference on. So each part is checked where it is exact:
  * per layer, teacher-forced: from the oracle's bf16 h_l, the kernel's h_{l+1}
    is within half a bf16 step plus 1e-3 * (|y| + rms(y)) of h_l + y_oracle;
  * LM head, teacher-forced: logits within 1e-3 * (|oracle| + rms) of the
    oracle applied to the kernel's own final h;
  * end to end: final h within 1e-2 * (|h| + rms), logits within 1e-2 * (|l| + rms).
"""
import numpy as np
import pytest

import oracle
import synth
from harness import MARGIN, assert_close, bf16_tensor

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


class StackCase:
    def __init__(self, spec, n_layers, vocab, seed):
        self.spec, self.n_layers, self.vocab, self.seed = spec, n_layers, vocab, seed
        self.lw = [synth.LayerWeights(spec, seed, layer=l) for l in range(n_layers)]
        self.routers = [w.router_bf16() for w in self.lw]
        self.sgates = [w.shared_gate_bf16() for w in self.lw]
        self.caches = []
        for w in self.lw:
            def src(e, w=w):
                key = synth.SHARED_EXPERT if e == "shared" else e
                return w.gate(key), w.up(key), w.down(key)
            self.caches.append((src, oracle.ExpertCache(4, src)))

    def lm_rows(self, rows):
        """fp32 LM-head rows (any subset), each regenerated from its own offset of one stream."""
        out = np.empty((len(rows), self.spec.hidden), dtype=np.float32)
        for i, v in enumerate(rows):
            synth.normal(self.seed, synth.stream_id(synth.KIND_LMHEAD), self.spec.hidden, std=synth.W_STD,
                         offset=int(v) * self.spec.hidden, out=out[i])
        return out

    def layer_args(self, l):
        return dict(router_bf16=self.routers[l], shared_gate_bf16=self.sgates[l], experts=self.caches[l][1],
                    top_k=self.spec.top_k)

    def trajectory(self, h_row):
        """Oracle trajectory of one row: [(h_l, y_l, idx_l)] per layer and the final h; None if some layer's
        top-k margin is below MARGIN."""
        h = h_row[None, :].copy()
        steps = []
        for l in range(self.n_layers):
            t = oracle.rmsnorm_bf16(h)
            if oracle.topk_margin(oracle.router_logits(self.routers[l], t)[0], self.spec.top_k) < MARGIN:
                return None
            h_next, _, y, idx, _ = oracle.stack_layer(h, self.layer_args(l))
            steps.append((h[0], y[0], idx[0]))
            h = h_next
        return steps, h[0]

    def inputs(self, m, row_seed0):
        rows, trajs = [], []
        rs = row_seed0
        while len(rows) < m:
            x = synth.to_bf16_bits(synth.normal(self.seed, synth.stream_id(synth.KIND_STACK_H, 0, 0, 0, rs),
                                                (self.spec.hidden,), std=1.0))
            rs += 1
            tr = self.trajectory(x)
            if tr is not None:
                rows.append(x)
                trajs.append(tr)
        return np.stack(rows), trajs

    def device(self):
        s = self.spec
        layers = []
        for l in range(self.n_layers):
            src = self.caches[l][0]
            layers.append(bfp.MoELayer.from_source(s.hidden, s.n_experts, s.ffn, s.top_k, s.shared_ffn, bfp.BFP4,
                                                   self.routers[l], self.sgates[l], src, lambda src=src: src("shared")))
        lm = np.empty(bfp.packed_size(8, self.vocab, s.hidden), dtype=np.uint8)
        chunk = 4096
        w = np.empty((chunk, s.hidden), dtype=np.float32)
        for r0 in range(0, self.vocab, chunk):
            n = min(chunk, self.vocab - r0)
            synth.normal(self.seed, synth.stream_id(synth.KIND_LMHEAD), (n * s.hidden,), std=synth.W_STD,
                         offset=r0 * s.hidden, out=w[:n].reshape(-1))
            part = bfp.encode(8, w[:n])
            off = bfp.packed_size(8, r0, s.hidden) if r0 else 0
            lm[off:off + part.nbytes] = part
        return layers, bfp.DeviceMatrix.from_host(8, self.vocab, s.hidden, lm)


def bf16_half_step(v):
    """Half the distance to the next bf16 value above |v| (the RNE error bound of a bf16 result)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-38)))
    return 2.0 ** (e - 8)


def run_stack(case, m, row_seed0, sample_vocab=None):
    h0, trajs = case.inputs(m, row_seed0)
    h_ref = np.stack([t[1] for t in trajs])
    layers, lm = case.device()
    ws = bfp.moe_stack_workspace(layers, lm, m)
    vrows = np.arange(case.vocab) if sample_vocab is None else sample_vocab

    # per layer, teacher-forced: one-layer stacks from the oracle's bf16 input of that layer
    for l in range(case.n_layers):
        ws1 = bfp.moe_stack_workspace([layers[l]], lm, m)
        h_in = np.stack([t[0][l][0] for t in trajs])
        y_or = np.stack([t[0][l][1] for t in trajs]).astype(np.float64)
        h = bf16_tensor(h_in)
        idx1 = torch.full((m, case.spec.top_k), -1, dtype=torch.int32, device="cuda")
        bfp.moe_stack_decode([layers[l]], lm, h, ws1, topk_idx=idx1)
        torch.cuda.synchronize()
        assert bfp.workspace_status(ws1) == bfp.BFP_OK
        idx_or = np.stack([t[0][l][2] for t in trajs])
        assert np.array_equal(idx1.cpu().numpy(), idx_or), f"layer {l}: selection differs from the oracle's"
        got = synth.bf16_bits_to_f32(h.cpu().numpy().view(np.uint16)).astype(np.float64)
        exact = synth.bf16_bits_to_f32(h_in).astype(np.float64) + y_or
        rms_y = np.sqrt(np.mean(y_or ** 2, axis=1, keepdims=True))
        bound = bf16_half_step(exact) + 1e-3 * (np.abs(y_or) + rms_y)
        worst = float(np.max(np.abs(got - exact) / bound))
        assert worst <= 1.0, f"layer {l}: |h_gpu - (h + y_oracle)| / bound = {worst:.3f}"

    # the whole stack
    h = bf16_tensor(h0)
    k = case.spec.top_k
    idx_all = torch.full((case.n_layers, m, k), -1, dtype=torch.int32, device="cuda")
    logits = bfp.moe_stack_decode(layers, lm, h, ws, topk_idx=idx_all)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    ia = idx_all.cpu().numpy()
    # layer 0 sees the same input on both sides; every layer's selection is k distinct experts
    assert np.array_equal(ia[0], np.stack([t[0][0][2] for t in trajs]))
    assert ia.min() >= 0 and ia.max() < case.spec.n_experts
    assert all(len(set(ia[l, r])) == k for l in range(case.n_layers) for r in range(m))
    h_gpu = h.cpu().numpy().view(np.uint16)
    assert_close(synth.bf16_bits_to_f32(h_gpu), synth.bf16_bits_to_f32(h_ref), "final hidden state", tol=1e-2)
    lm_rows = case.lm_rows(vrows)
    got = logits.cpu().numpy()[:, vrows]
    assert_close(got, oracle.lm_head_rows(h_gpu, lm_rows), "LM head on the kernel's final h")
    assert_close(got, oracle.lm_head_rows(h_ref, lm_rows), "end-to-end logits", tol=1e-2)
    # greedy next token on the stack's logits: a property that holds at any vocabulary size
    gws = bfp.greedy_workspace(m, case.vocab, logits.device)
    tok = bfp.greedy_tokens(logits, gws).cpu().numpy()
    full = logits.cpu().numpy()
    for r in range(m):
        t = int(tok[r])
        assert np.all(full[r] <= full[r, t]) and np.all(full[r, :t] < full[r, t]), f"row {r}: token {t}"
    # a second run from the same h gives the same bits
    h2 = bf16_tensor(h0)
    logits2 = bfp.moe_stack_decode(layers, lm, h2, ws)
    torch.cuda.synchronize()
    assert torch.equal(logits, logits2) and torch.equal(h, h2)
    # the greedy variant: the same logits, and the next tokens taken in the LM head's epilogue are the greedy
    # rule on them; without logits it still gives the same tokens
    h3 = bf16_tensor(h0)
    lg3 = torch.empty_like(logits)
    tok3 = bfp.moe_stack_decode_greedy(layers, lm, h3, ws, logits=lg3)
    h4 = bf16_tensor(h0)
    tok4 = bfp.moe_stack_decode_greedy(layers, lm, h4, ws)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert torch.equal(lg3, logits) and torch.equal(h3, h)
    assert np.array_equal(tok3.cpu().numpy(), tok) and torch.equal(tok4, tok3)


def test_tiny_stack_m8():
    case = StackCase(synth.TINY, n_layers=4, vocab=1000, seed=801)
    run_stack(case, 8, 0)


def test_tiny_stack_m1_odd_layers():
    case = StackCase(synth.TINY, n_layers=3, vocab=1001, seed=802)
    run_stack(case, 1, 50)


@pytest.mark.slow
def test_full_size_stack_sampled_logits():
    """Three full-size layers (hidden 2048, 256 experts, top-8, shared expert) and the full BFP8 LM head
    [151936 x 2048], 8 rows; logits checked on 512 sampled vocabulary rows."""
    case = StackCase(synth.FULL, n_layers=3, vocab=151936, seed=803)
    rng = np.random.default_rng(5)
    run_stack(case, 8, 0, sample_vocab=np.sort(rng.choice(151936, 512, replace=False)))


@pytest.mark.parametrize("spec,n_layers,seed", [(synth.TINY, 50, 811), (synth.FULL, 3, 812)], ids=["tiny_50", "full_3"])
def test_one_row_stack_in_one_launch_matches_layer_by_layer(spec, n_layers, seed):
    """With one row the stack runs up to 48 layers in one launch, the residual row passing from layer to layer
    inside it (50 layers: two launches); one-layer stacks chained through global memory give the same bits:
    the final h, every layer's selection and the logits."""
    case = StackCase(spec, n_layers=n_layers, vocab=1000, seed=seed)
    layers, lm = case.device()
    h0 = synth.to_bf16_bits(synth.normal(seed, synth.stream_id(synth.KIND_STACK_H, 0, 0, 0, 0), (spec.hidden,),
                                         std=1.0))[None, :]
    k = spec.top_k
    ws = bfp.moe_stack_workspace(layers, lm, 1)
    h_a = bf16_tensor(h0)
    idx_a = torch.full((n_layers, 1, k), -1, dtype=torch.int32, device="cuda")
    lg_a = bfp.moe_stack_decode(layers, lm, h_a, ws, topk_idx=idx_a)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    h_b = bf16_tensor(h0)
    idx_b = torch.full((n_layers, 1, k), -1, dtype=torch.int32, device="cuda")
    ws1 = bfp.moe_stack_workspace([layers[0]], lm, 1)
    for l in range(n_layers):
        lg_b = bfp.moe_stack_decode([layers[l]], lm, h_b, ws1, topk_idx=idx_b[l])
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws1) == bfp.BFP_OK
    assert torch.equal(idx_a, idx_b)
    assert torch.equal(h_a, h_b)
    assert torch.equal(lg_a, lg_b)
    # the same stack again on the same workspace (the exchange words carry the next launch's epochs)
    h_c = bf16_tensor(h0)
    lg_c = bfp.moe_stack_decode(layers, lm, h_c, ws)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    assert torch.equal(h_c, h_a) and torch.equal(lg_c, lg_a)
