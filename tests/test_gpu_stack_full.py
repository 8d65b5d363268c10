"""The 48-layer page-scale stack at full size, as the stack benchmark runs
it: every layer's slot pool capped at 128 of 512 experts (25 %), misses
from pinned host RAM, residual + RMSNorm between layers.  128 tokens (64
warm-up + 64) through the pooled stack must be bit-identical to the
all-resident stack; every layer's misses equal the LRU simulator's; sampled
(token, layer) points match the oracle on the GPU's own normalised input."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import MAX_ABS, REL_L2, W_RTOL, from_torch_bf16, to_torch_bf16

pytestmark = pytest.mark.gpu

N_LAYERS, N_TOKENS, SLOTS = 48, 128, 128
SAMPLES = [(0, 0), (5, 47), (64, 13), (90, 30), (127, 47), (127, 1)]  # (token, layer)
# Inner-layer inputs are not drawn, so nothing keeps their k-th/(k+1)-th
# logits apart; the compensated router resolves every gap down to about
# 1e-13 (bound 5e-10), so only a gap below 1e-9 may resolve differently.
NEAR_TIE = 1e-9


def _run(stack, x):
    import torch
    n = len(stack.layers)
    bufs = stack.buffers(1, record=True)
    xd = to_torch_bf16(x)
    out, idx, keep, xh = [], [], {}, []
    for t in range(x.shape[0]):
        xo = stack.forward(xd[t:t + 1], bufs)
        torch.cuda.synchronize()
        out.append(from_torch_bf16(xo.reshape(1, -1))[0])
        idx.append(bufs["idx"].reshape(n, -1).cpu().numpy())
        xh.append(from_torch_bf16(bufs["xhats"].reshape(n, -1)))
        for (ts, ls) in SAMPLES:
            if ts == t:
                keep[(ts, ls)] = (from_torch_bf16(bufs["xhats"][ls].reshape(1, -1)),
                                  from_torch_bf16(bufs["ys"][ls].reshape(1, -1)),
                                  bufs["w"][ls].reshape(-1).cpu().numpy())
    return np.stack(out), np.stack(idx), keep, np.stack(xh)


def test_full_stack_pool_is_bit_identical_and_matches_lru_and_oracle():
    from quantized_expert_ffn_gemv_gb300 import moe
    from quantized_expert_ffn_gemv_gb300.stack import MoeStack
    sampled = {ls for _, ls in SAMPLES}
    layers, kept, routers = [], {}, []
    for l in range(N_LAYERS):
        L = synth.make_layer(synth.PAGE, layer=l)
        layers.append(moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=1))
        routers.append((L.W_r, L.bias))
        if l in sampled:
            kept[l] = L
        del L

    class _Stack(MoeStack):
        def __init__(self, objs):
            self.layers, self.eps, self.H, self.k = objs, 1e-6, synth.PAGE.H, synth.PAGE.k
            import torch
            self.device = torch.device("cuda", 0)

    st = _Stack(layers)
    x = synth.activations(synth.PAGE, 1000, 0, N_TOKENS, stream=9)
    y_res, idx_res, _, _ = _run(st, x)
    for layer in st.layers:
        layer.configure(SLOTS)
    y_pool, idx_pool, keep, xhats = _run(st, x)
    assert np.array_equal(y_res, y_pool)
    assert np.array_equal(idx_res, idx_pool)
    for l, layer in enumerate(st.layers):
        steps = [sorted(idx_pool[t, l].tolist()) for t in range(N_TOKENS)]
        expect, _ = oracle.pool_sim(synth.PAGE.E, SLOTS, steps)
        log = layer.miss_log()
        log[:, 0] -= N_TOKENS  # steps count from the layer's creation: the resident run came first
        assert np.array_equal(log, expect), l
        stats, code = layer.stats()
        assert code == 0 and stats["misses"] == len(expect)
    sh = synth.PAGE
    # routing of every (token, layer) against the oracle on the GPU's own
    # normalised input: exact wherever the oracle's gap is at least 1e-9
    forced, min_gap = [], np.inf
    for l, (W_r, bias) in enumerate(routers):
        logits = oracle.router_logits(W_r, bias, xhats[:, l])
        for t in range(N_TOKENS):
            ri, _, _, gap = oracle.topk(logits[t], sh.k)
            min_gap = min(min_gap, gap)
            if not np.array_equal(idx_pool[t, l], ri):
                assert gap < NEAR_TIE, (t, l, gap)
                forced.append((t, l, gap))
    print(f"{N_TOKENS * N_LAYERS} (token, layer) selections against the oracle: smallest gap {min_gap:.3e}, "
          f"{len(forced)} decided inside a gap below {NEAR_TIE:g}: {forced}")
    for (t, l), (xh, yg, wg) in keep.items():
        L = kept[l]
        ref = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, xh)
        if not np.array_equal(idx_pool[t, l], ref["idx"][0]):
            assert ref["gap"][0] < NEAR_TIE, (t, l)
            ref = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, xh,
                                     force=idx_pool[t, l].reshape(1, -1))
        assert np.array_equal(idx_pool[t, l], ref["idx"][0]), (t, l)
        assert np.allclose(wg, ref["w"][0], rtol=W_RTOL, atol=1e-7), (t, l)
        yv = synth.bf16_to_f32(yg[0]).astype(np.float64)
        err = yv - ref["y"][0]
        assert np.linalg.norm(err) / np.linalg.norm(ref["y"][0]) <= REL_L2, (t, l)
        assert np.abs(err).max() <= MAX_ABS, (t, l)
    for layer in st.layers:
        layer.close()
