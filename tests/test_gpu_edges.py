"""Edge cases of the CUDA path against the oracle: the bench's own launch
configuration (a CUDA graph of back-to-back single-token calls, round-robin
over layer replicas, chained by programmatic dependent launch), empty and
oversized calls, the largest prefill call, and the degenerate selections
k = E (every expert) and k = 1, on the fused, batched and prefill paths."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import W_RTOL_TC, check_against_oracle, from_torch_bf16, make_gpu_layer, run, to_torch_bf16
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


def test_bench_configuration_graph_of_single_token_calls():
    """Page-scale layer, two replicas, 48 tokens captured as one CUDA graph of
    48 back-to-back calls and replayed twice: bit-identical to eager calls,
    sampled rows against the oracle."""
    import torch
    L = synth.make_layer(synth.PAGE, layer=0)
    n = 48
    x, _ = resampled_tokens(L, 7000, n)
    reps = [make_gpu_layer(L, max_tokens=1) for _ in range(2)]
    y_eager, idx_eager, w_eager = run(reps[0], x, T=1)
    xd = to_torch_bf16(x)
    yd = torch.empty_like(xd)
    idd = torch.empty((n, L.shape.k), dtype=torch.int32, device="cuda")
    wd = torch.empty((n, L.shape.k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for r in reps:
            r.forward(xd[0:1], yd[0:1])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(n):
            reps[t % 2].forward(xd[t:t + 1], yd[t:t + 1], idd[t:t + 1], wd[t:t + 1])
    for _ in range(2):
        yd.zero_()
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(from_torch_bf16(yd), y_eager)
        assert np.array_equal(idd.cpu().numpy(), idx_eager)
        assert np.array_equal(wd.cpu().numpy(), w_eager)
    check_against_oracle(L, x, from_torch_bf16(yd), idd.cpu().numpy(), wd.cpu().numpy(), rows=[0, 1, 23, 46, 47])
    for r in reps:
        stats, code = r.stats()
        assert code == 0
        r.close()


def test_empty_and_oversized_calls_are_rejected():
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    L = synth.make_layer(synth.SMALL, layer=0)
    g = make_gpu_layer(L, max_tokens=4)
    xd = torch.zeros((5, L.shape.H), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty_like(xd)
    for T in (0, 5):
        with pytest.raises(moe.MoeError) as ei:
            g.forward(xd[:T], yd[:T])
        assert ei.value.code == 1  # MOE_ERR_INVALID_ARG, nothing launched
    stats, code = g.stats()
    assert code == 0 and stats["forwards"] == 0
    g.close()


def test_largest_prefill_call():
    """T = 8192 (the largest call): routing of every token against the
    oracle's binary64 logits, sampled outputs element by element."""
    L = synth.make_layer(synth.SMALL, layer=3)
    sh = L.shape
    T = 8192
    x, _ = resampled_tokens(L, 90000, T)
    g = make_gpu_layer(L, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    logits = oracle.router_logits(L.W_r, L.bias, x)
    for t in range(T):
        ri, rw, _, _ = oracle.topk(logits[t], sh.k)
        assert np.array_equal(idx[t], ri), t
        assert np.allclose(w[t], rw, rtol=W_RTOL_TC, atol=1e-7), t
    check_against_oracle(L, x, y, idx, w, rows=np.r_[np.arange(0, T, 512), T - 1], w_rtol=W_RTOL_TC)
    g.close()


@pytest.mark.parametrize("k", [16, 1], ids=["k_eq_E", "k_1"])
@pytest.mark.parametrize("T", [1, 5, 40, 100], ids=["fused1", "fused5", "batched40", "prefill100"])
def test_degenerate_selections(k, T):
    """E = 16 experts with k = 16 (every expert selected, weights = softmax
    over all of them) and k = 1 (weight exactly 1)."""
    sh = synth.LayerShape(H=256, E=16, k=k, I=128)
    L = synth.make_layer(sh, layer=40 + k)
    x, _ = resampled_tokens(L, 500, T)
    g = make_gpu_layer(L, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(L, x, y, idx, w, w_rtol=W_RTOL_TC if T > 64 else 1e-5)
    if k == sh.E:
        assert np.array_equal(idx, np.tile(np.arange(sh.E, dtype=np.int32), (T, 1)))
    else:
        assert np.array_equal(w, np.ones((T, 1), np.float32))
    g.close()


@pytest.mark.parametrize("T", [1, 8])
def test_hidden_wider_than_one_down_strip_per_sm(T):
    """H = 4,096 has 256 down strips of 16 rows, more than the GPU has SMs:
    the fused kernel (one strip per CTA) declines and the batched kernels run,
    every output row against the oracle; a slot pool, which only the fused
    kernel serves, is refused when it is configured."""
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.LayerShape(H=4096, E=32, k=2, I=128)
    L = synth.make_layer(sh, layer=60)
    x, _ = resampled_tokens(L, 900, T)
    g = make_gpu_layer(L, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(L, x, y, idx, w)
    g.close()
    with pytest.raises(moe.MoeError) as e:
        make_gpu_layer(L, max_tokens=T, n_slots=2 * T)
    assert e.value.code == 2
