"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import check_against_oracle, make_gpu_layer, run, to_torch_bf16, from_torch_bf16
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def small():
    return synth.make_layer(synth.SMALL, layer=0)


@pytest.fixture(scope="module")
def page():
    return synth.make_layer(synth.PAGE, layer=0)


def test_small_layer_single_tokens(small):
    """64 experts top-4 + shared, H 1024, I 256: 16 tokens, one call each."""
    x, _ = resampled_tokens(small, 0, 16)
    g = make_gpu_layer(small, max_tokens=1)
    y, idx, w = run(g, x, T=1)
    check_against_oracle(small, x, y, idx, w)
    g.close()


@pytest.mark.parametrize("T", [2, 8, 13, 64])
def test_small_layer_batches_and_batch_invariance(small, T):
    x, _ = resampled_tokens(small, 100, 64)
    g1 = make_gpu_layer(small, max_tokens=1)
    y1, i1, w1 = run(g1, x, T=1)
    g = make_gpu_layer(small, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(small, x, y, idx, w, rows=np.arange(0, 64, 4))
    # a token's output does not depend on the batch it was computed in
    assert np.array_equal(y, y1) and np.array_equal(idx, i1) and np.array_equal(w, w1)
    g.close()
    g1.close()


def test_page_layer_single_tokens(page):
    """512 experts top-10 + shared, H 2048, I 512, Zipf-biased router."""
    x, _ = resampled_tokens(page, 0, 16)
    g = make_gpu_layer(page, max_tokens=1)
    y, idx, w = run(g, x, T=1)
    check_against_oracle(page, x, y, idx, w)
    g.close()


@pytest.mark.parametrize("T", [8, 64])
def test_page_layer_batches(page, T):
    x, _ = resampled_tokens(page, 1000, T)
    g = make_gpu_layer(page, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(page, x, y, idx, w, rows=np.arange(0, T, max(1, T // 8)))
    g1 = make_gpu_layer(page, max_tokens=1)
    y1, i1, _ = run(g1, x, T=1)
    assert np.array_equal(y, y1) and np.array_equal(idx, i1)
    g.close()
    g1.close()


def test_full_nibble_range_and_no_shared_expert():
    """Random nibbles (every q in -8..7) and random scales; also a layer
    without a shared expert."""
    sh = synth.LayerShape(H=512, E=16, k=3, I=192)
    L = synth.make_layer(sh, layer=77)
    rng = np.random.default_rng(9)
    mb = sh.matrix_bytes
    ex = L.experts.reshape(sh.E, -1)
    for m in range(3):
        R, K = (sh.I, sh.H) if m < 2 else (sh.H, sh.I)
        ex[:, m * mb:m * mb + R * K // 2] = rng.integers(0, 256, size=(sh.E, R * K // 2), dtype=np.uint8)
        # scales chosen so outputs stay in the range of the Gaussian layers
        # (|y| < 2), where the absolute bound is meaningful next to bf16 rounding
        sc = (np.abs(rng.normal(size=(sh.E, R * K // 32))) * 0.004).astype(np.float16)
        ex[:, m * mb + R * K // 2:(m + 1) * mb] = sc.view(np.uint8).reshape(sh.E, -1)
    x, _ = resampled_tokens(L, 0, 8)
    g = make_gpu_layer(L, max_tokens=8)
    y, idx, w = run(g, x, T=8)
    check_against_oracle(L, x, y, idx, w)
    g.close()
    L0 = synth.Layer(sh, 77, L.W_r, L.bias, L.experts, None)
    g0 = make_gpu_layer(L0, max_tokens=4, with_shared=False)
    y, idx, w = run(g0, x, T=4)
    check_against_oracle(L0, x, y, idx, w)
    g0.close()


def test_cuda_graph_replay_matches_eager(small):
    import torch
    x, _ = resampled_tokens(small, 300, 8)
    g = make_gpu_layer(small, max_tokens=1)
    y_ref, _, _ = run(g, x, T=1)
    xd = to_torch_bf16(x)
    yd = torch.empty_like(xd)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.forward(xd[0:1], yd[0:1])  # warm
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(8):
            g.forward(xd[t:t + 1], yd[t:t + 1])
    yd.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(from_torch_bf16(yd), y_ref)
    g.close()


def test_residual_rmsnorm_against_oracle():
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.PAGE
    x = synth.activations(sh, 5, 0, 16)
    yv = synth.activations(sh, 6, 0, 16)
    xd, yd = to_torch_bf16(x), to_torch_bf16(yv)
    xo, xh = torch.empty_like(xd), torch.empty_like(xd)
    moe.residual_rmsnorm(xd, yd, 1e-6, xo, xh)
    torch.cuda.synchronize()
    xo, xh = from_torch_bf16(xo), from_torch_bf16(xh)
    ulp_off = 0
    for t in range(16):
        ro = oracle.residual(x[t], yv[t])
        assert np.array_equal(xo[t], ro)  # exact: one rounding of an exact sum
        rh, rf = oracle.rmsnorm(ro, 1e-6)
        d = np.abs(xh[t].astype(np.int64) - rh.astype(np.int64))
        assert d.max() <= 1
        ulp_off += int((d > 0).sum())
    assert ulp_off <= 16 * 2048 * 1e-3  # only values next to a rounding tie may differ


def test_residual_rmsnorm_in_place_and_misaligned():
    """x_out may alias x (each thread reads its chunks before it writes them);
    a pointer off a 16-byte boundary is refused before any launch."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.PAGE
    x = synth.activations(sh, 7, 0, 4)
    yv = synth.activations(sh, 8, 0, 4)
    xd, yd = to_torch_bf16(x), to_torch_bf16(yv)
    xh = torch.empty_like(xd)
    moe.residual_rmsnorm(xd, yd, 1e-6, xd, xh)  # in place
    torch.cuda.synchronize()
    got = from_torch_bf16(xd)
    for t in range(4):
        assert np.array_equal(got[t], oracle.residual(x[t], yv[t]))
    buf = torch.empty(4 * 2048 + 8, dtype=torch.bfloat16, device="cuda")
    off = buf[1:1 + 4 * 2048].view(4, 2048)  # 2 bytes past a 16-byte boundary
    with pytest.raises(moe.MoeError) as e:
        moe.residual_rmsnorm(off, None, 1e-6, None, xh)
    assert e.value.code == 1


def test_activation_out_of_fp16_range_is_reported(small):
    from quantized_expert_ffn_gemv_gb300 import moe
    x, _ = resampled_tokens(small, 0, 1)
    x = x.copy()
    x[0, 5] = synth.f32_to_bf16(np.array([1e6], np.float32))[0]
    g = make_gpu_layer(small, max_tokens=1)
    run(g, x, T=1)
    stats, code = g.stats()
    assert code == 8 and stats["error"] == 8
    with pytest.raises(moe.MoeError):
        run(g, x, T=1)
    g.close()
