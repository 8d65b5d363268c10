"""Prefill path (T > 64: grouped GEMMs on the tensor cores) vs the CPU oracle."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import W_RTOL_TC, check_against_oracle, make_gpu_layer, run
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def small():
    return synth.make_layer(synth.SMALL, layer=0)


@pytest.mark.parametrize("T", [65, 200, 333])
def test_small_prefill_every_token(small, T):
    """64 experts top-4 + shared: several 128-token chunks and ragged tails."""
    x, _ = resampled_tokens(small, 2000, T)
    g = make_gpu_layer(small, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(small, x, y, idx, w, w_rtol=W_RTOL_TC)
    st, code = g.stats()
    assert code == 0 and st["forwards"] == 1
    assert st["hits"] == len(np.unique(idx))
    g.close()


def test_prefill_hot_and_cold_experts():
    """One expert every token selects (3 chunks of 128 at T = 300, the last
    ragged) and experts nobody selects (empty groups)."""
    sh = synth.SMALL
    L = synth.make_layer(sh, layer=5)
    bias = np.zeros(sh.E, np.float32)
    bias[7] = 50.0           # always selected
    bias[40:48] = -50.0      # never selected
    L = synth.Layer(sh, 5, L.W_r, bias, L.experts, L.shared)
    x, _ = resampled_tokens(L, 0, 300)
    g = make_gpu_layer(L, max_tokens=300)
    y, idx, w = run(g, x, T=300)
    assert np.all((idx == 7).any(axis=1))
    assert not np.isin(idx, np.arange(40, 48)).any()
    check_against_oracle(L, x, y, idx, w, w_rtol=W_RTOL_TC)
    g.close()


def test_prefill_full_nibble_range_without_shared_expert():
    """Every q in -8..7 with random scales; a layer with no shared expert."""
    sh = synth.LayerShape(H=512, E=16, k=3, I=192)
    L = synth.make_layer(sh, layer=78)
    rng = np.random.default_rng(10)
    mb = sh.matrix_bytes
    ex = L.experts.reshape(sh.E, -1)
    for m in range(3):
        R, K = (sh.I, sh.H) if m < 2 else (sh.H, sh.I)
        ex[:, m * mb:m * mb + R * K // 2] = rng.integers(0, 256, size=(sh.E, R * K // 2), dtype=np.uint8)
        sc = (np.abs(rng.normal(size=(sh.E, R * K // 32))) * 0.004).astype(np.float16)
        ex[:, m * mb + R * K // 2:(m + 1) * mb] = sc.view(np.uint8).reshape(sh.E, -1)
    L0 = synth.Layer(sh, 78, L.W_r, L.bias, L.experts, None)
    x, _ = resampled_tokens(L0, 0, 150)
    g = make_gpu_layer(L0, max_tokens=150, with_shared=False)
    y, idx, w = run(g, x, T=150)
    check_against_oracle(L0, x, y, idx, w, w_rtol=W_RTOL_TC)
    g.close()


def test_prefill_is_deterministic_and_layer_serves_all_paths(small):
    """Two prefill calls give identical bytes; the same layer object also runs
    decode (T = 1) and batched (T = 64) calls, which match the oracle."""
    x, _ = resampled_tokens(small, 3000, 256)
    g = make_gpu_layer(small, max_tokens=256)
    y1, i1, w1 = run(g, x, T=256)
    y2, i2, w2 = run(g, x, T=256)
    assert np.array_equal(y1, y2) and np.array_equal(i1, i2) and np.array_equal(w1, w2)
    yd, idd, wd = run(g, x[:4], T=1)
    check_against_oracle(small, x[:4], yd, idd, wd)
    yb, ib, wb = run(g, x[:64], T=64)
    check_against_oracle(small, x[:64], yb, ib, wb, rows=np.arange(0, 64, 8))
    assert np.array_equal(ib, i1[:64])
    g.close()


def test_page_prefill_chunk_of_4096():
    """512 experts top-10 + shared, H 2048, I 512, Zipf-biased router, one
    4,096-token call: routing of every token against the oracle's binary64
    logits, outputs of sampled tokens element by element."""
    L = synth.make_layer(synth.PAGE, layer=0)
    sh = L.shape
    T = 4096
    x, _ = resampled_tokens(L, 50000, T)
    g = make_gpu_layer(L, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    logits = oracle.router_logits(L.W_r, L.bias, x)
    for t in range(T):
        ri, rw, _, _ = oracle.topk(logits[t], sh.k)
        assert np.array_equal(idx[t], ri), t
        assert np.allclose(w[t], rw, rtol=W_RTOL_TC, atol=1e-7), t
    # the hottest expert spans many chunks; sample its first and last tokens too
    hot = np.bincount(idx.ravel(), minlength=sh.E).argmax()
    hot_tokens = np.nonzero((idx == hot).any(axis=1))[0]
    rows = np.unique(np.concatenate([np.arange(0, T, 256), [T - 1], hot_tokens[:2], hot_tokens[-2:]]))
    check_against_oracle(L, x, y, idx, w, rows=rows, w_rtol=W_RTOL_TC)
    g.close()


def test_prefill_needs_hidden_multiple_of_128():
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.LayerShape(H=192, E=8, k=2, I=64)
    L = synth.make_layer(sh, layer=1)
    with pytest.raises(moe.MoeError) as e:
        make_gpu_layer(L, max_tokens=65)
    assert e.value.code == 2
    g = make_gpu_layer(L, max_tokens=64)  # the batched path has no such limit
    g.close()
