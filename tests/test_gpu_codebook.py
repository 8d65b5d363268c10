"""The codebook weight format (16 non-linear levels per block scale) on the
fused decode kernel against the oracle: the small parity layer at one and
eight tokens per call (several tiles, a ragged last call), the page-scale
layer, and a slot pool (residency invariance and the LRU simulator)."""
import dataclasses

import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import check_against_oracle, make_gpu_layer, run
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu

SMALL_CB = dataclasses.replace(synth.SMALL, fmt=1)
PAGE_CB = dataclasses.replace(synth.PAGE, fmt=1)


@pytest.fixture(scope="module")
def small_cb():
    return synth.make_layer(SMALL_CB, layer=4)


@pytest.mark.parametrize("T", [1, 8])
def test_codebook_small_layer_against_oracle(small_cb, T):
    x, _ = resampled_tokens(small_cb, 600, 21)
    g = make_gpu_layer(small_cb, max_tokens=T)
    y, idx, w = run(g, x, T=T)
    check_against_oracle(small_cb, x, y, idx, w)
    st, code = g.stats()
    assert code == 0
    g.close()


def test_codebook_page_layer_sampled_rows():
    L = synth.make_layer(PAGE_CB, layer=2)
    x, _ = resampled_tokens(L, 800, 12)
    g = make_gpu_layer(L, max_tokens=1)
    y, idx, w = run(g, x, T=1)
    check_against_oracle(L, x, y, idx, w, rows=[0, 5, 11])
    g.close()


def test_codebook_pool_is_residency_invariant(small_cb):
    x, _ = resampled_tokens(small_cb, 900, 48)
    full = make_gpu_layer(small_cb, max_tokens=1)
    y0, i0, w0 = run(full, x, T=1)
    pool = make_gpu_layer(small_cb, max_tokens=1, n_slots=12)
    y1, i1, w1 = run(pool, x, T=1)
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)
    expect, _ = oracle.pool_sim(SMALL_CB.E, 12, [sorted(r.tolist()) for r in i1])
    assert np.array_equal(pool.miss_log(), expect)
    pool.close()
    full.close()


def test_codebook_refused_beyond_the_fused_kernel(small_cb):
    from quantized_expert_ffn_gemv_gb300 import moe
    with pytest.raises(moe.MoeError) as e:
        make_gpu_layer(small_cb, max_tokens=9)
    assert e.value.code == 2
