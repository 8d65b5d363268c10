"""Prefill on a pooled layer: the prompt path lends the pool's last slots
(Basalt README, section "Prompt chunks": the chunk's buffers are carved from
the expert cache's last slots and the experts in them are copied back
afterwards).  The call's output equals the resident layer's bit for bit,
the pool is exactly as before (decode outputs and the miss log, which must
equal the LRU simulator over the decode steps alone), and a pool too small
to lend the scratch is refused."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import make_gpu_layer, run
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


def test_pooled_prefill_lends_slots_and_gives_them_back():
    L = synth.make_layer(synth.PAGE, layer=4)
    T = 512
    x1, _ = resampled_tokens(L, 3000, 24)
    xp = synth.activations(L.shape, 4, 7000, T, stream=5)
    x2, _ = resampled_tokens(L, 4000, 24)
    full = make_gpu_layer(L, max_tokens=T)
    pool = make_gpu_layer(L, max_tokens=T, n_slots=128)
    outs = []
    for g in (full, pool):
        a = run(g, x1, T=1)
        b = run(g, xp, T=T)
        c = run(g, x2, T=1)
        outs.append((a, b, c))
    for part in range(3):
        for f, p in zip(outs[0][part], outs[1][part]):
            assert np.array_equal(f, p), part
    # the decode steps alone drive the pool
    i1, i2 = outs[1][0][1], outs[1][2][1]
    steps = [sorted(r.tolist()) for r in i1] + [sorted(r.tolist()) for r in i2]
    expect, _ = oracle.pool_sim(L.shape.E, 128, steps)
    assert np.array_equal(pool.miss_log(), expect)
    stats, code = pool.stats()
    assert code == 0 and stats["misses"] == len(expect)
    full.close()
    pool.close()


def test_pool_too_small_to_lend_is_refused():
    """A 4,096-token prefill scratch takes about 104 page-scale slots: an
    80-slot pool (the decode minimum, 8 tokens x top-10) cannot lend it and
    one staging slot, so configure refuses it (MOE_ERR_OUT_OF_MEMORY)."""
    from quantized_expert_ffn_gemv_gb300 import moe
    L = synth.make_layer(synth.PAGE, layer=5)
    with pytest.raises(moe.MoeError) as e:
        make_gpu_layer(L, max_tokens=4096, n_slots=80)  # 4,096-token scratch needs ~104 slots
    assert e.value.code == 3
