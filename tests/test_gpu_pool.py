"""The VRAM expert-slot pool on the GPU: misses match the LRU simulator,
output is bit-identical to the all-resident run, and copy failures or a
stalled copy server end in an error status (no GPU fault, no hang), in
both miss services (the kernel reading host memory, the host copy engine)."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import check_against_oracle, from_torch_bf16, make_gpu_layer, run, to_torch_bf16
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def small():
    return synth.make_layer(synth.SMALL, layer=0)


@pytest.mark.parametrize("service", [0, 1], ids=["copy_engine", "sm_pull"])
@pytest.mark.parametrize("T,S", [(1, 16), (4, 20)])
def test_pool_is_residency_invariant_and_matches_lru(small, T, S, service):
    x, _ = resampled_tokens(small, 500, 96)
    full = make_gpu_layer(small, max_tokens=T)
    y0, i0, w0 = run(full, x, T=T)
    pool = make_gpu_layer(small, max_tokens=T, n_slots=S)
    pool.set_miss_service(service)
    y1, i1, w1 = run(pool, x, T=T)
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)
    steps = [sorted(set(i1[t0:t0 + T].ravel().tolist())) for t0 in range(0, 96, T)]
    expect, _ = oracle.pool_sim(small.shape.E, S, steps)
    got = pool.miss_log()
    assert np.array_equal(got, expect)
    stats, code = pool.stats()
    assert code == 0
    assert stats["misses"] == len(expect)
    assert stats["hits"] + stats["misses"] == sum(len(s) for s in steps)
    assert stats["h2d_bytes"] == len(expect) * small.shape.expert_bytes
    check_against_oracle(small, x, y1, i1, w1, rows=np.arange(0, 96, 12))
    pool.close()
    full.close()


def test_failed_copy_is_an_error_not_zero_weights(small):
    from quantized_expert_ffn_gemv_gb300 import moe
    x, _ = resampled_tokens(small, 700, 8)
    pool = make_gpu_layer(small, max_tokens=1, n_slots=8)
    pool.set_miss_service(0)  # the host copy server moves the bytes (not the default: set explicitly)
    pool.debug_copy_faults(fail_copy_n=3)
    with pytest.raises(moe.MoeError) as ei:
        run(pool, x, T=1)
        run(pool, x, T=1)
    assert ei.value.code == 7  # sticky
    stats, code = pool.stats()
    assert code == 5 and stats["error"] == 5
    pool.close()


def test_stalled_copy_server_times_out(small):
    x, _ = resampled_tokens(small, 800, 1)
    pool = make_gpu_layer(small, max_tokens=1, n_slots=8)
    pool.set_miss_service(0)
    pool.set_wait_timeout_ns(200_000_000)
    pool.debug_copy_faults(pause=True)
    run(pool, x, T=1)  # the cold pool misses; nothing serves the doorbell
    stats, code = pool.stats()
    assert code == 6 and stats["error"] == 6 and stats["wait_ns"] >= 150_000_000
    pool.debug_copy_faults(pause=False)
    pool.close()


@pytest.mark.parametrize("service", [0, 1], ids=["copy_engine", "sm_pull"])
def test_seeded_pool_matches_lru_with_the_same_seed(small, service):
    """A pool seeded from a hot-expert profile: misses equal the simulator
    started from the same seed, output bit-identical to all-resident."""
    T, S = 1, 16
    x, _ = resampled_tokens(small, 900, 48)
    full = make_gpu_layer(small, max_tokens=T)
    y0, i0, w0 = run(full, x, T=T)
    # a profile: the experts the first 16 tokens select most often
    counts = np.bincount(i0[:16].ravel(), minlength=small.shape.E)
    seed = np.argsort(-counts, kind="stable")[:12].astype(np.int32)
    pool = make_gpu_layer(small, max_tokens=T, n_slots=S)
    pool.set_miss_service(service)
    pool.seed(seed)
    y1, i1, w1 = run(pool, x, T=T)
    assert np.array_equal(y0, y1) and np.array_equal(i0, i1) and np.array_equal(w0, w1)
    steps = [sorted(set(i1[t].tolist())) for t in range(48)]
    expect, _ = oracle.pool_sim(small.shape.E, S, steps, seed=seed.tolist())
    cold, _ = oracle.pool_sim(small.shape.E, S, steps)
    assert np.array_equal(pool.miss_log(), expect)
    assert len(expect) < len(cold)
    stats, code = pool.stats()
    assert code == 0 and stats["misses"] == len(expect)
    pool.close()
    full.close()


def test_seeding_errors(small):
    from quantized_expert_ffn_gemv_gb300 import moe
    full = make_gpu_layer(small, max_tokens=1)
    with pytest.raises(moe.MoeError) as ei:
        full.seed([0, 1])
    assert ei.value.code == 7  # every expert resident: no pool to seed
    pool = make_gpu_layer(small, max_tokens=1, n_slots=8)
    for bad in ([0, 0], [small.shape.E], list(range(9))):
        with pytest.raises(moe.MoeError) as ei:
            pool.seed(bad)
        assert ei.value.code == 1
    pool.seed([])  # an empty seed is the empty pool
    full.close()
    pool.close()


def test_pool_serves_up_to_eight_tokens_and_refuses_more(small):
    """A pooled layer runs the fused path (T <= 8); a call of 9 to 64 tokens
    is MOE_ERR_UNSUPPORTED before any launch (larger calls lend slots:
    tests/test_gpu_lend.py), and the layer stays usable."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    x, _ = resampled_tokens(small, 950, 9)
    pool = make_gpu_layer(small, max_tokens=9, n_slots=36)  # 36 >= 9 tokens x top-4
    xd = to_torch_bf16(x)
    yd = torch.empty_like(xd)
    with pytest.raises(moe.MoeError) as ei:
        pool.forward(xd, yd)
    assert ei.value.code == 2
    y, idx, w = run(pool, x[:8], T=8)
    check_against_oracle(small, x[:8], y, idx, w)
    stats, code = pool.stats()
    assert code == 0 and stats["forwards"] == 1
    pool.close()


@pytest.mark.parametrize("service", [0, 1], ids=["copy_engine", "sm_pull"])
def test_pool_with_calls_of_mixed_sizes(small, service):
    """One pooled layer called with 1, 3, 8, 2, 5, ... tokens per call: each
    call is one step of the LRU simulator (its union of selected experts),
    outputs bit-identical to the all-resident layer called the same way."""
    import torch
    sizes = [1, 3, 8, 2, 5, 1, 7, 4, 8, 6, 1, 2]
    n = sum(sizes)
    x, _ = resampled_tokens(small, 1200, n)
    full = make_gpu_layer(small, max_tokens=8)
    pool = make_gpu_layer(small, max_tokens=8, n_slots=40)
    pool.set_miss_service(service)
    outs = {}
    for name, layer in (("full", full), ("pool", pool)):
        xd = to_torch_bf16(x)
        yd = torch.empty_like(xd)
        idd = torch.empty((n, small.shape.k), dtype=torch.int32, device="cuda")
        wd = torch.empty((n, small.shape.k), dtype=torch.float32, device="cuda")
        t0 = 0
        for T in sizes:
            layer.forward(xd[t0:t0 + T], yd[t0:t0 + T], idd[t0:t0 + T], wd[t0:t0 + T])
            t0 += T
        torch.cuda.synchronize()
        outs[name] = (from_torch_bf16(yd), idd.cpu().numpy(), wd.cpu().numpy())
    for a, b in zip(outs["full"], outs["pool"]):
        assert np.array_equal(a, b)
    idx = outs["pool"][1]
    steps, t0 = [], 0
    for T in sizes:
        steps.append(sorted(set(idx[t0:t0 + T].ravel().tolist())))
        t0 += T
    expect, _ = oracle.pool_sim(small.shape.E, 40, steps)
    assert np.array_equal(pool.miss_log(), expect)
    check_against_oracle(small, x, *outs["pool"], rows=np.arange(0, n, 5))
    full.close()
    pool.close()


def test_copy_engine_service_never_times_out_under_stream_syncs():
    """The host copy server behind the doorbell, 10 runs of 200 tokens
    through 8 page-scale pooled layers (64 slots each), eager calls with a
    stream synchronize every 2 tokens: every run ends without a timeout and
    bit-identical to the all-resident layers.  The decode kernel waits for
    the copies, so a copy held behind the caller's queued work would end a
    call with MOE_ERR_TIMEOUT (bounded here at 0.5 s)."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    n_layers, n_tok, slots = 8, 200, 64
    layers = []
    for l in range(n_layers):
        L = synth.make_layer(synth.PAGE, layer=l)
        layers.append(moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=1))
        del L
    x = synth.activations(synth.PAGE, 5000, 0, n_tok)
    xd = to_torch_bf16(x)
    stream = torch.cuda.Stream()

    def once():
        ys = torch.empty((n_layers, n_tok, synth.PAGE.H), dtype=torch.bfloat16, device="cuda")
        with torch.cuda.stream(stream):
            for t in range(n_tok):
                for l, layer in enumerate(layers):
                    layer.forward(xd[t:t + 1], ys[l, t:t + 1], stream=stream)
                if t % 2 == 1:
                    stream.synchronize()
        torch.cuda.synchronize()
        return ys

    ref = once()
    for layer in layers:
        layer.configure(slots)
        layer.set_miss_service(0)
        layer.set_wait_timeout_ns(500_000_000)
    codes = []
    for run_no in range(10):
        for layer in layers:
            layer.configure(slots)
        ys = once()
        st = [layer.stats() for layer in layers]
        codes.append([c for _, c in st])
        assert all(c == 0 for c in codes[-1]), (run_no, codes[-1])
        assert torch.equal(ys.view(torch.int16), ref.view(torch.int16)), run_no
        assert sum(s["misses"] for s, _ in st) > 0
    for layer in layers:
        layer.close()
