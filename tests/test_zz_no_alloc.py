"""moe_route_noalloc: routing for callers that cannot allocate device memory
(for example code running inside a host framework that owns every device
allocation, or in a process whose device memory is reserved up front).

It must give the same routing as moe_forward's own routing step, call after
call, although its scratch is one fixed device array that every call reuses;
and that routing must be the oracle's.  This file is collected last so a
stop-at-first-failure run has already run every other test before it."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import W_RTOL, make_gpu_layer, to_torch_bf16
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


def _route(moe, W, b, xd, k):
    import torch
    T = xd.shape[0]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.route_noalloc(W, b, xd, k, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 8, 9, 64])
def test_noalloc_routing_matches_forward_and_oracle_twice(T):
    """T = 1 and 8 run the fused decode kernel in moe_forward, 9 and 64 the
    batched kernels; the allocation-free kernel stages logits for 8 tokens at
    a time, so 9 and 64 take several rounds and its top-k warps several
    tokens each.  Selection and weights equal moe_forward's bit for bit."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    L = synth.make_layer(synth.PAGE, layer=0)
    x, _ = resampled_tokens(L, 40 * T, T)
    g = make_gpu_layer(L, max_tokens=T)
    xd = to_torch_bf16(x)
    idx_ref = torch.empty((T, L.shape.k), dtype=torch.int32, device="cuda")
    w_ref = torch.empty((T, L.shape.k), dtype=torch.float32, device="cuda")
    g.forward(xd, topk_idx=idx_ref, topk_w=w_ref)
    torch.cuda.synchronize()
    idx_ref, w_ref = idx_ref.cpu().numpy(), w_ref.cpu().numpy()
    logits = oracle.router_logits(L.W_r, L.bias, x)
    for _ in range(2):  # two calls in a row share the same scratch array
        idx, w = _route(moe, g.W_r, g.bias, xd, L.shape.k)
        assert np.array_equal(idx, idx_ref)
        assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))
        for t in range(T):
            ri, rw, _, _ = oracle.topk(logits[t], L.shape.k)
            assert np.array_equal(idx[t], ri), t
            assert np.allclose(w[t], rw, rtol=W_RTOL, atol=1e-7), t
    g.close()


def test_noalloc_accepts_exactly_its_limit():
    """T * E = 65536 (64 tokens, 1024 experts), the largest call the array
    holds, against the oracle's top-k."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.LayerShape(H=256, E=1024, k=8, I=64)
    W = synth.router(sh, 5)
    x = synth.activations(sh, 5, 0, 64)
    Wd = torch.as_tensor(W).cuda()
    xd = to_torch_bf16(x)
    logits = oracle.router_logits(W, None, x)
    for _ in range(2):
        idx, w = _route(moe, Wd, None, xd, sh.k)
        for t in range(64):
            ri, rw, _, gap = oracle.topk(logits[t], sh.k)
            if gap >= 1e-9:
                assert np.array_equal(idx[t], ri), t
            assert np.allclose(w[t], rw, rtol=W_RTOL, atol=1e-7), t


def test_noalloc_non_finite_logits_rank_last():
    """A -inf bias and a NaN router row: those experts rank below every
    finite logit (NaN below -inf), so each token still gets k distinct
    experts, the oracle's choice among the finite ones."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    sh = synth.SMALL
    L = synth.make_layer(sh, layer=2)
    x, _ = resampled_tokens(L, 0, 16)
    bias = np.zeros(sh.E, np.float32)
    bias[:40] = -np.inf
    bias[40:] = 0.0
    W = L.W_r.copy()
    W[63, 5] = np.nan
    idx, w = _route(moe, torch.as_tensor(W).cuda(), torch.as_tensor(bias).cuda(), to_torch_bf16(x), sh.k)
    finite = np.arange(40, 63)
    Wf = L.W_r[finite]
    logits = oracle.router_logits(Wf, None, x)
    for t in range(16):
        ri, rw, _, gap = oracle.topk(logits[t], sh.k)
        if gap >= 1e-9:
            assert np.array_equal(idx[t], finite[ri]), t
        assert np.allclose(w[t], rw, rtol=W_RTOL, atol=1e-7), t
        assert len(set(idx[t].tolist())) == sh.k


def test_noalloc_rejects_sizes_beyond_its_array():
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    W = torch.zeros((4096, 64), dtype=torch.float32, device="cuda")
    x = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((32, 4), dtype=torch.int32, device="cuda")
    w = torch.empty((32, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.route_noalloc(W, None, x, 4, idx, w)  # 32 * 4096 logits > 65536
    assert e.value.code == 2


def test_noalloc_binding_checks_tensors():
    """Mismatched shapes, dtypes or layouts are refused before any launch."""
    import torch
    from quantized_expert_ffn_gemv_gb300 import moe
    W = torch.zeros((64, 128), dtype=torch.float32, device="cuda")
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((4, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((4, 2), dtype=torch.float32, device="cuda")
    bad = [
        (W[:, :64], None, x, idx, w),                                         # W_r width != H
        (W, None, x, idx[:3], w),                                             # topk_idx too short
        (W, None, x, idx, w.double()),                                        # wrong dtype
        (W, torch.zeros(63, device="cuda"), x, idx, w),                       # bias length
        (W, None, x, idx.t(), w),                                             # not contiguous / shape
        (W.cpu(), None, x, idx, w),                                           # wrong device
    ]
    for Wt, b, xt, it, wt in bad:
        with pytest.raises(ValueError):
            moe.route_noalloc(Wt, b, xt, 2, it, wt)
