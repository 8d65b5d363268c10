"""moe_route_noalloc: routing for callers that cannot allocate device memory
(for example code running inside a host framework that owns every device
allocation, or in a process whose device memory is reserved up front).

It must give the same routing as moe_forward's own routing step, call after
call, although its scratch is one fixed device array that every call reuses.
This file is collected last so a stop-at-first-failure run has already run
every other test before it."""
import numpy as np
import pytest

from quantized_expert_ffn_gemv_gb300 import synth
from tests.gpu_common import W_RTOL, make_gpu_layer, to_torch_bf16
from tests.inputs import resampled_tokens

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 8])
def test_noalloc_routing_matches_forward_twice(T):
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
    for _ in range(2):  # two calls in a row share the same scratch array
        idx = torch.full((T, L.shape.k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, L.shape.k), dtype=torch.float32, device="cuda")
        moe.route_noalloc(g.W_r, g.bias, xd, L.shape.k, idx, w)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy())
        assert np.allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=W_RTOL, atol=1e-7)
    g.close()


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
