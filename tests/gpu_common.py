"""Helpers shared by the GPU parity tests."""
import numpy as np

import oracle
from quantized_expert_ffn_gemv_gb300 import synth

REL_L2 = 2e-3   # per token row
MAX_ABS = 5e-3  # every element
W_RTOL = 1e-5   # routing weights (fp32 softmax vs binary64)
# Routing weights when the router runs on the tensor cores (prefill): the
# logits are sums of 2048 exact bf16 x bf16 products accumulated by the MMA
# unit in fp32 without IEEE round-to-nearest at every step; the logit error
# is about 1e-5 (100x inside the 1e-3 near-tie gap), so a weight may move
# by twice that relative.
W_RTOL_TC = 1e-4


def to_torch_bf16(x_u16, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_u16).view(np.int16)).to(device).view(torch.bfloat16)


def from_torch_bf16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_gpu_layer(L, max_tokens=1, n_slots=None, with_shared=True):
    from quantized_expert_ffn_gemv_gb300 import moe
    return moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared if with_shared else None,
                        max_tokens=max_tokens, n_slots=n_slots)


def run(layer, x_u16, T=None):
    """Run the GPU layer on x in calls of T tokens; returns (y u16, idx, w)."""
    import torch
    n = x_u16.shape[0]
    T = T or n
    k = layer.shape.k
    y = np.empty_like(x_u16)
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    xd = to_torch_bf16(x_u16)
    yd = torch.empty_like(xd)
    idd = torch.empty((n, k), dtype=torch.int32, device="cuda")
    wd = torch.empty((n, k), dtype=torch.float32, device="cuda")
    for t0 in range(0, n, T):
        t1 = min(n, t0 + T)
        layer.forward(xd[t0:t1], yd[t0:t1], idd[t0:t1], wd[t0:t1])
    torch.cuda.synchronize()
    y[:] = from_torch_bf16(yd)
    idx[:] = idd.cpu().numpy()
    w[:] = wd.cpu().numpy()
    return y, idx, w


def check_against_oracle(L, x_u16, y, idx, w, rows=None, w_rtol=W_RTOL):
    sh = L.shape
    rows = np.arange(x_u16.shape[0]) if rows is None else np.asarray(rows)
    ref = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, x_u16[rows], fmt=sh.fmt)
    assert np.array_equal(idx[rows], ref["idx"]), "routing differs from the oracle"
    assert np.allclose(w[rows], ref["w"], rtol=w_rtol, atol=1e-7)
    yg = synth.bf16_to_f32(y[rows]).astype(np.float64)
    r = ref["y"]
    err = yg - r
    rel = np.linalg.norm(err, axis=1) / np.linalg.norm(r, axis=1)
    assert rel.max() <= REL_L2, f"rel-L2 {rel.max():.3e}"
    assert np.abs(err).max() <= MAX_ABS, f"max-abs {np.abs(err).max():.3e}"
    # per element: the output's own bf16 rounding (half an ulp of the oracle
    # value) plus the fp16 rounding of the intermediate h (relative RMS about
    # 2e-4, so 2e-3 of the row RMS is a 7-sigma bound)
    mag = np.abs(r)
    e = np.floor(np.log2(np.maximum(mag, 1e-30)))
    half_ulp = np.ldexp(1.0, (e - 8).astype(np.int64))
    slack = 2e-3 * np.sqrt((r * r).mean(axis=1, keepdims=True))
    assert np.all(np.abs(err) <= half_ulp + slack), f"{(np.abs(err) > half_ulp + slack).sum()} elements off"
    return rel.max(), np.abs(err).max()
