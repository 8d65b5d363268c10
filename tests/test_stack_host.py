"""MoeStack's orchestration on the CPU, with stand-in layers.

The fused path (each layer's call adds the residual and normalises its own
input) and the path with a residual + RMSNorm kernel between the layers must
hand every layer the same input and give the same output, equal to the
plain pre-norm recursion x_{l+1} = bf16(x_l + y_l), y_l = f_l(rmsnorm(x_l)).
No call may be given an output that overlaps one of its inputs or another
output: the fused kernel's blocks read the inputs while others already write.
"""
import pytest
import torch

from quantized_expert_ffn_gemv_gb300 import moe
from quantized_expert_ffn_gemv_gb300.stack import MoeStack

H, K, EPS = 64, 2, 1e-6


def bf16(t):
    return t.to(torch.bfloat16)


def residual_norm(x, y, eps):
    """(bf16(x + y), bf16(rmsnorm(bf16(x + y)))), y may be None."""
    v = x.float() + (y.float() if y is not None else 0.0)
    xs = bf16(v)
    ms = (xs.float() ** 2).mean(dim=1, keepdim=True)
    return xs, bf16(xs.float() / torch.sqrt(ms + eps))


def disjoint(a, b):
    if a is None or b is None:
        return True
    a0, b0 = a.data_ptr(), b.data_ptr()
    return a0 + a.numel() * a.element_size() <= b0 or b0 + b.numel() * b.element_size() <= a0


class FakeLayer:
    """Stands in for moe.MoeLayer: y = f_l(xhat), a fixed elementwise map."""

    def __init__(self, l):
        self.l = l
        self.inputs = []

    def f(self, xh):
        return bf16(torch.tanh(xh.float() * (0.5 + 0.1 * self.l)) * 0.3)

    def _fill(self, idx, w):
        if idx is not None:
            idx.fill_(self.l)
        if w is not None:
            w.fill_(0.5)

    def forward(self, x, y, topk_idx=None, topk_w=None, stream=None):
        assert disjoint(x, y)
        self.inputs.append(x.clone())
        y.copy_(self.f(x))
        self._fill(topk_idx, topk_w)

    def forward_norm(self, x, y_prev, eps, x_out, xhat, y, topk_idx=None, topk_w=None, stream=None):
        outs = [o for o in (x_out, xhat, y) if o is not None]
        for o in outs:
            assert disjoint(o, x) and disjoint(o, y_prev)
        for i in range(len(outs)):
            for j in range(i + 1, len(outs)):
                assert disjoint(outs[i], outs[j])
        xs, xh = residual_norm(x, y_prev, eps)
        if x_out is not None:
            x_out.copy_(xs)
        xhat.copy_(xh)
        self.inputs.append(xh.clone())
        y.copy_(self.f(xh))
        self._fill(topk_idx, topk_w)


def fake_residual_rmsnorm(x, y, eps, x_out, xhat, stream=None):
    assert disjoint(xhat, x) and disjoint(xhat, y) and disjoint(xhat, x_out)
    xs, xh = residual_norm(x, y, eps)
    if x_out is not None:
        x_out.copy_(xs)
    xhat.copy_(xh)


def make_stack(n_layers, fused):
    st = MoeStack.__new__(MoeStack)
    st.layers = [FakeLayer(l) for l in range(n_layers)]
    st.eps, st.H, st.k, st.device = EPS, H, K, torch.device("cpu")
    st.fused = fused
    return st


def reference(x, n_layers):
    fs = [FakeLayer(l) for l in range(n_layers)]
    xhats = []
    for l in range(n_layers):
        _, xh = residual_norm(x, None, EPS)
        xhats.append(xh)
        x = bf16(x.float() + fs[l].f(xh).float())
    return x, xhats


@pytest.mark.parametrize("n_layers", [1, 2, 5])
@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("record", [False, True])
def test_fused_and_split_stacks_agree_with_the_recursion(monkeypatch, n_layers, T, record):
    monkeypatch.setattr(moe, "residual_rmsnorm", fake_residual_rmsnorm)
    g = torch.Generator().manual_seed(7 + n_layers + T)
    x = bf16(torch.randn(T, H, generator=g))
    want, want_xhats = reference(x, n_layers)
    results = {}
    for fused in (True, False):
        st = make_stack(n_layers, fused)
        bufs = st.buffers(T, record=record)
        for _ in range(2):  # the second call reuses every buffer
            for layer in st.layers:
                layer.inputs.clear()
            out = st.forward(x, bufs).clone()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), fused
        for l, layer in enumerate(st.layers):
            assert len(layer.inputs) == 1
            assert torch.equal(layer.inputs[0].view(torch.int16), want_xhats[l].view(torch.int16)), (fused, l)
        if record:
            results[fused] = {k: bufs[k].clone() for k in ("xhats", "ys", "idx", "w")}
    if record:
        for k in ("xhats", "ys", "idx", "w"):
            assert torch.equal(results[True][k].view(torch.int8), results[False][k].view(torch.int8)), k
