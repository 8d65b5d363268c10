"""A stack of MoE layers with residual + RMSNorm between them.

Per layer l (pre-norm, no learned weight, eps 1e-6):
    xhat_l  = bf16(x_l / sqrt(mean(x_l^2) + eps))
    y_l     = MoE_l(xhat_l)                        (moe_forward)
    x_{l+1} = bf16(x_l + y_l)
The stack's output is x_L.  Every layer owns its own VRAM expert-slot pool
(Betelgeuse news page, section 机制, 显存 row: per-layer slot budgets), fed
from its pinned host master copy on a miss.  Marshalling only: each step is
one of the library's kernels.
"""
import numpy as np

from . import moe


class MoeStack:
    def __init__(self, layers, max_tokens=1, n_slots=None, eps=1e-6, device=0, seeds=None):
        """layers: synth.Layer objects (router, bias, canonical blobs).
        n_slots: one slot budget for every layer, or one per layer (the
        Betelgeuse news page's 显存 row gives early layers more slots than
        late ones); None = every expert resident.  seeds: per layer, the
        experts a pool starts with (a hot-expert profile), or None."""
        import torch
        self.eps = eps
        budgets = n_slots if isinstance(n_slots, (list, tuple)) else [n_slots] * len(layers)
        if len(budgets) != len(layers):
            raise ValueError("one slot budget per layer")
        self.layers = [moe.MoeLayer(L.shape, L.W_r, L.bias, L.experts, L.shared, max_tokens=max_tokens,
                                    n_slots=b, device=device) for L, b in zip(layers, budgets)]
        if seeds is not None:
            self.seed(seeds)
        self.H = layers[0].shape.H
        self.k = layers[0].shape.k
        self.device = torch.device("cuda", device)
        self.link()

    fused = True  # residual + RMSNorm inside each layer's call (moe_forward_norm)

    def buffers(self, T, record=False):
        import torch
        n = len(self.layers)
        z = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device=self.device)
        b = {"x": z(2, T, self.H), "xhat": z(T, self.H), "y": z(2, T, self.H)}
        if record:
            b["xhats"] = z(n, T, self.H)
            b["ys"] = z(n, T, self.H)
            b["idx"] = z(n, T, self.k, dt=torch.int32)
            b["w"] = z(n, T, self.k, dt=torch.float32)
        return b

    def forward(self, x, bufs, stream=None):
        """x: torch bf16 [T, H] (device).  Returns the output x_L (a view into bufs).

        fused: each layer's call adds the residual and normalises its own input
        (one kernel per layer for T <= 8); otherwise a residual + RMSNorm
        kernel runs between the layers.  Both give bit-identical results."""
        rec = "xhats" in bufs
        T = x.shape[0]
        cur = 0
        bufs["x"][0][:T].copy_(x)
        if not self.fused:
            moe.residual_rmsnorm(bufs["x"][0][:T], None, self.eps, None, bufs["xhat"][:T], stream)
        y_prev = None
        for l, layer in enumerate(self.layers):
            y = bufs["ys"][l][:T] if rec else bufs["y"][l % 2][:T]
            idx = bufs["idx"][l][:T] if rec else None
            w = bufs["w"][l][:T] if rec else None
            nxt = 1 - cur
            if self.fused:
                # x_l = bf16(x_{l-1} + y_{l-1}) (x_0 = x), its RMSNorm, the layer
                xhat = bufs["xhats"][l][:T] if rec else bufs["xhat"][:T]
                x_out = None if y_prev is None else bufs["x"][nxt][:T]
                layer.forward_norm(bufs["x"][cur][:T], y_prev, self.eps, x_out, xhat, y, idx, w, stream=stream)
                if y_prev is not None:
                    cur = nxt
            else:
                if rec:
                    bufs["xhats"][l][:T].copy_(bufs["xhat"][:T])
                layer.forward(bufs["xhat"][:T], y, idx, w, stream=stream)
                # x_{l+1} = bf16(x_l + y_l); its RMSNorm feeds the next layer
                moe.residual_rmsnorm(bufs["x"][cur][:T], y, self.eps, bufs["x"][nxt][:T], bufs["xhat"][:T], stream)
                cur = nxt
            y_prev = y
        if self.fused:
            # x_L = bf16(x_{L-1} + y_{L-1})
            moe.residual_rmsnorm(bufs["x"][cur][:T], y_prev, self.eps, bufs["x"][1 - cur][:T], bufs["xhat"][:T],
                                 stream)
            cur = 1 - cur
        return bufs["x"][cur][:T]

    def link(self, hot=None):
        """Each layer warms L2 for the next one at the end of its decode call
        (router rows, shared expert, and hot[l + 1], a list of layer l + 1's
        most-selected experts, when given); the last layer links to none."""
        for l, layer in enumerate(self.layers):
            nxt = self.layers[l + 1] if l + 1 < len(self.layers) else None
            layer.set_next(nxt, None if (hot is None or nxt is None) else hot[l + 1])

    def seed(self, seeds):
        """Start every pooled layer's pool from its list of hot experts."""
        if len(seeds) != len(self.layers):
            raise ValueError("one seed list per layer")
        for l, sd in zip(self.layers, seeds):
            if sd is not None and l.n_slots < l.shape.E:
                l.seed(list(sd)[:l.n_slots])

    def set_miss_service(self, mode):
        """Miss service of every layer's pool (see MoeLayer.set_miss_service)."""
        for l in self.layers:
            l.set_miss_service(mode)

    def stats(self):
        return [l.stats()[0] for l in self.layers]

    def close(self):
        for l in self.layers:
            if getattr(l, "h", None):
                l.set_next(None)
        for l in self.layers:
            l.close()
