"""ctypes binding of the CUDA library (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's
kernels.  Functions mirror the C ABI names; ``MoeLayer`` bundles one layer
handle with the torch tensors whose lifetime it needs (router weights, slot
arena).  There is no CPU fallback: a missing library or GPU raises.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OUT_OF_MEMORY",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_COPY", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_STATE", 8: "MOE_ERR_DEVICE"}
EXPORTS = ["moe_expert_bytes", "moe_repack_expert", "moe_unpack_expert", "moe_layer_create",
           "moe_slot_pool_configure", "moe_forward", "moe_residual_rmsnorm", "moe_get_stats", "moe_get_miss_log",
           "moe_set_wait_timeout_ns", "moe_debug_copy_faults", "moe_destroy", "moe_status_string",
           "moe_route_noalloc", "moe_set_miss_service", "moe_slot_pool_seed", "moe_forward_norm",
           "moe_set_next_layer"]


class MoeError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")


class LayerDesc(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_experts", C.c_int32), ("top_k", C.c_int32), ("n_shared", C.c_int32),
                ("inter", C.c_int32), ("qblock", C.c_int32), ("max_tokens", C.c_int32), ("device", C.c_int32),
                ("router_w", C.c_void_p), ("router_bias", C.c_void_p), ("experts", C.c_void_p),
                ("shared", C.c_void_p), ("weight_format", C.c_int32)]


class Stats(C.Structure):
    _fields_ = [("forwards", C.c_uint64), ("hits", C.c_uint64), ("misses", C.c_uint64), ("h2d_bytes", C.c_uint64),
                ("wait_ns", C.c_uint64), ("n_slots", C.c_int32), ("error", C.c_int32), ("rechecks", C.c_uint64)]


_lib = None


def lib(build_if_missing=False):
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.CUDA_LIB
        if build_if_missing:
            path = _build.build_cuda()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path}); run __graft_entry__.build()")
        L = C.CDLL(path)
        p, i32, i64, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64
        L.moe_expert_bytes.argtypes = [i32, i32]
        L.moe_expert_bytes.restype = C.c_size_t
        for f in ("moe_repack_expert", "moe_unpack_expert"):
            getattr(L, f).argtypes = [p, i32, i32, p]
        L.moe_layer_create.argtypes = [C.POINTER(LayerDesc), C.POINTER(p)]
        L.moe_slot_pool_configure.argtypes = [p, i32, p, C.c_size_t]
        L.moe_slot_pool_seed.argtypes = [p, p, i32]
        L.moe_forward.argtypes = [p, p, i32, p, p, p, p]
        L.moe_forward_norm.argtypes = [p, p, p, i32, C.c_float, p, p, p, p, p, p]
        L.moe_residual_rmsnorm.argtypes = [p, p, i32, i32, C.c_float, p, p, p]
        L.moe_get_stats.argtypes = [p, C.POINTER(Stats)]
        L.moe_get_miss_log.argtypes = [p, p, i64, C.POINTER(i64)]
        L.moe_set_wait_timeout_ns.argtypes = [p, u64]
        L.moe_set_miss_service.argtypes = [p, i32]
        L.moe_set_next_layer.argtypes = [p, p, p, i32]
        L.moe_debug_copy_faults.argtypes = [p, i64, i32]
        L.moe_destroy.argtypes = [p]
        L.moe_destroy.restype = None
        L.moe_route_noalloc.argtypes = [p, p, p, i32, i32, i32, i32, p, p, p]
        L.moe_status_string.argtypes = [C.c_int]
        L.moe_status_string.restype = C.c_char_p
        for f in EXPORTS:
            if f not in ("moe_destroy", "moe_status_string", "moe_expert_bytes"):
                getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def status_string(code):
    try:
        return lib().moe_status_string(code).decode()
    except Exception:  # library missing: still name the code
        return STATUS.get(code, str(code))


def check(code, what):
    if code != MOE_OK:
        raise MoeError(code, what)


def expert_bytes(H, I):
    return int(lib().moe_expert_bytes(H, I))


def repack_expert(canon, H, I):
    canon = np.ascontiguousarray(canon, np.uint8)
    out = np.empty(expert_bytes(H, I), np.uint8)
    check(lib().moe_repack_expert(canon.ctypes.data, H, I, out.ctypes.data), "moe_repack_expert")
    return out


def unpack_expert(gpu, H, I):
    gpu = np.ascontiguousarray(gpu, np.uint8)
    out = np.empty(expert_bytes(H, I), np.uint8)
    check(lib().moe_unpack_expert(gpu.ctypes.data, H, I, out.ctypes.data), "moe_unpack_expert")
    return out


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check_tensors(device, items):
    """Each (name, tensor or None, dtype, shape) must match exactly, be
    contiguous and live on `device` (a CUDA device); a mismatch raises
    ValueError before anything reaches the library, so it is never an
    out-of-bounds device access."""
    for name, t, dt, shape in items:
        if t is None:
            continue
        if t.dtype != dt or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: expected {dt} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type != "cuda" or t.device != device:
            raise ValueError(f"{name} must be a CUDA tensor on {device}, got {t.device}")


def residual_rmsnorm(x, y, eps, x_out, xhat, stream=None):
    """x_out = bf16(x + y); xhat = bf16(rmsnorm(x_out)); torch bf16 CUDA tensors [T, H]."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be [T, H]")
    T, H = x.shape
    bf = torch.bfloat16
    _check_tensors(x.device, [("x", x, bf, (T, H)), ("y", y, bf, (T, H)), ("x_out", x_out, bf, (T, H)),
                              ("xhat", xhat, bf, (T, H))])
    check(lib().moe_residual_rmsnorm(x.data_ptr(), None if y is None else y.data_ptr(), T, H, eps,
                                     None if x_out is None else x_out.data_ptr(), xhat.data_ptr(),
                                     _stream_ptr(stream)), "moe_residual_rmsnorm")


def route_noalloc(W_r, bias, x, k, topk_idx, topk_w, stream=None):
    """Router + top-k without any device allocation (torch CUDA tensors).

    W_r float32 [E, H], bias float32 [E] or None, x bf16 [T, H]; writes
    topk_idx int32 [T, k] and topk_w float32 [T, k].  Shapes, dtypes,
    contiguity and device are checked here, so a mismatched tensor is an
    error and never an out-of-bounds device access."""
    import torch
    if x.dim() != 2 or W_r.dim() != 2:
        raise ValueError("x must be [T, H] and W_r [E, H]")
    T, H = x.shape
    E = W_r.shape[0]
    tensors = {"W_r": (W_r, torch.float32, (E, H)), "x": (x, torch.bfloat16, (T, H)),
               "topk_idx": (topk_idx, torch.int32, (T, k)), "topk_w": (topk_w, torch.float32, (T, k))}
    if bias is not None:
        tensors["bias"] = (bias, torch.float32, (E,))
    for name, (t, dt, shape) in tensors.items():
        if t.dtype != dt or tuple(t.shape) != shape:
            raise ValueError(f"{name}: expected {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != x.device or t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor on {x.device}")
    check(lib().moe_route_noalloc(W_r.data_ptr(), None if bias is None else bias.data_ptr(), x.data_ptr(), T, H,
                                  W_r.shape[0], k, topk_idx.data_ptr(), topk_w.data_ptr(), _stream_ptr(stream)),
          "moe_route_noalloc")


class MoeLayer:
    """One layer: handle + the device tensors it references.

    W_r float32 [E, H], bias float32 [E] or None, experts uint8 canonical blobs
    (numpy, E back to back), shared uint8 canonical blob or None.
    n_slots None = every expert resident."""

    def __init__(self, shape, W_r, bias, experts, shared, max_tokens=1, n_slots=None, device=0):
        import torch
        self.shape = shape
        self.device = torch.device("cuda", device)
        self.max_tokens = max_tokens
        self.W_r = torch.as_tensor(np.ascontiguousarray(W_r, np.float32)).to(self.device)
        self.bias = None if bias is None else torch.as_tensor(np.ascontiguousarray(bias, np.float32)).to(self.device)
        experts = np.ascontiguousarray(experts, np.uint8)
        shared_np = None if shared is None else np.ascontiguousarray(shared, np.uint8)
        d = LayerDesc(hidden=shape.H, n_experts=shape.E, top_k=shape.k, n_shared=0 if shared is None else 1,
                      inter=shape.I, qblock=32, max_tokens=max_tokens, device=device,
                      router_w=self.W_r.data_ptr(), router_bias=None if self.bias is None else self.bias.data_ptr(),
                      experts=experts.ctypes.data, shared=None if shared_np is None else shared_np.ctypes.data,
                      weight_format=getattr(shape, "fmt", 0))
        h = C.c_void_p()
        check(lib().moe_layer_create(C.byref(d), C.byref(h)), "moe_layer_create")
        self.h = h
        self.arena = None
        self.configure(shape.E if n_slots is None else n_slots)

    def configure(self, n_slots):
        import torch
        nbytes = n_slots * expert_bytes(self.shape.H, self.shape.I)
        if self.arena is None or self.arena.numel() < nbytes:
            self.arena = None
            self.arena = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        check(lib().moe_slot_pool_configure(self.h, n_slots, self.arena.data_ptr(), self.arena.numel()),
              "moe_slot_pool_configure")
        self.n_slots = n_slots

    def seed(self, experts):
        """Start the configured pool with these experts resident (expert i of the list in slot i)."""
        e = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
        check(lib().moe_slot_pool_seed(self.h, e.ctypes.data if len(e) else None, len(e)), "moe_slot_pool_seed")

    def _check_io(self, T, acts, topk_idx, topk_w):
        import torch
        H, k = self.shape.H, self.shape.k
        _check_tensors(self.device, [(n, t, torch.bfloat16, (T, H)) for n, t in acts] +
                       [("topk_idx", topk_idx, torch.int32, (T, k)), ("topk_w", topk_w, torch.float32, (T, k))])

    def forward(self, x, y=None, topk_idx=None, topk_w=None, stream=None):
        """x: torch bf16 [T, H] on the layer's device; returns y (bf16 [T, H])."""
        import torch
        if x.dim() != 2:
            raise ValueError("x must be [T, H]")
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        self._check_io(T, [("x", x), ("y", y)], topk_idx, topk_w)
        check(lib().moe_forward(self.h, x.data_ptr(), T, y.data_ptr(),
                                None if topk_idx is None else topk_idx.data_ptr(),
                                None if topk_w is None else topk_w.data_ptr(), _stream_ptr(stream)), "moe_forward")
        return y

    def forward_norm(self, x, y_prev, eps, x_out, xhat, y, topk_idx=None, topk_w=None, stream=None):
        """One pre-norm stack layer: x_out = bf16(x + y_prev), xhat = bf16(rmsnorm(x_out)),
        y = MoE(xhat).  torch bf16 [T, H] tensors on the layer's device; y_prev and
        x_out may be None."""
        if x.dim() != 2:
            raise ValueError("x must be [T, H]")
        self._check_io(x.shape[0], [("x", x), ("y_prev", y_prev), ("x_out", x_out), ("xhat", xhat), ("y", y)],
                       topk_idx, topk_w)
        opt = lambda t: None if t is None else t.data_ptr()
        check(lib().moe_forward_norm(self.h, x.data_ptr(), opt(y_prev), x.shape[0], eps, opt(x_out),
                                     xhat.data_ptr(), y.data_ptr(), opt(topk_idx), opt(topk_w),
                                     _stream_ptr(stream)), "moe_forward_norm")
        return y

    def stats(self):
        s = Stats()
        code = lib().moe_get_stats(self.h, C.byref(s))
        return {f: getattr(s, f) for f, _ in Stats._fields_}, code

    def miss_log(self, max_entries=1 << 20):
        out = np.empty((max_entries, 3), np.int32)
        n = C.c_int64()
        check(lib().moe_get_miss_log(self.h, out.ctypes.data, max_entries, C.byref(n)), "moe_get_miss_log")
        return out[:min(n.value, max_entries)].copy()

    def set_wait_timeout_ns(self, ns):
        check(lib().moe_set_wait_timeout_ns(self.h, ns), "moe_set_wait_timeout_ns")

    def set_miss_service(self, mode):
        """1 = the kernel reads misses from host memory (default), 0 = host copy engine behind the doorbell."""
        check(lib().moe_set_miss_service(self.h, int(mode)), "moe_set_miss_service")

    def set_next(self, nxt, hot=None):
        """Warm L2 for `nxt` (the layer called after this one) at the end of
        every decode call: its router rows, shared expert and the listed hot
        experts.  nxt None removes the link."""
        hot = np.ascontiguousarray(np.asarray([] if hot is None else hot, dtype=np.int32))
        check(lib().moe_set_next_layer(self.h, None if nxt is None else nxt.h, hot.ctypes.data if len(hot) else None,
                                       len(hot)), "moe_set_next_layer")
        self.next = nxt

    def debug_copy_faults(self, fail_copy_n=0, pause=False):
        check(lib().moe_debug_copy_faults(self.h, fail_copy_n, int(pause)), "moe_debug_copy_faults")

    def close(self):
        if getattr(self, "h", None):
            lib().moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
