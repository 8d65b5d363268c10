"""ctypes marshalling for the C oracle (moe_oracle.c).  Test infrastructure."""
import ctypes as C

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        i64, p = C.c_int64, C.c_void_p
        _lib.oracle_dequant_matrix.argtypes = [p, i64, i64, i64, p]
        _lib.oracle_levels.argtypes = [p]
        _lib.oracle_expert_bytes.argtypes = [i64, i64]
        _lib.oracle_expert_bytes.restype = i64
        _lib.oracle_router_logits.argtypes = [i64, i64, p, p, p, i64, p]
        _lib.oracle_topk.argtypes = [i64, i64, p, p, p, p]
        _lib.oracle_topk.restype = C.c_double
        _lib.oracle_expert.argtypes = [p, i64, i64, i64, p, p, p]
        _lib.oracle_moe_forward.argtypes = [i64, i64, i64, i64, p, p, p, p, p, i64, p, p, p, p, p, p, i64]
        _lib.oracle_rmsnorm.argtypes = [i64, p, C.c_double, p, p]
        _lib.oracle_residual.argtypes = [i64, p, p, p]
        _lib.oracle_to_bf16.argtypes = [i64, p, p]
        _lib.oracle_pool_sim.argtypes = [i64, i64, C.c_int, p, i64, i64, p, i64, p, i64, p]
        _lib.oracle_pool_sim.restype = i64
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def expert_bytes(H, I):
    return int(lib().oracle_expert_bytes(H, I))


def dequant_matrix(mat, R, K, fmt=0):
    """R x K float64 weights of one packed matrix (nibble plane + scale plane) of weight format fmt."""
    mat = _c(mat, np.uint8)
    out = np.empty((R, K), np.float64)
    lib().oracle_dequant_matrix(_ptr(mat), R, K, fmt, _ptr(out))
    return out


def levels():
    """The 16 levels of the codebook format (format 1)."""
    out = np.empty(16, np.float64)
    lib().oracle_levels(_ptr(out))
    return out


def router_logits(W_r, bias, x_bf16):
    """T x E float64 logits; W_r float32 [E,H], bias float32 [E] or None, x uint16 bf16 [T,H]."""
    W_r = _c(W_r, np.float32)
    E, H = W_r.shape
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((x.shape[0], E), np.float64)
    lib().oracle_router_logits(E, H, _ptr(W_r), _ptr(b), _ptr(x), x.shape[0], _ptr(out))
    return out


def topk(logits, k):
    """(idx ascending int32[k], w float64[k], by_rank int32[k], gap) for one token."""
    l = _c(logits, np.float64)
    E = l.shape[0]
    idx = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    br = np.empty(k, np.int32)
    gap = lib().oracle_topk(E, k, _ptr(l), _ptr(idx), _ptr(w), _ptr(br))
    return idx, w, br, gap


def expert(blob, H, I, x, fmt=0):
    """(y float64[H], h float64[I]) of one expert on float64 activations x[H]."""
    blob = _c(blob, np.uint8)
    x = _c(x, np.float64)
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64)
    lib().oracle_expert(_ptr(blob), H, I, fmt, _ptr(x), _ptr(y), _ptr(h))
    return y, h


def moe_forward(H, I, E, k, W_r, bias, experts, shared, x_bf16, force=None, fmt=0):
    """Layer on T tokens: dict(y [T,H] f64, idx [T,k], w [T,k], logits [T,E], gap [T])."""
    W_r = _c(W_r, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    ex = _c(experts, np.uint8)
    sh = None if shared is None else _c(shared, np.uint8)
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    T = x.shape[0]
    y = np.empty((T, H), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    gap = np.empty(T, np.float64)
    f = None if force is None else _c(force, np.int32).reshape(T, k)
    lib().oracle_moe_forward(H, I, E, k, _ptr(W_r), _ptr(b), _ptr(ex), _ptr(sh), _ptr(x), T, _ptr(y),
                             _ptr(idx), _ptr(w), _ptr(logits), _ptr(gap), _ptr(f), fmt)
    return dict(y=y, idx=idx, w=w, logits=logits, gap=gap)


def rmsnorm(x_bf16, eps=1e-6):
    """(xhat bf16 uint16 [H], xhat float64 [H]) for one token."""
    x = _c(x_bf16, np.uint16)
    H = x.shape[-1]
    out = np.empty(H, np.uint16)
    outf = np.empty(H, np.float64)
    lib().oracle_rmsnorm(H, _ptr(x), eps, _ptr(out), _ptr(outf))
    return out, outf


def residual(x_bf16, y_bf16):
    x = _c(x_bf16, np.uint16)
    y = _c(y_bf16, np.uint16)
    out = np.empty_like(x)
    lib().oracle_residual(x.size, _ptr(x), _ptr(y), _ptr(out))
    return out


def to_bf16(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_to_bf16(v.size, _ptr(v), _ptr(out))
    return out


def pool_sim(E, S, steps, init_full=False, max_miss=None, seed=None):
    """Replay a list of per-step expert selections; returns (misses [n,3] (step, e, slot), table [E]).
    seed: experts resident before the first step, seed[i] in slot i, last used
    before any step (Betelgeuse news page, section 机制, hot-expert profile
    seeding of the slot pool)."""
    maxsel = max([len(s) for s in steps] + [1])
    sel = np.full((len(steps), maxsel), -1, np.int32)
    for n, s in enumerate(steps):
        sel[n, :len(s)] = s
    if max_miss is None:
        max_miss = len(steps) * maxsel + 1
    out = np.empty((max_miss, 3), np.int32)
    table = np.empty(E, np.int32)
    sd = np.asarray([] if seed is None else seed, np.int32)
    n = lib().oracle_pool_sim(E, S, int(init_full), _ptr(sd) if len(sd) else None, len(sd), len(steps), _ptr(sel),
                              maxsel, _ptr(out), max_miss, _ptr(table))
    if n < 0:
        raise ValueError(f"pool simulation failed ({n})")
    return out[:n].copy(), table
