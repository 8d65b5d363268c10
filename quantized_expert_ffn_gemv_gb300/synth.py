"""Seeded synthetic inputs (weights, router bias, activations).

Marshalling for csrc/synth.c, which holds only the draws and the 4-bit block
quantizer that writes the canonical packed expert blob; none of the layer's
arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle take
their inputs from here.

Workload shapes follow the MoE layer of Qwen3.8-Flash-Next-style decode
(Betelgeuse news page, section 机制: 48 layers, 512 routed experts per
layer, top-10 routed plus 1 shared expert per token).
"""
import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

MASTER_SEED = 0x5EED2026
TAG_ROUTED, TAG_SHARED = 3, 4

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build_synth())
        u64, i64, p = C.c_uint64, C.c_int64, C.c_void_p
        _lib.synth_key.argtypes = [u64] * 5
        _lib.synth_key.restype = u64
        _lib.synth_normal_f64.argtypes = [u64, u64, u64, p]
        _lib.synth_quantize_rows.argtypes = [p, i64, i64, p, p]
        _lib.synth_quantize_rows_cb.argtypes = [p, i64, i64, p, p]
        _lib.synth_matrix_bytes.argtypes = [i64, i64]
        _lib.synth_matrix_bytes.restype = i64
        _lib.synth_expert_bytes.argtypes = [i64, i64]
        _lib.synth_expert_bytes.restype = i64
        _lib.synth_experts.argtypes = [u64, u64, u64, i64, i64, i64, i64, C.c_double, C.c_int, p, C.c_int]
        _lib.synth_experts.restype = C.c_int
        _lib.synth_router.argtypes = [u64, u64, i64, i64, p]
        _lib.synth_zipf_bias.argtypes = [u64, u64, i64, C.c_double, p, p]
        _lib.synth_x_bf16.argtypes = [u64, u64, u64, i64, i64, i64, p, p]
        _lib.synth_det_log.argtypes = [C.c_double]
        _lib.synth_det_log.restype = C.c_double
        _lib.synth_f64_to_f16.argtypes = [C.c_double]
        _lib.synth_f64_to_f16.restype = C.c_uint16
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


@dataclass(frozen=True)
class LayerShape:
    """H hidden, E routed experts, k routed per token, I expert intermediate."""
    H: int
    E: int
    k: int
    I: int
    zipf_s: float = 0.0      # 0: no router bias
    expert_sigma: float = 0.02
    fmt: int = 0             # weight format: 0 linear 4-bit (d * (u - 8)), 1 codebook (d * C[u])

    @property
    def matrix_bytes(self):
        return int(lib().synth_matrix_bytes(self.I, self.H))

    @property
    def expert_bytes(self):
        return int(lib().synth_expert_bytes(self.H, self.I))


# single layer, 64 experts top-4 (+1 shared), the small parity shape
SMALL = LayerShape(H=1024, E=64, k=4, I=256)
# single layer at page scale: 512 experts top-10 (+1 shared), Zipf(1.1) router bias
PAGE = LayerShape(H=2048, E=512, k=10, I=512, zipf_s=1.1)


def threads():
    return max(1, min(64, os.cpu_count() or 1))


def experts(shape, layer, e0=0, e1=None, seed=MASTER_SEED, tag=TAG_ROUTED, out=None):
    """Canonical blobs of experts [e0, e1) as a flat uint8 array (or into `out`)."""
    e1 = shape.E if e1 is None else e1
    n = e1 - e0
    if out is None:
        out = np.empty(n * shape.expert_bytes, np.uint8)
    assert out.nbytes >= n * shape.expert_bytes and out.flags.c_contiguous
    rc = lib().synth_experts(seed, layer, tag, shape.H, shape.I, e0, e1, shape.expert_sigma, shape.fmt, _p(out),
                             threads())
    if rc != 0:
        raise RuntimeError(f"synth_experts failed ({rc})")
    return out


def shared_expert(shape, layer, seed=MASTER_SEED):
    return experts(shape, layer, 0, 1, seed=seed, tag=TAG_SHARED)


def router(shape, layer, seed=MASTER_SEED):
    W = np.empty((shape.E, shape.H), np.float32)
    lib().synth_router(seed, layer, shape.E, shape.H, _p(W))
    return W


def zipf_bias(shape, layer, seed=MASTER_SEED):
    """(bias float32 [E], permutation int32 [E]); None, None without a Zipf exponent."""
    if shape.zipf_s == 0.0:
        return None, None
    b = np.empty(shape.E, np.float32)
    perm = np.empty(shape.E, np.int32)
    lib().synth_zipf_bias(seed, layer, shape.E, shape.zipf_s, _p(b), _p(perm))
    return b, perm


def activations(shape, layer, t0, T, stream=0, sub=None, seed=MASTER_SEED):
    """T tokens of N(0,1) bf16 activations (uint16 bit patterns) [T, H].

    sub[t] selects the resample draw of token t0+t (0 = first draw)."""
    x = np.empty((T, shape.H), np.uint16)
    s = None if sub is None else np.ascontiguousarray(sub, np.int32)
    lib().synth_x_bf16(seed, layer, stream, t0, T, shape.H, _p(s), _p(x))
    return x


def quantize_rows(w, fmt=0):
    """Quantize float32 [R, K] into (nibbles uint8 [R, K/2], scales uint16 [R, K/32])
    in weight format fmt (0 linear 4-bit, 1 codebook)."""
    w = np.ascontiguousarray(w, np.float32)
    R, K = w.shape
    nib = np.empty((R, K // 2), np.uint8)
    sc = np.empty((R, K // 32), np.uint16)
    (lib().synth_quantize_rows_cb if fmt == 1 else lib().synth_quantize_rows)(_p(w), R, K, _p(nib), _p(sc))
    return nib, sc


def pack_matrix(nib, scales):
    """Canonical packed bytes of one matrix from its planes."""
    return np.concatenate([np.ascontiguousarray(nib, np.uint8).ravel(),
                           np.ascontiguousarray(scales, np.uint16).view(np.uint8).ravel()])


@dataclass
class Layer:
    """One synthetic layer: router, bias, routed blobs (flat), shared blob."""
    shape: LayerShape
    index: int
    W_r: np.ndarray
    bias: np.ndarray
    experts: np.ndarray
    shared: np.ndarray


def make_layer(shape, layer=0, seed=MASTER_SEED, experts_out=None):
    b, _ = zipf_bias(shape, layer, seed)
    return Layer(shape, layer, router(shape, layer, seed), b,
                 experts(shape, layer, seed=seed, out=experts_out), shared_expert(shape, layer, seed))


def bf16_to_f32(x):
    return (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v):
    """Round float32 to bf16 (RNE) bit patterns; finite inputs."""
    u = np.ascontiguousarray(v, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
