"""The C-ABI library without a GPU: exports, argument checks, and the
lossless repack into the GPU layout (emulating the kernel's fragment
dequantization in numpy)."""
import os
import re

import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    build.build_cuda()
    from quantized_expert_ffn_gemv_gb300 import moe as m
    return m


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(moe):
    names = declared_symbols()
    assert "moe_forward" in names and "moe_layer_create" in names and len(names) >= 12
    lib = moe.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(moe.EXPORTS) == names


def test_status_strings(moe):
    for code in range(9):
        assert moe.status_string(code)
    assert moe.status_string(6).startswith("timed out")


def test_create_rejects_bad_descriptions_before_touching_the_gpu(moe):
    import ctypes as C
    h = C.c_void_p()
    assert moe.lib().moe_layer_create(None, C.byref(h)) == 1
    d = moe.LayerDesc(hidden=1024, n_experts=64, top_k=4, n_shared=1, inter=256, qblock=64, max_tokens=1)
    assert moe.lib().moe_layer_create(C.byref(d), C.byref(h)) == 2  # qblock must be 32
    d.qblock = 32
    d.hidden = 1000
    assert moe.lib().moe_layer_create(C.byref(d), C.byref(h)) in (1, 2)
    d.hidden = 1024
    d.max_tokens = 8193  # above the largest prefill chunk
    assert moe.lib().moe_layer_create(C.byref(d), C.byref(h)) == 2
    d.max_tokens, d.hidden = 65, 192  # prefill needs H % 128 == 0
    assert moe.lib().moe_layer_create(C.byref(d), C.byref(h)) == 2
    d.hidden = 1024
    assert h.value is None
    assert moe.lib().moe_forward(None, None, 1, None, None, None, None) == 1
    assert moe.lib().moe_forward_norm(None, None, None, 1, 1e-6, None, None, None, None, None, None) == 1
    assert moe.lib().moe_set_miss_service(None, 1) == 1
    assert moe.lib().moe_slot_pool_seed(None, None, 0) == 1
    assert moe.expert_bytes(2048, 512) == 1_769_472


@pytest.mark.parametrize("shape", [synth.SMALL, synth.PAGE, synth.LayerShape(H=128, E=4, k=2, I=64)])
def test_repack_round_trip_is_byte_identical(moe, shape):
    blob = synth.experts(shape, 7, 0, 1)
    gpu = moe.repack_expert(blob, shape.H, shape.I)
    assert gpu.nbytes == blob.nbytes
    assert np.array_equal(moe.unpack_expert(gpu, shape.H, shape.I), blob)
    # every nibble value, including u = 0 (q = -8), survives
    rnd = np.random.default_rng(1).integers(0, 256, size=blob.nbytes, dtype=np.uint8)
    assert np.array_equal(moe.unpack_expert(moe.repack_expert(rnd, shape.H, shape.I), shape.H, shape.I), rnd)


def emulate_a_fragments(gpu, H, I, which):
    """Rebuild a dense matrix from the GPU layout the way the kernel does:
    per strip, super-tile and lane, the magic-exponent fp16 dequantization of
    each word into the m16n8k16 A fragment, times the block scale."""
    if which in ("gate", "up"):
        R, K = I, H
        stride, nib_off = 18 * H, (0 if which == "gate" else 9 * H)
        sc_off, base = nib_off + 8 * H, 0
    else:
        R, K = H, I
        stride, nib_off, sc_off, base = 9 * I, 0, 8 * I, (I // 16) * 18 * H
    out = np.zeros((R, K))
    f16 = np.float16
    for s in range(R // 16):
        strip = gpu[base + s * stride:]
        for st in range(K // 64):
            words = strip[nib_off + st * 512:nib_off + st * 512 + 512].view(np.uint32).reshape(32, 4)
            scs = strip[sc_off + st * 64:sc_off + st * 64 + 64].view(np.float16).reshape(8, 4).astype(np.float64)
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                for kt in range(4):
                    w = int(words[lane, kt])
                    def halves(v):
                        return (np.array([v & 0xFFFF, v >> 16], np.uint16)).view(np.float16)
                    lo0 = halves((w & 0x000F000F) | 0x64006400) - f16(1032)
                    hi0 = halves((w & 0x00F000F0) | 0x64006400) * f16(1 / 16) - f16(72)
                    w8 = w >> 8
                    lo1 = halves((w8 & 0x000F000F) | 0x64006400) - f16(1032)
                    hi1 = halves((w8 & 0x00F000F0) | 0x64006400) * f16(1 / 16) - f16(72)
                    k0 = 64 * st + 16 * kt
                    blk = kt // 2
                    dg, dg8 = scs[g, 2 * blk], scs[g, 2 * blk + 1]
                    r0, r8 = 16 * s + g, 16 * s + g + 8
                    # PTX m16n8k16 A fragment: a0 (g, 2t..), a1 (g+8, 2t..), a2 (g, 2t+8..), a3 (g+8, 2t+8..)
                    out[r0, k0 + 2 * t:k0 + 2 * t + 2] = lo0.astype(np.float64) * dg
                    out[r8, k0 + 2 * t:k0 + 2 * t + 2] = lo1.astype(np.float64) * dg8
                    out[r0, k0 + 2 * t + 8:k0 + 2 * t + 10] = hi0.astype(np.float64) * dg
                    out[r8, k0 + 2 * t + 8:k0 + 2 * t + 10] = hi1.astype(np.float64) * dg8
    return out


def test_fragment_dequantization_reproduces_the_matrices(moe):
    sh = synth.LayerShape(H=128, E=2, k=1, I=64)
    rnd = np.random.default_rng(5)
    blob = synth.experts(sh, 3, 0, 1)
    # overwrite nibbles with every value 0..15 to cover q = -8 .. 7
    mb = sh.matrix_bytes
    for m in range(3):
        R, K = (sh.I, sh.H) if m < 2 else (sh.H, sh.I)
        blob[m * mb:m * mb + R * K // 2] = rnd.integers(0, 256, size=R * K // 2, dtype=np.uint8)
    gpu = moe.repack_expert(blob, sh.H, sh.I)
    for m, which in enumerate(("gate", "up", "down")):
        R, K = (sh.I, sh.H) if m < 2 else (sh.H, sh.I)
        ref = oracle.dequant_matrix(blob[m * mb:(m + 1) * mb], R, K)
        assert np.array_equal(emulate_a_fragments(gpu, sh.H, sh.I, which), ref), which


def test_binding_fails_loudly_without_the_library(moe, monkeypatch, tmp_path):
    """No CPU fallback: with the CUDA library missing every call raises."""
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(build, "CUDA_LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        moe.lib()
    with pytest.raises(RuntimeError, match="not built"):
        moe.expert_bytes(2048, 512)


def test_binding_checks_forward_tensors_before_the_library(moe, monkeypatch):
    """Shapes, dtypes, layouts and devices of forward / forward_norm /
    residual_rmsnorm are checked in the binding: a mismatch raises ValueError
    and never reaches the library (which here would fail the test)."""
    import torch

    def no_library():
        raise AssertionError("the library was called")

    monkeypatch.setattr(moe, "lib", no_library)
    sh = synth.SMALL
    layer = moe.MoeLayer.__new__(moe.MoeLayer)
    layer.shape, layer.device, layer.h = sh, torch.device("cuda", 0), None
    T, H, k = 3, sh.H, sh.k
    bf = torch.bfloat16
    x = torch.zeros(T, H, dtype=bf)
    good = dict(x=x, y=torch.zeros(T, H, dtype=bf), topk_idx=torch.zeros(T, k, dtype=torch.int32),
                topk_w=torch.zeros(T, k, dtype=torch.float32))
    bad = [
        dict(good, y=torch.zeros(T - 1, H, dtype=bf)),                          # y too short
        dict(good, y=torch.zeros(T, H, dtype=torch.float16)),                   # wrong dtype
        dict(good, topk_idx=torch.zeros(T, k + 1, dtype=torch.int32)),          # wrong k
        dict(good, topk_w=torch.zeros(T, k, dtype=torch.float64)),              # wrong dtype
        dict(good, x=torch.zeros(H, T, dtype=bf).t()),                          # not contiguous
        dict(good, x=torch.zeros(T, H + 8, dtype=bf), y=torch.zeros(T, H + 8, dtype=bf)),  # wrong H
        good,                                                                   # host tensors
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            layer.forward(**kw)
        with pytest.raises(ValueError):
            layer.forward_norm(kw["x"], None, 1e-6, None, kw["y"], torch.zeros_like(kw["y"]), kw["topk_idx"],
                               kw["topk_w"])
    with pytest.raises(ValueError):
        moe.residual_rmsnorm(x, torch.zeros(T, H + 8, dtype=bf), 1e-6, None, torch.zeros_like(x))
    with pytest.raises(ValueError):
        moe.residual_rmsnorm(x, None, 1e-6, None, torch.zeros_like(x))  # host tensors
