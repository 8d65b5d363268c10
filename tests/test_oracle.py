"""Pins of the CPU oracle against what the definition and mathematics fix.

Each test checks the oracle (moe_oracle.c) against something other than
itself: brute force, closed forms, an independently written numpy dense
path, or the generator's quantizer.  No GPU.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gemv_gb300 import synth
from tests.inputs import codebook_levels, dequant_numpy, expert_mats, resampled_tokens


def silu(z):
    return z / (1.0 + np.exp(-z))


# ---------------------------------------------------------------- top-k


def brute_topk(l, k):
    """The k-subset whose every member ranks before every non-member under
    (logit descending, index ascending); found by enumerating all subsets."""
    E = len(l)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(l[a] > l[b] or (l[a] == l[b] and a < b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    return np.array(found[0], np.int32)


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 13))
    k = int(rng.integers(1, min(4, E) + 1))
    # small integer logits make exact ties common
    l = rng.integers(-3, 4, size=E).astype(np.float64) * 0.5
    idx, w, by_rank, gap = oracle.topk(l, k)
    assert np.array_equal(idx, brute_topk(l, k))
    assert np.array_equal(np.sort(by_rank), idx)
    # rank order: logit descending, index ascending
    for a, b in zip(by_rank[:-1], by_rank[1:]):
        assert l[a] > l[b] or (l[a] == l[b] and a < b)
    # a full stable sort on (-l, index) gives the same set
    order = sorted(range(E), key=lambda e: (-l[e], e))
    assert np.array_equal(np.array(sorted(order[:k]), np.int32), idx)
    if k < E:
        assert gap == pytest.approx(l[order[k - 1]] - l[order[k]], abs=0)


def test_topk_k_equals_E_and_k_one():
    l = np.array([0.3, -1.0, 2.5, 0.3, 7.0])
    idx, w, _, gap = oracle.topk(l, 5)
    assert np.array_equal(idx, np.arange(5)) and math.isinf(gap)
    sm = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
    assert np.allclose(w, sm, rtol=1e-15, atol=0)
    idx, w, _, _ = oracle.topk(l, 1)
    assert idx.tolist() == [4] and w.tolist() == [1.0]


@pytest.mark.parametrize("seed", range(10))
def test_routing_weights_renormalised_softmax(seed):
    rng = np.random.default_rng(100 + seed)
    E, k = 512, 10
    l = rng.normal(size=E) * 2.0 - 1.1 * np.log(1.0 + rng.permutation(E))
    idx, w, _, _ = oracle.topk(l, k)
    assert abs(w.sum() - 1.0) <= 1e-15
    # softmax over all E, then renormalised over the selected k
    p = np.exp(l - l.max())
    p /= p.sum()
    ref = p[idx] / p[idx].sum()
    assert np.allclose(w, ref, rtol=1e-13, atol=0)
    assert np.all(w > 0)


def test_topk_ties_lower_index_wins():
    l = np.array([1.0, 2.0, 2.0, 2.0, 0.0])
    idx, _, by_rank, gap = oracle.topk(l, 2)
    assert idx.tolist() == [1, 2] and by_rank.tolist() == [1, 2] and gap == 0.0


# ---------------------------------------------------------------- dequantization and the quantizer


def test_dequant_matches_independent_decoder():
    rng = np.random.default_rng(7)
    R, K = 48, 128
    nib = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)  # every nibble value
    sc = rng.normal(size=(R, K // 32)).astype(np.float16)
    mat = synth.pack_matrix(nib, sc.view(np.uint16))
    a = oracle.dequant_matrix(mat, R, K)
    b = dequant_numpy(mat, R, K)
    assert np.array_equal(a, b)
    # element 0 of a row is the low nibble of byte 0, element 1 the high one
    n = nib.astype(np.int64)
    assert a[0, 0] == float(sc[0, 0]) * ((n[0, 0] & 15) - 8)
    assert a[0, 1] == float(sc[0, 0]) * ((n[0, 0] >> 4) - 8)
    assert a[3, 37] == float(sc[3, 1]) * ((n[3, 18] >> 4) - 8)


@pytest.mark.parametrize("sigma", [0.02, 1.0, 1e-3])
def test_quantizer_round_trip(sigma):
    rng = np.random.default_rng(11)
    R, K = 64, 256
    w = (rng.normal(size=(R, K)) * sigma).astype(np.float32)
    w[5, 32:64] = 0.0  # an all-zero block
    nib, sc = synth.quantize_rows(w)
    deq = oracle.dequant_matrix(synth.pack_matrix(nib, sc), R, K)
    d = np.repeat(sc.view(np.float16).astype(np.float64), 32, axis=1)
    # |w - d q| <= d/2 (plus one binary32 ulp of w for the rounding of w/d)
    err = np.abs(w.astype(np.float64) - deq)
    assert np.all(err <= d / 2 + np.spacing(np.abs(w)).astype(np.float64) + 1e-300)
    u = np.empty((R, K), np.int64)
    u[:, 0::2] = nib & 15
    u[:, 1::2] = nib >> 4
    q = u - 8
    assert q.min() >= -8 and q.max() <= 7
    # the block maximum maps to +-7
    blocks = np.abs(w.reshape(R, K // 32, 32))
    amax_pos = blocks.argmax(axis=2)
    qb = q.reshape(R, K // 32, 32)
    for r in range(R):
        for b in range(K // 32):
            if blocks[r, b].max() > 0:
                assert abs(qb[r, b, amax_pos[r, b]]) == 7
    # an all-zero block gives d = 0 and q = 0
    assert sc[5, 1] == 0 and np.all(q[5, 32:64] == 0)


def test_scale_is_fp16_of_amax_over_7():
    w = np.zeros((1, 32), np.float32)
    w[0, 3] = -0.7
    nib, sc = synth.quantize_rows(w)
    assert sc.view(np.float16)[0, 0] == np.float16(0.7 / 7)  # numpy rounds f64->f16 RNE
    assert (int(nib[0, 1]) >> 4) - 8 == -7


# ---------------------------------------------------------------- the layer against a dense numpy path


def dense_layer(W_r, bias, blobs, shared, H, I, k, x_bf16, fmt=0):
    """Independent dense float64 evaluation: every matrix fully dequantized
    (numpy decoder), softmax over all experts renormalised over the top k."""
    E = W_r.shape[0]
    x = synth.bf16_to_f32(x_bf16).astype(np.float64)
    l = W_r.astype(np.float64) @ x + (0 if bias is None else bias.astype(np.float64))
    order = sorted(range(E), key=lambda e: (-l[e], e))
    S = sorted(order[:k])
    p = np.exp(l - l.max())
    p /= p.sum()
    wts = p[S] / p[S].sum()
    eb = 3 * (I * H // 2 + I * H // 16)
    y = np.zeros(H)
    for wj, e in zip(wts, S):
        g, u, d = expert_mats(blobs[e * eb:(e + 1) * eb], H, I, fmt)
        y += wj * (d @ (silu(g @ x) * (u @ x)))
    if shared is not None:
        g, u, d = expert_mats(shared, H, I, fmt)
        y += d @ (silu(g @ x) * (u @ x))
    return y, np.array(S, np.int32), wts


@pytest.mark.parametrize("fmt", [0, 1], ids=["linear", "codebook"])
def test_dense_toy_four_experts(fmt):
    """E = 4, k = 4, H = 64, I = 32: the MoE result equals
    sum_e softmax_e FFN_e(x) + FFN_shared(x) on fully dequantized weights,
    in both weight formats."""
    sh = synth.LayerShape(H=64, E=4, k=4, I=32, expert_sigma=0.3, fmt=fmt)
    L = synth.make_layer(sh, layer=900)
    x = synth.activations(sh, 900, 0, 3)
    r = oracle.moe_forward(64, 32, 4, 4, L.W_r, L.bias, L.experts, L.shared, x, fmt=fmt)
    for t in range(3):
        y, S, wts = dense_layer(L.W_r, L.bias, L.experts, L.shared, 64, 32, 4, x[t], fmt)
        assert np.array_equal(r["idx"][t], np.arange(4))
        assert np.allclose(r["w"][t], wts, rtol=1e-13, atol=0)
        assert np.allclose(r["y"][t], y, rtol=1e-12, atol=1e-14)


def test_small_layer_against_numpy_einsum():
    """64 experts top-4 + shared, H 1024, I 256: oracle vs a numpy float64
    einsum over the dequantized matrices of the selected experts."""
    sh = synth.SMALL
    L = synth.make_layer(sh, layer=0)
    x, _ = resampled_tokens(L, 0, 3)
    r = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, x)
    eb = sh.expert_bytes
    xs = synth.bf16_to_f32(x).astype(np.float64)
    for t in range(3):
        S = r["idx"][t]
        mats = [expert_mats(L.experts[e * eb:(e + 1) * eb], sh.H, sh.I) for e in S]
        G = np.stack([m[0] for m in mats])
        U = np.stack([m[1] for m in mats])
        D = np.stack([m[2] for m in mats])
        h = silu(np.einsum("eih,h->ei", G, xs[t])) * np.einsum("eih,h->ei", U, xs[t])
        ye = np.einsum("ehi,ei->eh", D, h)
        g0, u0, d0 = expert_mats(L.shared, sh.H, sh.I)
        y = np.einsum("e,eh->h", r["w"][t], ye) + d0 @ (silu(g0 @ xs[t]) * (u0 @ xs[t]))
        assert np.allclose(r["y"][t], y, rtol=1e-12, atol=1e-14)
        y2, S2, _ = dense_layer(L.W_r, L.bias, L.experts, L.shared, sh.H, sh.I, sh.k, x[t])
        assert np.array_equal(S2, S)


# ---------------------------------------------------------------- closed forms


def test_zero_input_gives_zero_output():
    sh = synth.LayerShape(H=128, E=8, k=2, I=64, zipf_s=1.1)
    L = synth.make_layer(sh, layer=901)
    x = np.zeros((1, 128), np.uint16)
    r = oracle.moe_forward(128, 64, 8, 2, L.W_r, L.bias, L.experts, L.shared, x)
    assert np.all(r["y"] == 0.0)
    assert np.array_equal(r["logits"][0], L.bias.astype(np.float64))


def test_identical_experts_give_twice_one_ffn():
    """All routed experts and the shared one identical: y = 2 FFN(x), whatever
    the routing (the routed weights sum to 1)."""
    sh = synth.LayerShape(H=128, E=8, k=3, I=64)
    L = synth.make_layer(sh, layer=902)
    one = L.experts[:sh.expert_bytes]
    experts = np.tile(one, sh.E)
    x = synth.activations(sh, 902, 0, 2)
    r = oracle.moe_forward(128, 64, 8, 3, L.W_r, None, experts, one, x)
    for t in range(2):
        g, u, d = expert_mats(one, 128, 64)
        xs = synth.bf16_to_f32(x[t]).astype(np.float64)
        y1 = d @ (silu(g @ xs) * (u @ xs))
        assert np.allclose(r["y"][t], 2 * y1, rtol=1e-12, atol=1e-15)


def test_zero_shared_expert_gives_routed_sum():
    sh = synth.LayerShape(H=128, E=8, k=2, I=64)
    L = synth.make_layer(sh, layer=903)
    zero = np.zeros_like(L.shared)  # every scale 0 -> every weight 0
    x = synth.activations(sh, 903, 0, 2)
    a = oracle.moe_forward(128, 64, 8, 2, L.W_r, None, L.experts, zero, x)
    b = oracle.moe_forward(128, 64, 8, 2, L.W_r, None, L.experts, None, x)
    assert np.array_equal(a["y"], b["y"])
    eb = sh.expert_bytes
    for t in range(2):
        xs = synth.bf16_to_f32(x[t]).astype(np.float64)
        ref = np.zeros(128)
        for wj, e in zip(a["w"][t], a["idx"][t]):
            ref += wj * oracle.expert(L.experts[e * eb:(e + 1) * eb], 128, 64, xs)[0]
        assert np.allclose(a["y"][t], ref, rtol=1e-13, atol=1e-16)


def test_hand_built_expert_closed_form():
    """One block of constant weights: W_g = 1 (d=1, q=1), W_u = 1 (d=0.5,
    q=2), W_d = 1/64 (d=1/64, q=1); x = e_0 gives g = u = 1 for every row,
    h = silu(1) = 1/(1+e^-1), and y_r = I * h / 64."""
    H, I = 64, 64
    def const(R, K, q, d):
        nib = np.full((R, K // 2), (q + 8) | ((q + 8) << 4), np.uint8)
        sc = np.full((R, K // 32), np.float16(d)).view(np.uint16)
        return synth.pack_matrix(nib, sc)
    blob = np.concatenate([const(I, H, 1, 1.0), const(I, H, 2, 0.5), const(H, I, 1, 1.0 / 64)])
    x = np.zeros(H)
    x[0] = 1.0
    y, h = oracle.expert(blob, H, I, x)
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(h, s1, rtol=1e-15, atol=0)
    assert np.allclose(y, I * s1 / 64, rtol=1e-15, atol=0)
    # x = 2 e_0 + e_1: g = u = 3, h = 3 * 3 / (1 + e^-3)
    x[1] = 1.0
    x[0] = 2.0
    y, h = oracle.expert(blob, H, I, x)
    assert np.allclose(h, 9.0 / (1.0 + math.exp(-3.0)), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- RMSNorm and residual


def test_rmsnorm_closed_forms():
    H = 256
    c = np.float32(0.75)
    x = np.full(H, synth.f32_to_bf16(np.array([c]))[0], np.uint16)
    xh, xf = oracle.rmsnorm(x, eps=1e-6)
    expect = 0.75 / math.sqrt(0.75 ** 2 + 1e-6)
    assert np.allclose(xf, expect, rtol=1e-15)
    assert np.all(xh == oracle.to_bf16(np.array([expect]))[0])
    z, zf = oracle.rmsnorm(np.zeros(H, np.uint16))
    assert np.all(zf == 0.0) and np.all(z == 0)
    # alternating +-a: mean of squares a^2
    v = np.where(np.arange(H) % 2 == 0, 2.0, -2.0).astype(np.float32)
    xh, xf = oracle.rmsnorm(synth.f32_to_bf16(v))
    assert np.allclose(np.abs(xf), 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-15)


def test_bf16_rounding_is_round_to_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -9), 1e-40, 3.0e38])
    out = oracle.to_bf16(v)
    assert out[0] == 0x3F80 and out[1] == 0x3F82 and out[2] == 0xBF80
    ref = synth.f32_to_bf16(v.astype(np.float32))
    assert out[3] == ref[3] and out[4] == ref[4]
    rng = np.random.default_rng(3)
    r = rng.normal(size=10000).astype(np.float32).astype(np.float64)  # exact in binary32
    assert np.array_equal(oracle.to_bf16(r), synth.f32_to_bf16(r.astype(np.float32)))


def test_residual_exact_sum_rounded_once():
    a = synth.f32_to_bf16(np.array([1.0, 256.0, -3.0], np.float32))
    b = synth.f32_to_bf16(np.array([2.0 ** -8, 1.0, 3.0], np.float32))
    out = oracle.residual(a, b)
    # 1 + 2^-8 ties to 1.0; 257 is halfway between 256 and 258 -> 256; -3+3 = 0
    assert out.tolist() == [0x3F80, 0x4380, 0x0000]


# ---------------------------------------------------------------- forced selection and the gap


def numpy_layer(L, sh, x_u16, sel):
    """Independent float64 layer for a given selection: softmax of the
    selected logits (numpy router), dense expert maths from the numpy decoder."""
    xs = synth.bf16_to_f32(x_u16).astype(np.float64)
    l = L.W_r.astype(np.float64) @ xs + (0.0 if L.bias is None else L.bias.astype(np.float64))
    ls = l[sel]
    w = np.exp(ls - ls.max())
    w /= w.sum()
    eb = sh.expert_bytes
    y = np.zeros(sh.H)
    for wj, e in zip(w, sel):
        g, u, d = expert_mats(L.experts[e * eb:(e + 1) * eb], sh.H, sh.I)
        y += wj * (d @ (silu(g @ xs) * (u @ xs)))
    g, u, d = expert_mats(L.shared, sh.H, sh.I)
    return y + d @ (silu(g @ xs) * (u @ xs)), w, l


def test_forced_selection_and_gap():
    """force= replaces the selection (weights: softmax over the forced set);
    forcing the oracle's own choice changes nothing; gap is the distance
    between the k-th and (k+1)-th largest logits."""
    sh = synth.LayerShape(H=128, E=8, k=3, I=64, zipf_s=1.1)
    L = synth.make_layer(sh, layer=905)
    x = synth.activations(sh, 905, 0, 3)
    r = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, x)
    same = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, x, force=r["idx"])
    for key in ("y", "idx", "w"):
        assert np.array_equal(r[key], same[key]), key
    forced = np.tile(np.array([1, 4, 7], np.int32), (3, 1))
    f = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, L.W_r, L.bias, L.experts, L.shared, x, force=forced)
    for t in range(3):
        y, w, l = numpy_layer(L, sh, x[t], forced[t])
        assert np.array_equal(f["idx"][t], forced[t])
        assert np.allclose(f["w"][t], w, rtol=1e-12, atol=0)
        assert np.allclose(f["y"][t], y, rtol=1e-11, atol=1e-14)
        srt = np.sort(l)[::-1]
        assert r["gap"][t] == pytest.approx(srt[sh.k - 1] - srt[sh.k], abs=1e-12)
        assert r["gap"][t] >= 0.0


def test_all_logits_tied_picks_the_lowest_indices_with_zero_gap():
    """Every router row the same and no bias: all logits tie, the selection
    is experts 0..k-1, the weights are 1/k and the gap is exactly 0."""
    sh = synth.LayerShape(H=128, E=8, k=3, I=64)
    L = synth.make_layer(sh, layer=906)
    W = np.tile(L.W_r[:1], (sh.E, 1))
    x = synth.activations(sh, 906, 0, 2)
    r = oracle.moe_forward(sh.H, sh.I, sh.E, sh.k, W, None, L.experts, L.shared, x)
    assert np.array_equal(r["idx"], np.tile(np.arange(sh.k, dtype=np.int32), (2, 1)))
    assert np.all(r["w"] == 1.0 / 3.0) or np.allclose(r["w"], 1.0 / 3.0, rtol=1e-15, atol=0)
    assert np.all(r["gap"] == 0.0)


# ---------------------------------------------------------------- the codebook weight format


def test_codebook_levels_are_the_normal_quantiles():
    lv = oracle.levels()
    ref = codebook_levels()
    assert np.array_equal(lv, ref)
    assert np.all(np.diff(lv) > 0) and np.array_equal(lv, -lv[::-1]) and lv[-1] == 127
    # every level is an integer, exact in binary16 (what the GPU multiplies)
    assert np.array_equal(lv.astype(np.float16).astype(np.float64), lv)


def test_codebook_dequant_matches_independent_decoder():
    rng = np.random.default_rng(17)
    R, K = 32, 128
    nib = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)  # every nibble value
    sc = (rng.normal(size=(R, K // 32)) * 0.01).astype(np.float16)
    mat = synth.pack_matrix(nib, sc.view(np.uint16))
    a = oracle.dequant_matrix(mat, R, K, fmt=1)
    assert np.array_equal(a, dequant_numpy(mat, R, K, fmt=1))
    assert a[2, 1] == float(sc[2, 0]) * codebook_levels()[nib[2, 0] >> 4]


@pytest.mark.parametrize("sigma", [0.02, 1.0])
def test_codebook_quantizer_picks_the_nearest_level(sigma):
    """The generator's codebook quantizer: d = fp16(amax / 127), each element
    the nearest level of w / d (ties to the lower index, re-derived here by
    brute force); dequantized error within half the widest level gap."""
    rng = np.random.default_rng(19)
    R, K = 32, 256
    w = (rng.normal(size=(R, K)) * sigma).astype(np.float32)
    w[3, 64:96] = 0.0
    nib, sc = synth.quantize_rows(w, fmt=1)
    lv = codebook_levels()
    d = sc.view(np.float16).astype(np.float64)
    assert np.array_equal(sc.view(np.float16),
                          (np.abs(w.reshape(R, K // 32, 32)).max(axis=2).astype(np.float64) / 127).astype(np.float16))
    u = np.empty((R, K), np.int64)
    u[:, 0::2] = nib & 15
    u[:, 1::2] = nib >> 4
    dd = np.repeat(d, 32, axis=1)
    t = np.where(dd > 0, w.astype(np.float64) / np.where(dd > 0, dd, 1), 0)
    want = np.argmin(np.abs(t[..., None] - lv[None, None, :]), axis=2)  # first minimum: the lower index
    nz = dd > 0
    assert np.array_equal(u[nz], want[nz])
    assert np.all(u[~nz] == 8)
    deq = oracle.dequant_matrix(synth.pack_matrix(nib, sc), R, K, fmt=1)
    gap = np.max(np.diff(lv)) / 2
    assert np.all(np.abs(w.astype(np.float64) - deq) <= dd * gap + 1e-30)


def test_codebook_closed_forms():
    """x = 0 gives y = 0; identical experts give the same output whatever the routing."""
    sh = synth.LayerShape(H=128, E=8, k=2, I=64, fmt=1)
    L = synth.make_layer(sh, layer=31)
    x0 = np.zeros((1, 128), np.uint16)
    r = oracle.moe_forward(128, 64, 8, 2, L.W_r, L.bias, L.experts, L.shared, x0, fmt=1)
    assert np.all(r["y"] == 0.0)
    eb = sh.expert_bytes
    one = L.experts[:eb]
    same = np.tile(one, 8)
    x = synth.activations(sh, 31, 0, 2)
    a = oracle.moe_forward(128, 64, 8, 2, L.W_r, None, same, one, x, fmt=1)
    for t in range(2):
        ya, _ = oracle.expert(one, 128, 64, synth.bf16_to_f32(x[t]).astype(np.float64), fmt=1)
        assert np.allclose(a["y"][t], 2 * ya, rtol=1e-12, atol=1e-15)
