"""Test inputs: the seeded generator plus the near-tie resampling rule.

Tokens whose k-th and (k+1)-th largest router logits (binary64, from the
oracle) differ by less than GAP are redrawn from the next sub-seed, so that
any summation order with an error below GAP/2 selects the same experts.
"""
import numpy as np

import oracle
from quantized_expert_ffn_gemv_gb300 import synth

GAP = 1e-3


def resampled_tokens(layer, t0, T, stream=0, gap=GAP, max_redraw=64):
    """(x bf16 [T,H], sub [T]) with every token's top-k boundary gap >= gap."""
    sh = layer.shape
    sub = np.zeros(T, np.int32)
    x = synth.activations(sh, layer.index, t0, T, stream=stream, sub=sub)
    for _ in range(max_redraw):
        l = oracle.router_logits(layer.W_r, layer.bias, x)
        bad = []
        for t in range(T):
            srt = np.sort(l[t])[::-1]
            if sh.k < sh.E and srt[sh.k - 1] - srt[sh.k] < gap:  # k = E: no boundary to guard
                bad.append(t)
        if not bad:
            return x, sub
        for t in bad:
            sub[t] += 1
            x[t] = synth.activations(sh, layer.index, t0 + t, 1, stream=stream, sub=sub[t:t + 1])[0]
    raise RuntimeError("could not resample near-ties")


def codebook_levels():
    """The codebook format's 16 levels from their definition: the standard
    normal's quantiles at (u + 1/2)/16, scaled so the outermost is 127,
    rounded to integers (scipy's inverse normal CDF, independent of the
    oracle's and the library's own tables)."""
    from scipy.stats import norm
    z = norm.ppf((np.arange(16) + 0.5) / 16)
    return np.round(127 * z / z[-1])


def dequant_numpy(mat, R, K, fmt=0):
    """Independent numpy decoder of one packed matrix (nibble plane + scale plane)."""
    mat = np.asarray(mat, np.uint8)
    nib = mat[:R * K // 2].reshape(R, K // 2)
    sc = mat[R * K // 2:R * K // 2 + R * K // 16].view(np.float16).reshape(R, K // 32).astype(np.float64)
    u = np.empty((R, K), np.int64)
    u[:, 0::2] = nib & 15
    u[:, 1::2] = nib >> 4
    v = codebook_levels()[u] if fmt == 1 else (u - 8)
    return v * np.repeat(sc, 32, axis=1)


def expert_mats(blob, H, I, fmt=0):
    mb = I * H // 2 + I * H // 16
    b = np.asarray(blob, np.uint8)
    return (dequant_numpy(b[:mb], I, H, fmt), dequant_numpy(b[mb:2 * mb], I, H, fmt),
            dequant_numpy(b[2 * mb:3 * mb], H, I, fmt))
