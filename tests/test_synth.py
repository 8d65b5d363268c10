"""The seeded input generator: determinism, layout sizes, distributions."""
import numpy as np

from quantized_expert_ffn_gemv_gb300 import synth


def test_page_scale_sizes():
    sh = synth.PAGE
    assert sh.matrix_bytes == 589_824
    assert sh.expert_bytes == 1_769_472
    assert sh.E * sh.expert_bytes == 905_969_664
    assert synth.SMALL.matrix_bytes == 147_456 and synth.SMALL.expert_bytes == 442_368


def test_counter_based_slices_are_independent_of_threading():
    sh = synth.SMALL
    a = synth.experts(sh, 3, 0, 8)
    b = np.concatenate([synth.experts(sh, 3, e, e + 1) for e in range(8)])
    assert np.array_equal(a, b)
    assert not np.array_equal(a[:1000], synth.experts(sh, 4, 0, 1)[:1000])


def test_normal_stream_moments():
    out = np.empty(200_000, np.float64)
    synth.lib().synth_normal_f64(synth.lib().synth_key(1, 2, 3, 4, 5), 0, out.size, out.ctypes.data)
    assert abs(out.mean()) < 0.01 and abs(out.std() - 1.0) < 0.01
    # any start offset reproduces the same values
    part = np.empty(101, np.float64)
    synth.lib().synth_normal_f64(synth.lib().synth_key(1, 2, 3, 4, 5), 777, 101, part.ctypes.data)
    assert np.array_equal(part, out[777:878])


def test_router_and_activation_distributions():
    sh = synth.PAGE
    W = synth.router(sh, 0)
    assert abs(W.std() * np.sqrt(sh.H) - 1.0) < 0.01
    x = synth.bf16_to_f32(synth.activations(sh, 0, 0, 64))
    assert abs(x.std() - 1.0) < 0.02
    x2 = synth.activations(sh, 0, 5, 1, sub=np.array([1]))
    assert not np.array_equal(x2[0], synth.activations(sh, 0, 5, 1)[0])


def test_zipf_bias():
    b, perm = synth.zipf_bias(synth.PAGE, 0)
    assert sorted(perm.tolist()) == list(range(512))
    ref = (-1.1 * np.log(1.0 + perm)).astype(np.float32)
    assert np.allclose(b, ref, rtol=0, atol=1e-6)
    assert b[perm.tolist().index(0)] == 0.0


def test_expert_weight_scale():
    sh = synth.SMALL
    blob = synth.experts(sh, 0, 0, 1)
    sc = blob[sh.I * sh.H // 2: sh.I * sh.H // 2 + sh.I * sh.H // 16].view(np.float16).astype(np.float64)
    # scale = amax/7 of 32 N(0, 0.02^2) draws, about 2.07 sigma / 7
    assert 0.004 < sc.mean() < 0.008
