"""The seeded input generator: reproducible, thread-count independent, right moments."""
import numpy as np

import synthetic


def test_counter_based_streams_are_reproducible():
    a = synthetic.normal_bf16((1000, 37), seed=0, stream=3, sigma=1.0)
    b = synthetic.normal_bf16((1000, 37), seed=0, stream=3, sigma=1.0)
    c = synthetic.normal_bf16((1000, 37), seed=0, stream=4, sigma=1.0)
    np.testing.assert_array_equal(a, b)
    assert np.mean(a == c) < 0.01
    # a prefix of a longer fill is the shorter fill (element n depends only on n)
    long = synthetic.normal_bf16((5000, 37), seed=0, stream=3, sigma=1.0)
    np.testing.assert_array_equal(long.ravel()[: a.size], a.ravel())


def test_normal_moments_and_scale():
    v = synthetic.bf16_bits_to_f32(synthetic.normal_bf16((2_000_000,), seed=1, stream=9, sigma=0.02))
    assert abs(v.mean()) < 1e-4
    assert abs(v.std() - 0.02) < 2e-4
    assert abs(np.mean(np.abs(v) < 0.02) - 0.6827) < 3e-3


def test_bf16_rounding_helpers():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-5], np.float32)
    bits = synthetic.f32_to_bf16_bits(x)
    back = synthetic.bf16_bits_to_f32(bits)
    # 1.00390625 is halfway between 1 and 1+2^-7: ties to even -> 1.0
    np.testing.assert_array_equal(back[:4], np.array([1.0, 1.0, 1.0078125, -2.5], np.float32))
    assert abs(back[4] - 3.0e-5) <= 2 ** -9 * 3.0e-5


def test_zipf_bias_skews_load():
    wl = synthetic.Workload("zipf_T512_H64_I64_E64_k4", 512, 64, 64, 64, 4, zipf_s=1.2, router_std=0.02 * 8)
    inp = synthetic.make_inputs(wl, want=("x", "logits"))
    top1 = np.argmax(inp["logits"], axis=1)
    counts = np.bincount(top1, minlength=64)
    assert counts.max() > 0.3 * wl.T  # one expert dominates under the bias
