"""The seeded input generator: determinism, distribution and fp16 rounding."""
import numpy as np

import synth
from synth.configs import TINY, TWO_B, GEMV_SHAPES

MASK = (1 << 64) - 1


def test_splitmix64_stream_matches_counter_form():
    # Sequential SplitMix64 from state s yields mix(s + G), mix(s + 2G), ...; the counter form used for
    # random access must give the same numbers as the stateful generator started at the stream base.
    L = synth.lib()
    import ctypes
    st = ctypes.c_uint64(12345)
    seq = [L.synth_splitmix64_next(ctypes.byref(st)) for _ in range(5)]
    st2 = ctypes.c_uint64(12345)
    assert seq == [L.synth_splitmix64_next(ctypes.byref(st2)) for _ in range(5)]
    assert len(set(seq)) == 5
    # counter form: draws of one stream are distinct and depend on (seed, tensor id)
    a = [L.synth_draw(1, 7, i) for i in range(4)]
    b = [L.synth_draw(1, 8, i) for i in range(4)]
    c = [L.synth_draw(2, 7, i) for i in range(4)]
    assert a != b and a != c and len(set(a)) == 4


def test_normal_moments_and_determinism():
    x = synth.normal_f32(3, 11, 1 << 20, 0.0, 1.0)
    assert abs(float(x.mean())) < 5e-3
    assert abs(float(x.std()) - 1.0) < 5e-3
    # fourth moment of a standard normal is 3
    assert abs(float((x.astype(np.float64) ** 4).mean()) - 3.0) < 0.05
    np.testing.assert_array_equal(x, synth.normal_f32(3, 11, 1 << 20, 0.0, 1.0))
    # the element stream does not depend on how many elements are requested
    np.testing.assert_array_equal(x[:1000], synth.normal_f32(3, 11, 1000, 0.0, 1.0))


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 0.02,
        rng.standard_normal(20000).astype(np.float32) * 1e-5,      # subnormal range
        (rng.standard_normal(20000) * 3e4).astype(np.float32),     # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -24,
                  1.5 * 2.0 ** -24, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11], dtype=np.float32),
    ])
    L = synth.lib()
    mine = np.array([L.synth_f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_f16_generation_equals_rounded_f32():
    a16 = synth.normal_f16(5, 9, 50000, 0.0, 0.02)
    a32 = synth.normal_f32(5, 9, 50000, 0.0, 0.02)
    np.testing.assert_array_equal(a16, a32.astype(np.float16).view(np.uint16))


def test_tokens_uniform():
    t = synth.tokens(1, 200000, 32000)
    assert t.min() >= 0 and t.max() < 32000
    counts = np.bincount(t // 1000, minlength=32)
    assert counts.min() > 0.9 * 200000 / 32


def test_model_shapes_and_gains():
    w = synth.model_weights(TINY)
    assert w["embed"].shape == (4096, 256) and w["lm_head"].shape == (4096, 256)
    lay = w["layers"][1]
    assert lay["wq"].shape == (256, 256) and lay["w_down"].shape == (256, 704)
    assert (w["final_norm"] == 0x3C00).all() and (lay["attn_norm"] == 0x3C00).all()
    s = synth.as_f32(lay["w_up"]).std()
    assert abs(s - 0.02) < 0.001


def test_byte_model_of_the_2b_config():
    # L*(d(Hq dh + 2 Hkv dh) + d Hq dh + 3 d F) + V d, in fp16 bytes
    assert TWO_B.weight_bytes_per_token() == 3_899_392_000
    assert TWO_B.kv_bytes_per_token(128) == 51_200 * 128
    assert len(GEMV_SHAPES) == 25 and GEMV_SHAPES[7].seed == 1000 + 5 * 1 + 2
