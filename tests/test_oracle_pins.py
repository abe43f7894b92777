"""Pins of the CPU oracle against facts that do not come from the oracle itself: the binary16 format as
numpy implements it, brute-force fp64 matrix products, closed forms of RMSNorm, RoPE, softmax attention
and SiLU, and whole-model special cases that reduce to library routines or to a simpler model.
"""
import dataclasses

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth
from synth.configs import TINY, TINY_DECODE, ModelConfig


def small_cfg(**kw):
    base = dict(name="pin", n_layers=1, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
                vocab=128, seed=42, gain_std=0.05)
    base.update(kw)
    return ModelConfig(**base)


def f16(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32(bits):
    return synth.as_f32(bits)


# ---- binary16 --------------------------------------------------------------------------------------

def test_half_decode_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    mine = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(mine[finite], ref[finite])
    assert np.array_equal(np.isnan(mine), np.isnan(ref)) and np.array_equal(np.isinf(mine), np.isinf(ref))


def test_half_encode_matches_numpy_rne():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000), rng.standard_normal(5000) * 1e-6,
                        rng.standard_normal(5000) * 4e4,
                        # exact ties between neighbouring halves, both parities, normal and subnormal
                        (np.arange(1024, 1100) + 0.5) * 2.0 ** -10, (np.arange(0, 60) + 0.5) * 2.0 ** -24,
                        [0.0, -0.0, 65504.0, 65519.0, 65520.0, 7e4, 2.0 ** -25, 3 * 2.0 ** -26]])
    mine = np.array([oracle.double_to_half(float(x)) for x in v], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


# ---- GEMV: brute force in fp64 ---------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 1), (1, 33), (17, 1), (5, 7), (17, 33), (64, 256), (300, 2560)])
def test_gemv_against_fp64_matmul(M, K):
    W = synth.normal_f16(7, M * 1000 + K, (M, K), 0.0, 1.0 / np.sqrt(K))
    x = synth.normal_f32(7, 99, K, 0.0, 1.0)
    y64 = f32(W).astype(np.float64) @ x.astype(np.float64)
    y = oracle.gemv(W, x, 32)
    absdot = np.abs(f32(W).astype(np.float64)) @ np.abs(x.astype(np.float64))
    assert np.max(np.abs(y - y64)) <= 1e-3 * max(np.max(np.abs(y64)), 1e-30)
    assert np.all(np.abs(y - y64) <= 1e-3 * absdot + 1e-6)
    np.testing.assert_allclose(oracle.gemv(W, x.astype(np.float64), 64), y64, rtol=1e-12, atol=1e-12)


# ---- RMSNorm ---------------------------------------------------------------------------------------

def test_rmsnorm_unit_rms_and_gain():
    x = synth.normal_f32(1, 1, 2560, 0.3, 2.0)
    ones = np.full(2560, 0x3C00, dtype=np.uint16)
    u = oracle.rmsnorm(x, ones, 1e-5, 64)
    assert abs(np.sqrt(np.mean(u ** 2)) - np.sqrt(np.mean(x.astype(np.float64) ** 2) / (np.mean(x.astype(np.float64) ** 2) + 1e-5))) < 1e-12
    u32 = oracle.rmsnorm(x, ones, 0.0, 32)
    assert abs(np.sqrt(np.mean(u32.astype(np.float64) ** 2)) - 1.0) < 1e-6
    g = synth.normal_f16(1, 2, 2560, 1.0, 0.1)
    ug = oracle.rmsnorm(x, g, 0.0, 64)
    np.testing.assert_allclose(ug / f32(g), oracle.rmsnorm(x, ones, 0.0, 64), rtol=1e-12)
    # scale invariance by an exact power of two (eps = 0)
    np.testing.assert_allclose(oracle.rmsnorm(4 * x, g, 0.0, 64), ug, rtol=1e-12)


def test_rmsnorm_closed_forms():
    ones = np.full(8, 0x3C00, dtype=np.uint16)
    c, eps = 0.5, 1e-5
    u = oracle.rmsnorm(np.full(8, c), ones, eps, 64)
    np.testing.assert_allclose(u, c / np.sqrt(c * c + eps), rtol=1e-14)
    assert np.all(oracle.rmsnorm(np.zeros(8), ones, eps, 64) == 0.0)


# ---- RoPE ------------------------------------------------------------------------------------------

def test_rope_identity_at_position_zero():
    v = synth.normal_f32(2, 3, 128, 0.0, 1.0)
    np.testing.assert_array_equal(oracle.rope(v, 0, 10000.0, 32), v)


def test_rope_pairing_and_frequencies_closed_form():
    # dh = 8: dimension i pairs with i + 4 and turns by pos * theta^(-2i/8)
    theta, pos, dh = 10000.0, 3, 8
    for i in range(4):
        e = np.zeros(dh)
        e[i] = 1.0
        out = oracle.rope(e, pos, theta, 64)
        ang = pos * theta ** (-2.0 * i / dh)
        expect = np.zeros(dh)
        expect[i], expect[i + 4] = np.cos(ang), np.sin(ang)
        np.testing.assert_allclose(out, expect, atol=1e-15)
        e2 = np.zeros(dh)
        e2[i + 4] = 1.0
        expect2 = np.zeros(dh)
        expect2[i], expect2[i + 4] = -np.sin(ang), np.cos(ang)
        np.testing.assert_allclose(oracle.rope(e2, pos, theta, 64), expect2, atol=1e-15)


def test_rope_is_a_rotation_with_relative_positions():
    q = synth.normal_f32(2, 4, 128, 0.0, 1.0).astype(np.float64)
    k = synth.normal_f32(2, 5, 128, 0.0, 1.0).astype(np.float64)
    for p in (1, 17, 1000, 8191):
        np.testing.assert_allclose(np.linalg.norm(oracle.rope(q, p, 10000.0, 64)), np.linalg.norm(q), rtol=1e-12)
    # composition: R(p1) R(p2) = R(p1 + p2), and scores depend only on p1 - p2
    np.testing.assert_allclose(oracle.rope(oracle.rope(q, 5, 10000.0, 64), 9, 10000.0, 64),
                               oracle.rope(q, 14, 10000.0, 64), atol=1e-12)
    s1 = oracle.rope(q, 40, 10000.0, 64) @ oracle.rope(k, 7, 10000.0, 64)
    s2 = oracle.rope(q, 140, 10000.0, 64) @ oracle.rope(k, 107, 10000.0, 64)
    assert abs(s1 - s2) < 1e-9
    # the fp32 version stays within fp32 rounding of the fp64 one
    q32 = q.astype(np.float32)
    np.testing.assert_allclose(oracle.rope(q32, 777, 10000.0, 32), oracle.rope(q32.astype(np.float64), 777, 10000.0, 64),
                               atol=2e-6)


# ---- attention -------------------------------------------------------------------------------------

def test_attention_single_position_returns_v():
    q = synth.normal_f32(3, 1, 128, 0.0, 1.0)
    K = synth.normal_f16(3, 2, (1, 128), 0.0, 1.0)
    V = synth.normal_f16(3, 3, (1, 128), 0.0, 1.0)
    np.testing.assert_array_equal(oracle.attention(q, K, V, 32), f32(V)[0])


def test_attention_equal_keys_give_mean_of_v():
    q = synth.normal_f32(3, 4, 64, 0.0, 1.0)
    K = np.repeat(synth.normal_f16(3, 5, (1, 64), 0.0, 1.0), 37, axis=0)
    V = synth.normal_f16(3, 6, (37, 64), 0.0, 1.0)
    np.testing.assert_allclose(oracle.attention(q, K, V, 64), f32(V).astype(np.float64).mean(0), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.attention(q, K, V, 32), f32(V).astype(np.float64).mean(0), atol=2e-6)


def test_attention_against_scipy_softmax():
    for c, dh in ((1, 64), (2, 64), (129, 128), (1000, 128)):
        q = synth.normal_f32(4, c, dh, 0.0, 1.0)
        K = synth.normal_f16(4, c + 1, (c, dh), 0.0, 1.0)
        V = synth.normal_f16(4, c + 2, (c, dh), 0.0, 1.0)
        s = (f32(K).astype(np.float64) @ q.astype(np.float64)) / np.sqrt(dh)
        ref = softmax(s) @ f32(V).astype(np.float64)
        np.testing.assert_allclose(oracle.attention(q, K, V, 64), ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(oracle.attention(q, K, V, 32), ref, atol=1e-5)


def test_attention_two_positions_closed_form():
    # with two positions the weight of the first is sigmoid(s0 - s1)
    q = np.zeros(64)
    q[0] = 8.0
    K = f16(np.array([[1.0] + [0.0] * 63, [0.5] + [0.0] * 63]))
    V = f16(np.array([[1.0] * 64, [-1.0] * 64]))
    w0 = expit((8.0 - 4.0) / 8.0)
    np.testing.assert_allclose(oracle.attention(q, K, V, 64), np.full(64, w0 - (1 - w0)), rtol=1e-14)


# ---- SiLU, argmax ----------------------------------------------------------------------------------

def test_silu_values():
    assert oracle.silu(0.0, 64) == 0.0
    assert abs(oracle.silu(40.0, 64) - 40.0) < 1e-12 and abs(oracle.silu(-40.0, 64)) < 1e-15
    for z in (-5.5, -1.0, -1e-3, 0.25, 1.0, 3.0):
        assert abs(oracle.silu(z, 64) - z * expit(z)) < 1e-15
        assert abs(oracle.silu(z, 32) - z * expit(z)) < 1e-6 * max(1.0, abs(z))


def test_argmax_lowest_index_on_ties():
    v = np.array([0.0, 2.0, -1.0, 2.0, 2.0], dtype=np.float32)
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.array([-3.0, -3.0])) == 0


# ---- whole-model special cases ---------------------------------------------------------------------

def _ln(x, g, eps):
    # eps reaches the oracle as an fp32 field of its config struct
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x) + float(np.float32(eps))) * f32(g)


def test_zero_layer_model_is_norm_then_lm_head():
    cfg = small_cfg(n_layers=0)
    w = synth.model_weights(cfg)
    m = oracle.Model(cfg, w, 8, 64)
    for t in (0, 5, 127):
        expect = f32(w["lm_head"]).astype(np.float64) @ _ln(f32(w["embed"][t]), w["final_norm"], cfg.rms_eps)
        np.testing.assert_allclose(m.forward(t), expect, rtol=1e-12, atol=1e-13)


def test_layer_with_zero_output_projections_is_identity():
    cfg = small_cfg(n_layers=2)
    w = synth.model_weights(cfg)
    for lay in w["layers"]:
        lay["wo"][:] = 0
        lay["w_down"][:] = 0
    w0 = dict(w, layers=[])
    a = oracle.Model(cfg, w, 8, 32)
    b = oracle.Model(dataclasses.replace(cfg, n_layers=0), w0, 8, 32)
    for t in (3, 9, 100, 3):
        np.testing.assert_array_equal(a.forward(t), b.forward(t))


def test_gqa_equals_mha_with_repeated_kv_heads():
    cfg = small_cfg(n_layers=2, n_heads=4, n_kv_heads=2)
    w = synth.model_weights(cfg)
    dh = cfg.head_dim
    mha = dataclasses.replace(cfg, n_kv_heads=4)
    wm = dict(w, layers=[])
    for lay in w["layers"]:
        rep = lambda W: np.concatenate([W[(h // 2) * dh:(h // 2 + 1) * dh] for h in range(4)])  # noqa: E731
        wm["layers"].append(dict(lay, wk=rep(lay["wk"]), wv=rep(lay["wv"])))
    a, b = oracle.Model(cfg, w, 16, 32), oracle.Model(mha, wm, 16, 32)
    for t in synth.tokens(5, 10, cfg.vocab):
        np.testing.assert_array_equal(a.forward(int(t)), b.forward(int(t)))


def test_uniform_attention_layer_adds_wo_times_mean_v():
    # Wq = 0 makes every score 0, so attention averages the cached V rows; Wd = 0 removes the FFN.
    cfg = small_cfg(n_layers=1)
    w = synth.model_weights(cfg)
    lay = w["layers"][0]
    lay["wq"][:] = 0
    lay["w_down"][:] = 0
    m = oracle.Model(cfg, w, 16, 64)
    toks = [7, 8, 9, 10, 11]
    for p, t in enumerate(toks):
        logits = m.forward(t)
        dh, group = cfg.head_dim, cfg.n_heads // cfg.n_kv_heads
        o = np.concatenate([np.mean([f32(m.kv_row(0, 1, h // group, j)).astype(np.float64) for j in range(p + 1)], axis=0)
                            for h in range(cfg.n_heads)])
        x = f32(w["embed"][t]).astype(np.float64) + f32(lay["wo"]).astype(np.float64) @ o
        expect = f32(w["lm_head"]).astype(np.float64) @ _ln(x, w["final_norm"], cfg.rms_eps)
        np.testing.assert_allclose(logits, expect, rtol=1e-10, atol=1e-12)


def test_ffn_block_is_swiglu():
    # Wo = 0 removes attention, leaving x + Wd (silu(Wg u) * (Wu u)) with u = rmsnorm(x) * g_ffn.
    cfg = small_cfg(n_layers=1)
    w = synth.model_weights(cfg)
    lay = w["layers"][0]
    lay["wo"][:] = 0
    m = oracle.Model(cfg, w, 8, 64)
    t = 77
    x0 = f32(w["embed"][t]).astype(np.float64)
    u = _ln(x0, lay["ffn_norm"], cfg.rms_eps)
    g, up = f32(lay["w_gate"]) @ u, f32(lay["w_up"]) @ u
    x = x0 + f32(lay["w_down"]).astype(np.float64) @ (g * expit(g) * up)
    expect = f32(w["lm_head"]).astype(np.float64) @ _ln(x, w["final_norm"], cfg.rms_eps)
    np.testing.assert_allclose(m.forward(t), expect, rtol=1e-10, atol=1e-12)


def test_cached_keys_are_rotated_projections():
    cfg = small_cfg(n_layers=1)
    w = synth.model_weights(cfg)
    m = oracle.Model(cfg, w, 8, 64)
    lay, dh = w["layers"][0], cfg.head_dim
    for p, t in enumerate([4, 50, 51]):
        m.forward(t)
        u = _ln(f32(w["embed"][t]), lay["attn_norm"], cfg.rms_eps)
        k = f32(lay["wk"]).astype(np.float64) @ u
        v = f32(lay["wv"]).astype(np.float64) @ u
        ang = p * cfg.rope_theta ** (-2.0 * np.arange(dh // 2) / dh)
        for h in range(cfg.n_kv_heads):
            kh = k[h * dh:(h + 1) * dh]
            a, b = kh[:dh // 2], kh[dh // 2:]
            rot = np.concatenate([a * np.cos(ang) - b * np.sin(ang), b * np.cos(ang) + a * np.sin(ang)])
            np.testing.assert_array_equal(m.kv_row(0, 0, h, p), rot.astype(np.float16).view(np.uint16))
            np.testing.assert_array_equal(m.kv_row(0, 1, h, p), v[h * dh:(h + 1) * dh].astype(np.float16).view(np.uint16))


def test_fp32_oracle_within_rounding_of_fp64_on_tiny():
    w = synth.model_weights(TINY)
    p = synth.prompt(TINY_DECODE)
    t32, L32 = oracle.generate(TINY, w, p, TINY_DECODE.decode_len, precision=32)
    t64, L64 = oracle.generate(TINY, w, p, TINY_DECODE.decode_len, precision=64)
    assert np.max(np.abs(L32 - L64)) < 1e-4
    s = np.sort(L64, axis=1)
    margin = s[:, -1] - s[:, -2]
    for i in range(len(t32)):
        if margin[i] > 1e-3:
            assert t32[i] == t64[i]
        else:
            break


def test_oracle_rejects_bad_config_and_full_cache():
    cfg = small_cfg(n_heads=3, n_kv_heads=2)
    with pytest.raises(ValueError):
        oracle.Model(cfg, synth.model_weights(small_cfg()), 4)
    cfg = small_cfg()
    m = oracle.Model(cfg, synth.model_weights(cfg), 2)
    m.forward(1)
    m.forward(2)
    with pytest.raises(ValueError):
        m.forward(3)


def test_prompt_positions_without_logits_leave_the_same_state():
    """Skipping the LM head at prompt positions (prefill) changes nothing the next forward sees."""
    cfg = small_cfg(n_layers=2)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(3, 9, cfg.vocab)
    a = oracle.Model(cfg, w, 16)
    la = a.prefill(prompt)
    b = oracle.Model(cfg, w, 16)
    lb = [b.forward(t) for t in prompt][-1]
    np.testing.assert_array_equal(la, lb)
    np.testing.assert_array_equal(a.forward(5), b.forward(5))
    assert a.pos == b.pos == len(prompt) + 1


def test_attention_heads_on_several_threads_change_no_sum():
    """Past 256 positions the heads run on several threads, each with its own score row: the logits must be
    bit-identical to a single-threaded run."""
    cfg = small_cfg(n_layers=1, n_heads=8, n_kv_heads=2)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(4, 300, cfg.vocab)
    before = oracle.threads()
    try:
        oracle.set_threads(1)
        one = oracle.Model(cfg, w, 320).prefill(prompt)
        oracle.set_threads(4)
        four = oracle.Model(cfg, w, 320).prefill(prompt)
    finally:
        oracle.set_threads(before)
    np.testing.assert_array_equal(one, four)
