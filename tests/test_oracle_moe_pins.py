"""Pins of the oracle's sparse-MoE FFN (FP8 E4M3 experts with row scales, top-k softmax router) and of the FP8
weights the generator writes: each checked against a library routine, an identity or a special case, so that
a wrong code table, a transposed scale, a misordered selection or a mixed-up expert index fails one of them."""
import numpy as np
import pytest

import oracle
import synth
from synth.configs import MOE_TINY

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("this torch has no float8_e4m3fn", allow_module_level=True)


def e4m3_lib(codes):
    """E4M3 ("fn") codes to float64 through torch's float8_e4m3fn: the library decode."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_of_every_code_matches_the_library():
    codes = np.arange(256, dtype=np.uint8)
    mine = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    np.testing.assert_array_equal(mine, e4m3_lib(codes))
    # landmarks of the format: 1.0, the largest finite, the smallest normal and subnormal, NaN
    assert mine[0x38] == 1.0 and mine[0x7E] == 448.0 and mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])


def test_generator_fp8_encoding_is_round_to_nearest_even_and_saturates():
    L = synth.lib()
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(20000) * 30, rng.standard_normal(5000) * 1e-3,
                           np.array([0.0, -0.0, 448.0, 447.9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9 * 2.5,
                                     1.0 + 1 / 16, 1.0 + 3 / 16, -(1.0 + 1 / 16)])]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448.0]
    mine = np.array([L.synth_f32_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, ref)
    assert L.synth_f32_to_e4m3(1e6) == 0x7E and L.synth_f32_to_e4m3(-1e6) == 0xFE and L.synth_f32_to_e4m3(460.0) == 0x7E


def test_fp8_rows_reconstruct_the_drawn_weights_within_e4m3_precision():
    q, s = synth.e4m3_rows(5, 42, 16, 512, 0.02)
    w = synth.normal_f32(5, 42, (16, 512), 0.0, 0.02).astype(np.float64)
    deq = e4m3_lib(q) * s[:, None]
    assert np.allclose(s, np.abs(w).max(axis=1).astype(np.float32) / np.float32(448.0), rtol=1e-6)
    # E4M3 keeps 3 mantissa bits: error at most half a step (2^-4 relative) or half the subnormal step
    assert np.all(np.abs(deq - w) <= np.maximum(np.abs(w) * 2.0 ** -4, s[:, None] * 2.0 ** -10) * (1 + 1e-6))


def test_fp8_gemv_matches_brute_force_on_library_decoded_weights():
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, size=(37, 203), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38  # no NaN codes in a weight
    s = rng.uniform(1e-4, 2e-3, 37).astype(np.float32)
    x = rng.standard_normal(203)
    ref = (e4m3_lib(q) * s.astype(np.float64)[:, None]) @ x
    np.testing.assert_allclose(oracle.gemv_fp8(q, s, x, 64), ref, rtol=1e-12, atol=1e-15)


def test_topk_takes_the_largest_lowest_index_first_and_renormalises_the_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    r = np.array([0.5, 2.0, -1.0, 2.0, 0.25, 2.0, 1.5, -3.0])
    idx, w = oracle.topk_softmax(r, 4)
    assert idx.tolist() == [1, 3, 5, 6]  # three ties at 2.0 by index, then 1.5
    full = scipy_special.softmax(r)
    np.testing.assert_allclose(w, full[idx] / full[idx].sum(), rtol=1e-14)
    assert abs(w.sum() - 1.0) < 1e-15


def _tiny_moe(seed=3):
    cfg = MOE_TINY
    return cfg, synth.moe_weights(cfg)


def _swiglu_expert(lay, e, u):
    g = (e4m3_lib(lay["gate_q"][e]) * lay["gate_s"][e][:, None]) @ u
    up = (e4m3_lib(lay["up_q"][e]) * lay["up_s"][e][:, None]) @ u
    a = g / (1.0 + np.exp(-g)) * up
    return (e4m3_lib(lay["down_q"][e]) * lay["down_s"][e][:, None]) @ a


def test_identical_experts_reduce_the_moe_ffn_to_one_swiglu_expert():
    cfg, w = _tiny_moe()
    lay = w["layers"][0]
    for k in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s"):
        lay[k][:] = lay[k][0]
    m = oracle.Model(cfg, w, 8, 64)
    u = np.random.default_rng(3).standard_normal(cfg.d_model)
    np.testing.assert_allclose(m.moe_ffn(0, u), _swiglu_expert(lay, 0, u), rtol=1e-9, atol=1e-12)


def test_moe_ffn_is_invariant_under_a_joint_permutation_of_experts_and_router_rows():
    cfg, w = _tiny_moe()
    u = np.random.default_rng(4).standard_normal(cfg.d_model)
    before = oracle.Model(cfg, w, 8, 64).moe_ffn(1, u)
    perm = np.random.default_rng(5).permutation(cfg.n_experts)
    lay = w["layers"][1]
    for k in ("router", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s"):
        lay[k] = np.ascontiguousarray(lay[k][perm])
    after = oracle.Model(cfg, w, 8, 64).moe_ffn(1, u)
    np.testing.assert_allclose(after, before, rtol=1e-12, atol=1e-15)


def test_moe_ffn_uses_the_routed_experts_with_their_softmax_weights():
    """A router whose logits order is known: the output is the weighted sum of exactly those experts."""
    scipy_special = pytest.importorskip("scipy.special")
    cfg, w = _tiny_moe()
    lay = w["layers"][0]
    u = np.zeros(cfg.d_model)
    u[0] = 1.0
    # router logits = router[:, 0] (fp16): experts 6, 1, 4, 3 lead in that order
    col = np.array([0.0, 0.75, -0.5, 0.25, 0.5, -0.25, 1.0, -1.0], dtype=np.float16)
    lay["router"] = np.zeros_like(lay["router"])
    lay["router"][:, 0] = col.view(np.uint16)
    m = oracle.Model(cfg, w, 8, 64)
    got = m.moe_ffn(0, u)
    # the routing margin: 4th selected logit (0.25) minus the best unselected one (0.0)
    assert m.route_margin() == 0.25 and m.route_margin() == np.inf
    sel = [6, 1, 4, 3]
    ids, gaps = m.route()  # the routing record of layer 0: the experts in selection order and its gap
    assert list(ids[0]) == sel and gaps[0] == 0.25
    wts = scipy_special.softmax(col.astype(np.float64)[sel])
    ref = sum(wt * _swiglu_expert(lay, e, u) for wt, e in zip(wts, sel))
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-12)


def test_moe_oracle_fp32_agrees_with_fp64():
    cfg, w = _tiny_moe()
    prompt = synth.tokens(cfg.seed, 10, cfg.vocab)
    _, l32 = oracle.generate(cfg, w, prompt, 6, precision=32)
    _, l64 = oracle.generate(cfg, w, prompt, 6, precision=64)
    assert np.max(np.abs(l32 - l64)) < 1e-4
