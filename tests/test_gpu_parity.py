"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Tolerances (the acceptance bar of this port): GEMV relative error <= 1e-3 against fp64; logits max |diff|
<= 2e-2 at every step; greedy tokens identical wherever the oracle's top-1/top-2 margin exceeds 2e-2, with
teacher forcing (the oracle's tokens fed to both sides) so one permitted divergence cannot cascade.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from synth.configs import GEMV_SHAPES, TINY, TINY_DECODE, TWO_B, ModelConfig

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2
MARGIN = 2e-2


@pytest.fixture(scope="module")
def kie():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import persistent_monokernel_decode_gb300 as k
    k.build()
    return k


def margins(logits):
    s = np.sort(logits, axis=-1)
    return s[..., -1] - s[..., -2]


def check_run(dec, cfg, w, prompt, n, max_seq):
    """Prefill + teacher-forced decode against the oracle; returns the max logit error seen."""
    ref_tokens, ref_logits = oracle.generate(cfg, w, prompt, n, max_seq=max_seq)
    dec.reset()
    dec.prefill(prompt)
    err = float(np.max(np.abs(dec.logits() - ref_logits[0])))
    assert err <= LOGIT_TOL, f"prefill logits differ by {err}"
    toks, logits = dec.decode_forced(ref_tokens)
    diff = np.max(np.abs(logits - ref_logits[1:]), axis=1)
    assert diff.max() <= LOGIT_TOL, f"step {int(diff.argmax())}: logits differ by {diff.max()}"
    sure = margins(ref_logits[:-1]) > MARGIN
    assert np.array_equal(toks[sure], ref_tokens[sure])
    return max(err, float(diff.max())), ref_tokens, ref_logits


# ---- GEMV -----------------------------------------------------------------------------------------------

def gemv_check(kie, W, x, n_cta=0):
    import torch
    M, K = W.shape
    Wd = torch.from_numpy(W.view(np.int16)).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    packed = kie.gemv_pack(Wd, n_cta)
    y = kie.gemv(packed, xd, M, K, n_cta).cpu().numpy()
    torch.cuda.synchronize()
    y64 = oracle.gemv(W, synth.as_f32(x).astype(np.float64), 64)
    rel = np.max(np.abs(y - y64)) / max(np.max(np.abs(y64)), 1e-30)
    assert rel <= 1e-3, (M, K, rel)
    absdot = oracle.gemv(W & 0x7FFF, np.abs(synth.as_f32(x)).astype(np.float64), 64)
    assert np.all(np.abs(y - y64) <= 1e-3 * absdot + 1e-6)
    return rel


@pytest.mark.parametrize("M,K,n_cta", [(2, 8, 0), (2, 8, 1), (34, 264, 3), (1000, 2056, 0), (66, 520, 5),
                                       (4096, 704, 0), (32000, 256, 0)])
def test_gemv_small_and_ragged(kie, M, K, n_cta):
    W = synth.normal_f16(11, M + K, (M, K), 0.0, 1.0 / np.sqrt(K))
    x = synth.normal_f16(11, 7, K, 0.0, 1.0)
    gemv_check(kie, W, x, n_cta)


@pytest.mark.parametrize("shape", GEMV_SHAPES, ids=lambda s: f"{s.M}x{s.K}")
def test_gemv_sweep_shapes(kie, shape):
    W, x = synth.gemv_operands(shape)
    gemv_check(kie, W, x)


# ---- tiny decoder ---------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(kie):
    w = synth.model_weights(TINY)
    wl = TINY_DECODE
    dec = kie.Decoder(TINY, w, max_seq=wl.prompt_len + wl.decode_len)
    yield w, dec
    dec.close()


def test_tiny_teacher_forced_parity(tiny):
    w, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    check_run(dec, TINY, w, prompt, TINY_DECODE.decode_len, TINY_DECODE.prompt_len + TINY_DECODE.decode_len)


def test_tiny_free_running_greedy_matches_until_a_close_call(tiny):
    w, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    n = TINY_DECODE.decode_len
    ref_tokens, ref_logits = oracle.generate(TINY, w, prompt, n)
    dec.reset()
    dec.prefill(prompt)
    toks = dec.decode(n)
    m = margins(ref_logits[:-1])
    first_close = int(np.argmax(m <= MARGIN)) if np.any(m <= MARGIN) else n
    assert np.array_equal(toks[:first_close], ref_tokens[:first_close])
    assert dec.position == len(prompt) + n


def test_split_calls_equal_one_call(tiny):
    _, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    dec.reset()
    dec.prefill(prompt)
    whole = dec.decode(20)
    dec.reset()
    dec.prefill(prompt[:5])
    dec.prefill(prompt[5:])
    parts = np.concatenate([dec.decode(7), dec.decode(1), dec.decode(12)])
    assert np.array_equal(whole, parts)


def test_prefill_in_pieces_equals_whole(tiny):
    _, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    dec.reset()
    dec.prefill(prompt)
    a = dec.logits()
    dec.reset()
    for i in range(0, len(prompt), 3):
        dec.prefill(prompt[i:i + 3])
    np.testing.assert_array_equal(dec.logits(), a)


def test_prefill_equals_teacher_forced_decode_of_the_prompt(tiny):
    """prefill(P) then the next token's logits equal those of prefill(P[0]) followed by a teacher-forced decode of
    P[1:] (the batched tensor-core prefill against the decode kernel, token by token): within twice the logit
    tolerance of each other (each is within the tolerance of the oracle), and the same greedy token."""
    _, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    dec.reset()
    dec.prefill(prompt)
    batched = dec.logits()
    dec.reset()
    dec.prefill(prompt[:1])
    dec.decode_forced(prompt[1:], want_logits=False)
    stepped = dec.logits()
    assert dec.position == len(prompt)
    assert float(np.max(np.abs(batched - stepped))) <= 2 * LOGIT_TOL
    if margins(batched) > 2 * MARGIN:
        assert int(np.argmax(batched)) == int(np.argmax(stepped))


def test_batched_prefill_across_chunks_is_independent_of_the_cut(kie):
    """A 300-token prompt spans three 128-token prefill chunks; prefilled whole or in uneven pieces it must
    leave bit-identical logits (every sum runs in an order the chunking does not change), and both must match
    the oracle."""
    cfg = dataclasses.replace(TINY, seed=14)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(14, 300, cfg.vocab)
    dec = kie.Decoder(cfg, w, max_seq=320)
    dec.reset()
    dec.prefill(prompt)
    whole = dec.logits()
    dec.reset()
    for a, b in ((0, 100), (100, 101), (101, 250), (250, 300)):
        dec.prefill(prompt[a:b])
    np.testing.assert_array_equal(dec.logits(), whole)
    assert dec.position == 300
    _, ref_logits = oracle.generate(cfg, w, prompt, 0, max_seq=320)
    assert float(np.max(np.abs(whole - ref_logits[0]))) <= LOGIT_TOL
    dec.close()


def test_prefill_attention_pieces_are_independent_of_the_cut(kie):
    """A 1,200-token prompt spans three 512-position attention pieces (split and merged) and ten 128-token
    chunks: whole, in uneven pieces (cuts inside and at piece and chunk boundaries) and teacher-forced decode
    afterwards must agree bit for bit, the cached K/V rows included, and match the oracle."""
    cfg = dataclasses.replace(TINY, seed=15)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(15, 1200, cfg.vocab)
    forced = synth.tokens(16, 4, cfg.vocab)
    dec = kie.Decoder(cfg, w, max_seq=1216)
    dec.prefill(prompt)
    whole = dec.logits()
    _, whole_steps = dec.decode_forced(forced)
    dec.reset()
    for a, b in ((0, 511), (511, 513), (513, 640), (640, 1023), (1023, 1024), (1024, 1200)):
        dec.prefill(prompt[a:b])
    np.testing.assert_array_equal(dec.logits(), whole)
    _, steps = dec.decode_forced(forced)
    np.testing.assert_array_equal(steps, whole_steps)
    ref_tokens, ref_logits = oracle.generate(cfg, w, prompt, 0, max_seq=1216)
    assert float(np.max(np.abs(whole - ref_logits[0]))) <= LOGIT_TOL
    dec.close()


def test_forced_decode_can_start_a_sequence(tiny, kie):
    """kie_decode_forced_routed without a prior prefill ingests the forced tokens like a prompt (the first emitted
    token is -1); afterwards it is an ordinary teacher-forced decode, and expert arguments are refused for a dense
    model."""
    w, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    ref_tokens, ref_logits = oracle.generate(TINY, w, prompt, 6, max_seq=dec.max_seq)
    dec.reset()
    toks, logits, own = dec.decode_forced_routed(np.concatenate([prompt, ref_tokens]), want_experts=False)
    assert toks[0] == -1 and own is None
    P = len(prompt)
    assert float(np.max(np.abs(logits[P - 1:] - ref_logits))) <= LOGIT_TOL
    sure = margins(ref_logits[:-1]) > MARGIN
    assert np.array_equal(toks[P:][sure], ref_tokens[sure])
    dec.reset()
    with pytest.raises(kie.KieError) as e:
        dec.decode_forced_routed(prompt, want_experts=True)
    assert e.value.code == kie.KIE_ERR_INVALID


def test_profile_attention_leaves_the_sequence_alone(tiny):
    """The attention step run alone (profiling) changes neither the position nor the current logits, and decode
    afterwards still matches the oracle."""
    w, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    dec.reset()
    dec.prefill(prompt)
    before = dec.logits()
    dec.profile_attention(len(prompt), TINY.n_layers)
    assert dec.position == len(prompt)
    np.testing.assert_array_equal(dec.logits(), before)
    ref_tokens, ref_logits = oracle.generate(TINY, w, prompt, 4, max_seq=dec.max_seq)
    _, logits = dec.decode_forced(ref_tokens)
    assert float(np.max(np.abs(logits - ref_logits[1:]))) <= LOGIT_TOL


def test_api_errors(tiny, kie):
    _, dec = tiny
    dec.reset()
    with pytest.raises(kie.KieError) as e:
        dec.decode(1)
    assert e.value.code == kie.KIE_ERR_INVALID
    with pytest.raises(kie.KieError) as e:
        dec.prefill([TINY.vocab])
    assert e.value.code == kie.KIE_ERR_INVALID
    dec.prefill([1, 2, 3])
    with pytest.raises(kie.KieError) as e:
        dec.decode(dec.max_seq)
    assert e.value.code == kie.KIE_ERR_CAPACITY
    assert dec.position == 3


def test_barrier_stats(tiny):
    _, dec = tiny
    dec.reset()
    dec.prefill(synth.prompt(TINY_DECODE))
    dec.decode(4)
    st = dec.barrier_stats()
    assert st["barriers"] == 4 * (5 * TINY.n_layers + 1)
    assert 0 < st["mean_latency_ns"] <= st["mean_wait_ns"] + 1e-9
    assert st["total_ns"] > 0


def test_wait_limit_ends_a_stuck_launch_cleanly(tiny, kie):
    """One CTA skips one grid-barrier arrival: every other CTA's bounded wait runs out, the launch returns
    KIE_ERR_TIMEOUT, and the context is usable again afterwards."""
    w, dec = tiny
    prompt = synth.prompt(TINY_DECODE)
    dec.reset()
    dec.prefill(prompt)
    dec.set_timeout_ns(20_000_000)
    dec.debug_skip_arrival(cta=3, barrier=2)
    with pytest.raises(kie.KieError) as e:
        dec.decode(4)
    assert e.value.code == kie.KIE_ERR_TIMEOUT
    dec.set_timeout_ns(1_000_000_000)
    check_run(dec, TINY, w, prompt, 8, dec.max_seq)


# ---- structure variants ---------------------------------------------------------------------------------

VARIANTS = {
    # GQA 4:1 with dh = 128 and a non-multiple-of-256 width, gains != 1 (folding exercised)
    "gqa_dh128": ModelConfig("v1", n_layers=3, d_model=384, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=1000,
                             vocab=1000, seed=5, gain_std=0.1),
    # the largest group the attention step supports (8 query heads per KV head), dh = 64
    "group8_dh64": ModelConfig("v2", n_layers=2, d_model=512, n_heads=8, n_kv_heads=1, head_dim=64, ffn_dim=1376,
                               vocab=2050, seed=6, gain_std=0.05),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_structure_variants(kie, name):
    cfg = VARIANTS[name]
    w = synth.model_weights(cfg)
    prompt = synth.tokens(cfg.seed, 40, cfg.vocab)
    dec = kie.Decoder(cfg, w, max_seq=64)
    check_run(dec, cfg, w, prompt, 20, 64)
    dec.close()


def test_long_context_split_kv(kie):
    """Tiny model at 1,500 positions: split-KV with the maximum number of pieces, long chunks, several
    online-softmax sub-chunks per piece."""
    cfg = dataclasses.replace(TINY, seed=9)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(9, 1500, cfg.vocab)
    dec = kie.Decoder(cfg, w, max_seq=1516)
    check_run(dec, cfg, w, prompt, 12, 1516)
    dec.close()


def split_kv(c: int, smax: int):
    """The kernel's split of c attended positions into pieces: (pieces, positions per piece)."""
    S = min(smax, -(-c // 32))
    return S, -(-c // S)


def test_context_with_an_empty_split_kv_piece(kie):
    """Contexts where the split leaves the last piece of each KV head with no positions (its partial is
    m = -inf, l = 0, o = 0): the merge must weigh it zero. The context is found from this device's CTA count."""
    cfg = dataclasses.replace(TINY, seed=12)
    w = synth.model_weights(cfg)
    dec = kie.Decoder(cfg, w, max_seq=2048)
    smax = max(1, dec.n_cta // cfg.n_kv_heads)
    empty = [c for c in range(1, 2040) if (lambda S, C: (S - 1) * C >= c)(*split_kv(c, smax))]
    assert empty, "no context below 2,040 leaves a piece empty on this device"
    c = empty[0]
    prompt = synth.tokens(12, c - 1, cfg.vocab)  # the first decode step attends over c positions
    check_run(dec, cfg, w, prompt, 6, 2048)
    dec.close()


# ---- long context at the 2B widths -------------------------------------------------------------------------

def test_long_context_at_2b_widths(kie):
    """The long-context workload's shape on two layers: the 2B widths (d 2,560, 20 query heads of 128 over 4 KV
    heads, F 7,680, vocab 32,000), a prompt of 8,192 ids, then 8 teacher-forced decode steps against the oracle.
    The prefill runs the tensor-core attention with groups of 5 query heads over 16 pieces of 512 positions and
    their merge; every decode step splits about 8,200 positions over 38 pieces per KV head of several 32-position
    sub-chunks each (the oracle takes a couple of minutes on the host cores)."""
    cfg = dataclasses.replace(TWO_B, name="llama2b_L2", n_layers=2)
    w = synth.model_weights(cfg)
    prompt = synth.tokens(TWO_B.seed, 8192, cfg.vocab)
    dec = kie.Decoder(cfg, w, max_seq=8192 + 8)
    try:
        smax = max(1, dec.n_cta // cfg.n_kv_heads)
        S, C = split_kv(8193, smax)
        assert C > 32, "the decode steps must give each piece several sub-chunks"
        check_run(dec, cfg, w, prompt, 8, 8192 + 8)
    finally:
        dec.close()


# ---- the 2B workload at full size, in the launch configuration the bench times ---------------------------

@pytest.fixture(scope="module")
def two_b(kie):
    w = synth.model_weights(TWO_B)
    dec = kie.Decoder(TWO_B, w, max_seq=128 + 1024)
    yield w, dec
    dec.close()


def test_2b_every_decode_step_matches_oracle(two_b):
    """The bench workload in full: the 2B model, prompt of 128 ids, and all 1,024 decode steps teacher-forced
    against the oracle, logits compared at every step (the oracle takes a few minutes on the host cores)."""
    w, dec = two_b
    prompt = synth.tokens(TWO_B.seed, 128, TWO_B.vocab)
    check_run(dec, TWO_B, w, prompt, 1024, 128 + 1024)


def test_2b_full_decode_properties(two_b):
    """All 1,024 greedy tokens of the bench workload: valid ids, position bookkeeping, and identical tokens
    when the same decode is split into two calls."""
    _, dec = two_b
    prompt = synth.tokens(TWO_B.seed, 128, TWO_B.vocab)
    dec.reset()
    dec.prefill(prompt)
    whole = dec.decode(1024)
    assert whole.min() >= 0 and whole.max() < TWO_B.vocab
    assert dec.position == 128 + 1024
    dec.reset()
    dec.prefill(prompt)
    parts = np.concatenate([dec.decode(300), dec.decode(724)])
    assert np.array_equal(whole, parts)
    st = dec.barrier_stats()
    assert st["barriers"] == 724 * (5 * TWO_B.n_layers + 1)
