"""GPU parity of the sparse-MoE decode (router, top-k softmax, FP8 E4M3 experts with row scales) against the
oracle's MoE FFN, through the C ABI.

Same bar as the dense model: logits max |diff| <= 2e-2, greedy tokens identical wherever the oracle's top-1/top-2
margin exceeds 2e-2, teacher forcing so one permitted divergence cannot cascade. The expert selection is itself a
floating-point decision (a top-k over router logits) that the two sides take from logits rounded differently, so
it is teacher-forced too: the oracle runs free and records the experts every layer of every forward selected, and
the GPU is given those (kie_decode_forced_routed). Every step's logits are then compared, with no exemption. The
GPU also returns the selection it would have made itself; it must equal the oracle's wherever the oracle's
routing gap (its k-th router logit minus its best unselected one) is at least ROUTE_EPS. ROUTE_EPS = 1e-3 against
router logits of standard deviation ~0.9 and a GPU/oracle hidden-state discrepancy of ~1e-4 relative (fp16
RMSNorm-gain folds, fp32 summation order) leaves a factor of ten; closer gaps are ties that either side may break
either way, and the selections there are only checked to be valid (distinct ids in range).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from synth.configs import MOE_DECODE, MOE_M, MOE_TINY

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2
MARGIN = 2e-2
ROUTE_EPS = 1e-3


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


def oracle_run(cfg, w, prompt, n, max_seq):
    """Greedy oracle decode (fp32) with the routing of every forward: route[0] is the last prompt
    position's margin, route[i + 1] that of decode step i."""
    m = oracle.Model(cfg, w, max_seq, 32)
    m.prefill(prompt[:-1])
    m.route_margin()
    cur = m.forward(int(prompt[-1]))
    route, logits, toks = [m.route_margin()], [cur], []
    for _ in range(n):
        toks.append(oracle.argmax(cur))
        cur = m.forward(toks[-1])
        logits.append(cur)
        route.append(m.route_margin())
    return np.array(toks, dtype=np.int32), np.stack(logits), np.array(route)


def oracle_run_routed(cfg, w, prompt, n, max_seq):
    """Greedy oracle decode (fp32) recording every forward's routing, prompt positions included:
    (tokens [n], logits [n + 1, V] from the last prompt position on, ids [P + n, L, k], gaps [P + n, L])."""
    m = oracle.Model(cfg, w, max_seq, 32)
    ids, gaps = [], []

    def record():
        i, g = m.route()
        ids.append(i)
        gaps.append(g)

    for t in prompt[:-1]:
        m.forward(int(t), want_logits=False)
        record()
    cur = m.forward(int(prompt[-1]))
    record()
    logits, toks = [cur], []
    for _ in range(n):
        toks.append(oracle.argmax(cur))
        cur = m.forward(toks[-1])
        logits.append(cur)
        record()
    return np.array(toks, dtype=np.int32), np.stack(logits), np.stack(ids), np.stack(gaps)


def check_selection(own, ids, gaps, n_experts):
    """The GPU's own selection equals the oracle's (as a set) wherever every layer's gap is clear; elsewhere it is
    a valid selection. Returns the number of (forward, layer) decisions compared."""
    assert own.min() >= 0 and own.max() < n_experts
    assert all(len(set(r)) == r.size for r in own.reshape(-1, own.shape[-1]))
    clear = gaps >= ROUTE_EPS
    same = np.sort(own, axis=-1) == np.sort(ids, axis=-1)
    bad = np.argwhere(clear & ~same.all(axis=-1))
    assert bad.size == 0, f"(forward, layer) {bad[:5].tolist()}: GPU {own[tuple(bad[0])]} vs oracle {ids[tuple(bad[0])]}"
    return int(clear.sum())


def check_run(dec, cfg, w, prompt, n, max_seq):
    """The whole sequence (prompt and n teacher-forced decode steps) through the decode kernel with the oracle's
    expert selections imposed: logits compared at every step from the last prompt position on, greedy tokens where
    the margin is clear, the GPU's own selection where the routing gap is clear."""
    ref_tokens, ref_logits, ids, gaps = oracle_run_routed(cfg, w, prompt, n, max_seq)
    P = len(prompt)
    seq = np.concatenate([np.asarray(prompt, dtype=np.int32), ref_tokens])
    dec.reset()
    toks, logits, own = dec.decode_forced_routed(seq, forced_experts=ids)
    diff = np.max(np.abs(logits[P - 1:] - ref_logits), axis=1)
    assert diff.max() <= LOGIT_TOL, f"step {int(diff.argmax())}: logits differ by {diff.max()}"
    sure = margins(ref_logits[:-1]) > MARGIN
    assert np.array_equal(toks[P:][sure], ref_tokens[sure])
    compared = check_selection(own, ids, gaps, cfg.n_experts)
    assert compared >= 0.5 * gaps.size, f"only {compared} of {gaps.size} routing decisions are clear of a tie"
    return ref_tokens, ref_logits


@pytest.fixture(scope="module")
def tiny(kie):
    w = synth.moe_weights(MOE_TINY)
    dec = kie.Decoder(MOE_TINY, w, max_seq=64)
    yield w, dec
    dec.close()


def test_moe_tiny_teacher_forced_parity(tiny):
    w, dec = tiny
    check_run(dec, MOE_TINY, w, synth.tokens(MOE_TINY.seed, 12, MOE_TINY.vocab), 24, 64)


def test_moe_tiny_free_routing_prefill_and_steps_where_routing_is_clear(tiny):
    """The regular entry points (prefill, kie_decode_forced) route on their own: where no layer of a forward holds a
    near-tie (oracle routing margin >= ROUTE_EPS), its logits must match the oracle's."""
    w, dec = tiny
    prompt = synth.tokens(MOE_TINY.seed, 12, MOE_TINY.vocab)
    ref_tokens, ref_logits, route = oracle_run(MOE_TINY, w, prompt, 24, 64)
    settled = route >= ROUTE_EPS
    dec.reset()
    dec.prefill(prompt)
    assert not settled[0] or np.max(np.abs(dec.logits() - ref_logits[0])) <= LOGIT_TOL
    toks, logits = dec.decode_forced(ref_tokens)
    diff = np.max(np.abs(logits - ref_logits[1:]), axis=1)
    assert diff[settled[1:]].max(initial=0.0) <= LOGIT_TOL
    assert settled.sum() >= len(settled) // 2


def test_moe_forced_routing_is_applied(tiny):
    """Imposing a selection other than the model's own changes the logits, and imposing the model's own selection
    changes nothing (bit for bit): the override reaches both the producer's expert stream and the weights."""
    w, dec = tiny
    seq = synth.tokens(MOE_TINY.seed + 5, 10, MOE_TINY.vocab)
    dec.reset()
    _, free_logits, own = dec.decode_forced_routed(seq)
    dec.reset()
    _, same_logits, own2 = dec.decode_forced_routed(seq, forced_experts=own)
    np.testing.assert_array_equal(same_logits, free_logits)
    np.testing.assert_array_equal(own2, own)
    other = (own + 1) % MOE_TINY.n_experts  # still distinct ids within a layer
    dec.reset()
    _, other_logits, own3 = dec.decode_forced_routed(seq, forced_experts=other)
    np.testing.assert_array_equal(own3[0, 0], own[0, 0])  # the first layer of the first forward is unaffected
    assert np.max(np.abs(other_logits - free_logits)) > 1e-3


def test_moe_tiny_free_running_greedy_matches_until_a_close_call(tiny):
    w, dec = tiny
    prompt = synth.tokens(MOE_TINY.seed, 12, MOE_TINY.vocab)
    ref_tokens, ref_logits, route = oracle_run(MOE_TINY, w, prompt, 24, 64)
    dec.reset()
    dec.prefill(prompt)
    toks = dec.decode(24)
    close = (margins(ref_logits[:-1]) <= MARGIN) | (route[:-1] < ROUTE_EPS)
    first_close = int(np.argmax(close)) if np.any(close) else 24
    assert np.array_equal(toks[:first_close], ref_tokens[:first_close])
    assert dec.position == 36


def test_moe_tiny_split_calls_and_prefill_pieces_are_exact(tiny):
    _, dec = tiny
    prompt = synth.tokens(MOE_TINY.seed, 12, MOE_TINY.vocab)
    dec.reset()
    dec.prefill(prompt)
    a = dec.logits()
    whole = dec.decode(20)
    dec.reset()
    dec.prefill(prompt[:5])
    dec.prefill(prompt[5:6])
    dec.prefill(prompt[6:])
    assert np.array_equal(dec.logits(), a)
    parts = np.concatenate([dec.decode(7), dec.decode(1), dec.decode(12)])
    assert np.array_equal(whole, parts)
    st = dec.barrier_stats()
    # 5 grid phases per MoE layer (the router is folded into the QKV and WO phases), + the LM head
    assert st["barriers"] == 12 * (5 * MOE_TINY.n_layers + 1)


def test_moe_joint_expert_permutation_leaves_the_logits_bit_identical(kie):
    """Renumbering the experts (router rows and expert matrices together) selects the same experts in the same
    order, so every CUDA-side sum is taken in the same order: the logits must not change by a single bit."""
    w = synth.moe_weights(MOE_TINY)
    prompt = synth.tokens(MOE_TINY.seed, 6, MOE_TINY.vocab)
    forced = synth.tokens(MOE_TINY.seed + 1, 5, MOE_TINY.vocab)
    dec = kie.Decoder(MOE_TINY, w, max_seq=32)
    dec.prefill(prompt)
    _, before = dec.decode_forced(forced)
    dec.close()
    perm = np.random.default_rng(7).permutation(MOE_TINY.n_experts)
    for lay in w["layers"]:
        for k in ("router", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s"):
            lay[k] = np.ascontiguousarray(lay[k][perm])
    dec = kie.Decoder(MOE_TINY, w, max_seq=32)
    dec.prefill(prompt)
    _, after = dec.decode_forced(forced)
    dec.close()
    assert np.array_equal(before, after)


# structure variants: one routed expert (weight exactly 1), every expert routed, several router logits per
# lane (40 experts), the largest router (256 experts), widths with full and ragged 512-code FP8 blocks, and
# experts wide enough that some CTAs stack two experts' gate/up tiles and others do not
MOE_VARIANTS = {
    "top1": dict(top_k=1),
    "all_experts": dict(top_k=8),
    "e40_k3": dict(n_experts=40, top_k=3),
    "e256_k8": dict(n_experts=256, top_k=8, n_layers=1),
    "wide_ragged": dict(d_model=784, ffn_dim=528, expert_ffn=528, top_k=2, n_layers=1),
    # 2,560 gate/up rows over 152 CTAs: 16 rows (two experts stacked per tile) or 18 (one expert per tile)
    "wide_experts": dict(ffn_dim=1280, expert_ffn=1280, top_k=3, n_layers=1),
}


@pytest.mark.parametrize("name", sorted(MOE_VARIANTS))
def test_moe_structure_variants(kie, name):
    cfg = dataclasses.replace(MOE_TINY, name="moe_" + name, **MOE_VARIANTS[name])
    w = synth.moe_weights(cfg)
    dec = kie.Decoder(cfg, w, max_seq=40)
    try:
        check_run(dec, cfg, w, synth.tokens(cfg.seed, 9, cfg.vocab), 8, 40)
    finally:
        dec.close()


# ---- the MoE workload at full size (64 experts of width 1,024, top 4, 24 layers), bench launch shape ------

@pytest.fixture(scope="module")
def moe_m(kie):
    w = synth.moe_weights(MOE_M)
    dec = kie.Decoder(MOE_M, w, max_seq=MOE_DECODE.capacity)
    yield w, dec
    dec.close()


def test_moe_m_sampled_steps_match_oracle(moe_m):
    """The bench workload's 256-token prompt and the first 16 decode steps, tokens and expert selections
    teacher-forced from the oracle, logits compared at every step."""
    w, dec = moe_m
    check_run(dec, MOE_M, w, synth.prompt(MOE_DECODE), 16, MOE_DECODE.capacity)


def test_moe_m_full_decode_properties(moe_m):
    """All 512 greedy tokens of the bench workload: valid ids, positions, identical tokens when split."""
    _, dec = moe_m
    n = MOE_DECODE.decode_len
    prompt = synth.prompt(MOE_DECODE)
    dec.reset()
    dec.prefill(prompt)
    whole = dec.decode(n)
    assert whole.min() >= 0 and whole.max() < MOE_M.vocab
    assert dec.position == len(prompt) + n
    dec.reset()
    dec.prefill(prompt)
    parts = np.concatenate([dec.decode(200), dec.decode(n - 200)])
    assert np.array_equal(whole, parts)
    assert dec.barrier_stats()["barriers"] == (n - 200) * (5 * MOE_M.n_layers + 1)
