"""kie_decode_noalloc: greedy decode that allocates no device memory.

Some callers of this library cannot call cudaMalloc once they are running (their device memory is owned and
capped by a host framework's allocator, or their loop must not hit cudaMalloc/cudaFree, which can
synchronise the device). For them kie_decode_noalloc keeps the per-launch scratch in one static device array.
These tests check it against the regular entry point, kie_decode, through the C ABI: same tokens and the same
final logits (within the parity tolerance) over two calls in a row, and a clear error when a model's scratch
does not fit the array. This file is collected last on purpose, and it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest

import synth
from synth.configs import MOE_TINY, TINY, TINY_DECODE, ModelConfig

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2


@pytest.fixture(scope="module")
def kie():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import persistent_monokernel_decode_gb300 as k
    k.build()
    return k


def two_calls_each_way(kie, cfg, prompt, n1, n2, max_seq):
    import torch
    w = synth.moe_weights(cfg) if getattr(cfg, "n_experts", 0) else synth.model_weights(cfg)
    dec = kie.Decoder(cfg, w, max_seq=max_seq)
    try:
        dec.prefill(prompt)
        ref = np.concatenate([dec.decode(n1), dec.decode(n2)])
        ref_logits = dec.logits()
        ref_pos = dec.position

        dec.reset()
        dec.prefill(prompt)
        out = torch.full((n1 + n2,), -1, dtype=torch.int32, device="cuda")
        dec.decode_noalloc(n1, out[:n1])
        dec.decode_noalloc(n2, out[n1:])
        got = out.cpu().numpy()
        assert np.array_equal(got, ref)
        assert dec.position == ref_pos
        assert np.max(np.abs(dec.logits() - ref_logits)) <= LOGIT_TOL
    finally:
        dec.close()


def test_noalloc_matches_decode_tiny(kie):
    prompt = synth.prompt(TINY_DECODE)
    two_calls_each_way(kie, TINY, prompt, 12, 9, TINY_DECODE.prompt_len + 32)


def test_noalloc_matches_decode_gqa_dh128(kie):
    cfg = ModelConfig("na", n_layers=2, d_model=384, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=1000,
                      vocab=1000, seed=21, gain_std=0.1)
    two_calls_each_way(kie, cfg, synth.tokens(21, 40, cfg.vocab), 7, 7, 64)


def test_noalloc_matches_decode_sparse_moe(kie):
    """The sparse-MoE kernel (router logits and the routed experts' selection in the scratch) through the
    no-allocation entry point."""
    two_calls_each_way(kie, MOE_TINY, synth.tokens(MOE_TINY.seed, 10, MOE_TINY.vocab), 6, 5, 32)


def test_noalloc_checks_the_output_tensor(kie):
    """The binding refuses an output tensor the kernel could write past: wrong dtype, too short, on the host."""
    import torch
    dec = kie.Decoder(TINY, synth.model_weights(TINY), max_seq=32)
    try:
        dec.prefill([1, 2, 3])
        for bad in (torch.empty(4, dtype=torch.int64, device="cuda"), torch.empty(3, dtype=torch.int32, device="cuda"),
                    torch.empty(4, dtype=torch.int32), torch.empty(8, dtype=torch.int32, device="cuda")[::2]):
            with pytest.raises(ValueError):
                dec.decode_noalloc(4, bad)
        assert dec.position == 3
    finally:
        dec.close()


def test_noalloc_and_regular_calls_interleave(kie):
    import torch
    w = synth.model_weights(TINY)
    prompt = synth.prompt(TINY_DECODE)
    dec = kie.Decoder(TINY, w, max_seq=64)
    try:
        dec.prefill(prompt)
        ref = dec.decode(15)
        dec.reset()
        dec.prefill(prompt)
        out = torch.empty(5, dtype=torch.int32, device="cuda")
        a = dec.decode(5)
        dec.decode_noalloc(5, out)
        c = dec.decode(5)
        assert np.array_equal(np.concatenate([a, out.cpu().numpy(), c]), ref)
    finally:
        dec.close()


def test_noalloc_wait_limit_then_a_clean_decode(kie):
    """A grid-barrier arrival skipped on purpose (host-side hook, no GPU fault) during a no-allocation decode: the
    bounded waits run out, the call reports KIE_ERR_TIMEOUT from the static array's control block, and the ctx
    then decodes correctly again (teacher-forced against the oracle)."""
    import torch

    import oracle
    w = synth.model_weights(TINY)
    prompt = synth.prompt(TINY_DECODE)
    dec = kie.Decoder(TINY, w, max_seq=64)
    try:
        dec.prefill(prompt)
        dec.set_timeout_ns(20_000_000)
        dec.debug_skip_arrival(cta=3, barrier=2)
        out = torch.empty(4, dtype=torch.int32, device="cuda")
        with pytest.raises(kie.KieError) as e:
            dec.decode_noalloc(4, out)
        assert e.value.code == kie.KIE_ERR_TIMEOUT
        assert dec.position == 0  # a timed-out launch resets the sequence
        dec.set_timeout_ns(1_000_000_000)
        ref_tokens, ref_logits = oracle.generate(TINY, w, prompt, 8, max_seq=64)
        dec.prefill(prompt)
        toks, logits = dec.decode_forced(ref_tokens)
        assert np.max(np.abs(logits - ref_logits[1:])) <= LOGIT_TOL
        # and the skip was consumed by the timed-out call: a no-allocation decode now runs to the end
        dec.reset()
        dec.prefill(prompt)
        dec.decode_noalloc(4, out)
        assert dec.position == len(prompt) + 4
    finally:
        dec.close()


def test_noalloc_rejects_scratch_beyond_the_static_array(kie):
    # eight query heads of 128 on one KV head: the split-KV partials, one per CTA of the grid, take n_cta * 8 * 128
    # * 4 bytes, more than the 512 KB array from about 128 CTAs on (152 on GB300)
    cfg = ModelConfig("big", n_layers=1, d_model=256, n_heads=8, n_kv_heads=1, head_dim=128, ffn_dim=256,
                      vocab=256, seed=3)
    import torch
    dec = kie.Decoder(cfg, synth.model_weights(cfg), max_seq=16)
    if dec.n_cta * 8 * 128 * 4 <= 512 * 1024:
        dec.close()
        pytest.skip(f"with {dec.n_cta} CTAs this model's scratch fits the static array")
    try:
        dec.prefill([1, 2, 3])
        out = torch.empty(2, dtype=torch.int32, device="cuda")
        with pytest.raises(kie.KieError) as e:
            dec.decode_noalloc(2, out)
        assert e.value.code == kie.KIE_ERR_INVALID
        assert "scratch" in str(e.value)
        assert dec.position == 3
    finally:
        dec.close()
