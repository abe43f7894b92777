"""Tensor-parallel decode protocol on the CPU: two gloo ranks, each computing its shard of a tiny model's decode
(persistent_monokernel_decode_gb300.tp: Megatron-style partition, two partial-sum reductions per layer through
sequence-flagged mailboxes with bounded waits) must reproduce the oracle's logits; a rank that never posts makes
its peer's wait run out with an error instead of hanging. No GPU is involved: the mailboxes live in shared
memory, standing in for peer-mapped HBM.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def _rms(x, g, eps):
    return (x / np.sqrt(np.mean(x.astype(np.float32) ** 2, dtype=np.float32) + np.float32(eps))).astype(np.float32) * g


def _rope(v, pos, theta):
    dh = v.shape[-1]
    half = dh // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / dh)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    a, b = v[..., :half].copy(), v[..., half:].copy()
    out = np.empty_like(v)
    out[..., :half] = a * c - b * s
    out[..., half:] = b * c + a * s
    return out


def _shard_decode(cfg, w, shard, mbox, tokens, timeout_s, skip_post_at=None):
    """Forward `tokens` one position at a time on this rank's shard; returns the full logits of every position
    (assembled by a third exchange of zero-padded LM-head slices)."""
    from persistent_monokernel_decode_gb300 import tp
    d, dh, F, V = cfg.d_model, cfg.head_dim, cfg.ffn_dim, cfg.vocab
    G = cfg.n_heads // cfg.n_kv_heads
    q0, q1 = shard.q_heads
    k0, k1 = shard.kv_heads
    f0, f1 = shard.ffn_rows
    v0, v1 = shard.vocab_rows
    L = cfg.n_layers
    K = np.zeros((L, k1 - k0, len(tokens), dh), np.float32)
    Vc = np.zeros_like(K)
    seq = 0
    out = []

    def reduce(partial):
        nonlocal seq
        seq += 1
        if skip_post_at == seq:
            raise RuntimeError("skipped")
        return tp.allreduce(mbox, seq, partial, timeout_s)

    for pos, tok in enumerate(tokens):
        x = _f16(w["embed"][tok])
        for l in range(L):
            lw = w["layers"][l]
            u = _rms(x, _f16(lw["attn_norm"]), cfg.rms_eps)
            Wq = _f16(lw["wq"]).reshape(cfg.n_heads, dh, d)[q0:q1]
            Wk = _f16(lw["wk"]).reshape(cfg.n_kv_heads, dh, d)[k0:k1]
            Wv = _f16(lw["wv"]).reshape(cfg.n_kv_heads, dh, d)[k0:k1]
            q = _rope(Wq @ u, pos, cfg.rope_theta)
            k = _rope(Wk @ u, pos, cfg.rope_theta)
            K[l, :, pos] = k.astype(np.float16).astype(np.float32)
            Vc[l, :, pos] = (Wv @ u).astype(np.float16).astype(np.float32)
            o = np.empty((q1 - q0, dh), np.float32)
            for h in range(q1 - q0):
                kv = h // G
                s = (K[l, kv, :pos + 1] @ q[h]) / np.float32(np.sqrt(dh))
                p = np.exp(s - s.max())
                o[h] = (p / p.sum()) @ Vc[l, kv, :pos + 1]
            Wo = _f16(lw["wo"])[:, q0 * dh:q1 * dh]
            x = x + reduce(Wo @ o.reshape(-1))
            u = _rms(x, _f16(lw["ffn_norm"]), cfg.rms_eps)
            g = _f16(lw["w_gate"])[f0:f1] @ u
            up = _f16(lw["w_up"])[f0:f1] @ u
            a = (g / (1 + np.exp(-g))) * up
            x = x + reduce(_f16(lw["w_down"])[:, f0:f1] @ a)
        logits = np.zeros(V, np.float32)
        logits[v0:v1] = _f16(w["lm_head"])[v0:v1] @ _rms(x, _f16(w["final_norm"]), cfg.rms_eps)
        out.append(reduce(logits))  # zero-padded slices: the sum is their concatenation, exactly
    return np.stack(out)


class _Padded:
    """Exchanges carry d floats (residual deltas) or vocab floats (the logits): the mailbox is sized for the
    larger, and a shorter partial is zero-padded."""

    def __init__(self, mbox, width):
        self.m, self.width, self.n = mbox, width, width

    def post(self, seq, partial):
        full = np.zeros(self.width, np.float32)
        full[:partial.size] = partial
        self.n = partial.size
        self.m.post(seq, full)

    def take(self, seq, timeout_s):
        return self.m.take(seq, timeout_s)[:self.n]


def _worker(rank, world, port, shm_name, mode, q):
    sys.path.insert(0, ROOT)
    try:
        import torch.distributed as dist
        from multiprocessing import shared_memory

        import synth
        from persistent_monokernel_decode_gb300 import tp
        from synth.configs import ModelConfig
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
        cfg = ModelConfig("tp", n_layers=2, d_model=128, n_heads=4, n_kv_heads=2, head_dim=32, ffn_dim=192,
                          vocab=256, seed=31, gain_std=0.05)
        w = synth.model_weights(cfg)
        tokens = synth.tokens(31, 7, cfg.vocab)
        shm = shared_memory.SharedMemory(name=shm_name)
        buf = np.ndarray((world * tp.Mailbox.floats_per_rank(world, cfg.vocab),), dtype=np.float64, buffer=shm.buf)
        mbox = tp.Mailbox(buf, world, cfg.vocab, rank)
        shard = tp.partition(cfg.n_heads, cfg.n_kv_heads, cfg.ffn_dim, cfg.vocab, world, rank)
        dist.barrier()
        box = _Padded(mbox, cfg.vocab)
        if mode == "ok":
            logits = _shard_decode(cfg, w, shard, box, tokens, timeout_s=10.0)
            q.put((rank, "ok", logits))
        else:  # rank 1 never posts its third exchange; rank 0 must time out there, not hang
            try:
                _shard_decode(cfg, w, shard, box, tokens, timeout_s=0.5, skip_post_at=3 if rank == 1 else None)
                q.put((rank, "finished", None))
            except tp.ReductionTimeout as e:
                q.put((rank, "timeout", str(e)))
            except RuntimeError as e:
                q.put((rank, "skipped", str(e)))
        del buf
        shm.close()
        dist.destroy_process_group()
    except Exception as e:  # report, do not hang the parent
        q.put((rank, "error", repr(e)))


def _run(mode):
    import multiprocessing as mp
    from multiprocessing import shared_memory

    from persistent_monokernel_decode_gb300 import tp
    world, vocab = 2, 256
    ctx = mp.get_context("spawn")
    size = 8 * world * tp.Mailbox.floats_per_rank(world, vocab)
    shm = shared_memory.SharedMemory(create=True, size=size)
    np.ndarray((size // 8,), dtype=np.float64, buffer=shm.buf)[:] = 0
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, shm.name, mode, q)) for r in range(world)]
    try:
        for p in procs:
            p.start()
        res = {}
        for _ in range(world):
            r, status, payload = q.get(timeout=120)
            res[r] = (status, payload)
        for p in procs:
            p.join(timeout=30)
        return res
    finally:
        for p in procs:
            if p.is_alive():
                p.kill()
        shm.close()
        shm.unlink()


def test_partition_covers_every_head_row_and_vocab_id_once():
    from persistent_monokernel_decode_gb300 import tp
    for world in (1, 2, 4):
        shards = [tp.partition(20, 4, 7680, 32000, world, r) for r in range(world)]
        for field, total in (("q_heads", 20), ("kv_heads", 4), ("ffn_rows", 7680), ("vocab_rows", 32000)):
            spans = [getattr(s, field) for s in shards]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        for s in shards:  # each rank's query heads are exactly the groups of its KV heads
            assert s.q_heads == (s.kv_heads[0] * 5, s.kv_heads[1] * 5)
    with pytest.raises(ValueError):
        tp.partition(20, 4, 7680, 32000, 3, 0)


def test_argmax_key_orders_like_the_kernel():
    from persistent_monokernel_decode_gb300 import tp
    keys = [tp.argmax_key(v, i) for i, v in enumerate([-1.0, 2.5, 2.5, -0.0, 0.0, -3.0])]
    assert max(range(len(keys)), key=keys.__getitem__) == 1  # the largest value, the lowest index on ties
    assert tp.argmax_key(-0.5, 0) < tp.argmax_key(0.25, 9) < tp.argmax_key(1.0, 3)


def test_two_rank_tp_decode_matches_the_oracle():
    import oracle
    import synth
    from synth.configs import ModelConfig
    res = _run("ok")
    assert res[0][0] == "ok" and res[1][0] == "ok", res
    np.testing.assert_array_equal(res[0][1], res[1][1])  # fixed-order sums: identical on both ranks
    cfg = ModelConfig("tp", n_layers=2, d_model=128, n_heads=4, n_kv_heads=2, head_dim=32, ffn_dim=192,
                      vocab=256, seed=31, gain_std=0.05)
    w = synth.model_weights(cfg)
    tokens = synth.tokens(31, 7, cfg.vocab)
    m = oracle.Model(cfg, w, len(tokens))
    ref = np.stack([m.forward(int(t)) for t in tokens])
    assert np.max(np.abs(res[0][1] - ref)) < 1e-3


def test_a_peer_that_never_posts_ends_the_wait_with_an_error():
    res = _run("skip")
    assert res[1][0] == "skipped", res
    assert res[0][0] == "timeout", res
    assert "partial 3 of rank 1" in res[0][1]
