"""Host side of the C ABI, no GPU: the library loads and exports every declared entry point, the per-CTA
tile layout is a bijection with contiguous tiles, buffer planning and configuration checks behave."""
import os
import re

import numpy as np
import pytest

import persistent_monokernel_decode_gb300 as kie
from synth.configs import MOE_M, MOE_TINY, TINY, TWO_B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    kie.build()
    yield


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "kie.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kie_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound():
    names = declared_entry_points()
    assert len(names) >= 20
    L = kie.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in kie.SIGNATURES, f"{n} has no ctypes signature in the binding"
    assert set(kie.SIGNATURES) == set(names)


@pytest.mark.parametrize("M,K,n", [(2, 8, 1), (2, 8, 152), (34, 264, 3), (768, 256, 152), (1408, 704, 152),
                                   (100, 520, 7), (64, 2560, 5)])
def test_packed_layout_is_a_bijection_with_contiguous_tiles(M, K, n):
    off = np.array([[kie.packed_offset(M, K, n, r, c) for c in range(K)] for r in range(M)], dtype=np.int64)
    assert np.array_equal(np.sort(off.ravel()), np.arange(M * K))
    for cta in range(n):
        r0, r1 = kie.rows_of_cta(M, n, cta)
        if r1 == r0:
            continue
        block = off[r0:r1]
        assert block.min() == r0 * K and block.max() == r1 * K - 1  # the CTA's region is contiguous
        for g0 in range(0, r1 - r0, 32):
            rows = min(32, r1 - r0 - g0)
            for k0 in range(0, K, 256):
                w = min(256, K - k0)
                tile = block[g0:g0 + rows, k0:k0 + w]
                # one row-major run of rows*w elements
                assert np.array_equal(tile.ravel() - tile.min(), np.arange(rows * w))


@pytest.mark.parametrize("M,K,n", [(2, 16, 1), (256, 256, 152), (256, 128, 152), (34, 784, 3), (66, 528, 5),
                                   (100, 1040, 7), (2048, 1024, 152)])
def test_fp8_packed_layout_is_a_bijection_with_contiguous_tiles(M, K, n):
    """FP8 expert matrices: one-byte codes in 512-code column blocks, so a full 32-row tile is again 16 KB. Each
    tile is one contiguous run of its rows; in a full 512-code block the 16-code chunk q of an odd row sits at
    chunk q ^ 4 of the row, elsewhere rows are plain row-major."""
    off = np.array([[kie.packed_offset_fp8(M, K, n, r, c) for c in range(K)] for r in range(M)], dtype=np.int64)
    assert np.array_equal(np.sort(off.ravel()), np.arange(M * K))
    for r in range(M):
        for k0 in range(0, K, 512):
            w = min(512, K - k0)
            row = off[r, k0:k0 + w]
            base = row.min()
            assert row.max() == base + w - 1  # a row of a tile is one run of w bytes
            c = np.arange(w)
            want = c if (w < 512 or r % 2 == 0) else ((c // 16) ^ 4) * 16 + c % 16
            assert np.array_equal(row - base, want), (r, k0)
    for cta in range(n):
        r0, r1 = kie.rows_of_cta(M, n, cta)
        if r1 == r0:
            continue
        block = off[r0:r1]
        assert block.min() == r0 * K and block.max() == r1 * K - 1
        for g0 in range(0, r1 - r0, 32):
            rows = min(32, r1 - r0 - g0)
            for k0 in range(0, K, 512):
                w = min(512, K - k0)
                tile = block[g0:g0 + rows, k0:k0 + w]
                assert np.array_equal(np.sort(tile.ravel()) - tile.min(), np.arange(rows * w))
                assert np.array_equal(tile.min(axis=1) - tile.min(), np.arange(rows) * w)  # rows in order
                assert tile.min() % 16 == 0 and (rows * w) % 16 == 0  # a legal bulk copy
    assert kie.packed_offset_fp8(M, K + 8, n, 0, 0) == -1  # K must be a multiple of 16


@pytest.mark.parametrize("M,K", [(128, 64), (256, 128), (200, 200), (768, 256), (136, 72)])
def test_tensor_core_tile_layout_is_canonical(M, K):
    """The prefill's tensor-core copy: an injective map into ceil(M/128) x ceil(K/64) tiles of 16 KB, each 8-row x
    8-column block one run of 128 bytes with rows 16 bytes apart (the no-swizzle core matrix), core matrices 128 B
    apart along K and 1 KB apart along M: the strides the tensor-core descriptors are given."""
    off = np.array([[kie.tc_tile_offset(M, K, r, c) for c in range(K)] for r in range(M)], dtype=np.int64)
    KT, MT = (K + 63) // 64, (M + 127) // 128
    assert off.min() >= 0 and off.max() < MT * KT * 16384 and len(np.unique(off)) == M * K
    assert np.all(off % 2 == 0)
    for r in range(0, M - 7, 8):
        for c in range(0, K - 7, 8):
            blk = off[r:r + 8, c:c + 8]
            assert np.array_equal(blk - blk[0, 0], np.arange(8)[:, None] * 16 + np.arange(8)[None, :] * 2)
            if (c + 8) % 64 and c + 15 < K:
                assert off[r, c + 8] - off[r, c] == 128          # next core matrix along K
            if (r + 8) % 128 and r + 15 < M:
                assert off[r + 8, c] - off[r, c] == 1024         # next 8-row group
    assert kie.tc_tile_offset(M, K + 4, 0, 0) == -1             # K must be a multiple of 8


def test_moe_buffer_plan_without_a_device():
    cfg = kie.make_config(MOE_M, 768)
    s = kie.kie_query_buffers(cfg, 152, kie.make_moe_config(MOE_M))
    E, d, F, L = MOE_M.n_experts, MOE_M.d_model, MOE_M.expert_ffn, MOE_M.n_layers
    assert s.weights_bytes >= L * E * 3 * F * d  # every expert of every layer is resident
    assert s.weights_bytes < L * E * 3 * F * d * 1.1 + (2 << 30)
    assert s.kv_bytes >= MOE_M.kv_bytes_per_token(768)
    dense = kie.kie_query_buffers(kie.make_config(MOE_TINY, 64), 152)
    sparse = kie.kie_query_buffers(kie.make_config(MOE_TINY, 64), 152, kie.make_moe_config(MOE_TINY))
    assert sparse.weights_bytes > dense.weights_bytes


@pytest.mark.parametrize("field,value", [("n_experts", 0), ("n_experts", 257), ("top_k", 0), ("top_k", 9)])
def test_unsupported_moe_configs_are_rejected(field, value):
    moe = kie.make_moe_config(MOE_TINY)
    setattr(moe, field, value)
    with pytest.raises(kie.KieError) as e:
        kie.kie_query_buffers(kie.make_config(MOE_TINY, 64), 152, moe)
    assert e.value.code == kie.KIE_ERR_INVALID
    cfg = kie.make_config(MOE_TINY, 64)
    cfg.d_model = 264  # a multiple of 8 but not of 16
    with pytest.raises(kie.KieError):
        kie.kie_query_buffers(cfg, 152, kie.make_moe_config(MOE_TINY))
    moe = kie.make_moe_config(MOE_TINY)
    moe.top_k = moe.n_experts + 1 if moe.n_experts < 8 else 9
    with pytest.raises(kie.KieError):
        kie.kie_query_buffers(kie.make_config(MOE_TINY, 64), 152, moe)


@pytest.mark.parametrize("M,n", [(2, 1), (2, 152), (256, 152), (3584, 152), (15360, 152), (32000, 152), (10, 3)])
def test_row_split_pairs_cover_and_balance(M, n):
    spans = [kie.rows_of_cta(M, n, i) for i in range(n)]
    assert spans[0][0] == 0 and spans[-1][1] == M
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    sizes = [r1 - r0 for r0, r1 in spans]
    assert all(s % 2 == 0 for s in sizes)
    assert max(sizes) - min(sizes) <= 2


def test_buffer_plan_without_a_device():
    cfg = kie.make_config(TWO_B, 1152)
    s = kie.kie_query_buffers(cfg, 152)
    assert s.n_cta == 152
    assert s.weights_bytes >= TWO_B.weight_bytes_per_token() + TWO_B.vocab * TWO_B.d_model * 2
    assert s.kv_bytes >= TWO_B.kv_bytes_per_token(1152)
    assert s.workspace_bytes < 64 << 20
    t = kie.kie_query_buffers(kie.make_config(TINY, 48), 152)
    assert t.weights_bytes >= TINY.weight_bytes_per_token()


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("n_kv_heads", 3), ("vocab", 4095), ("d_model", 260),
                                         ("n_layers", 0), ("ffn_dim", 700), ("max_seq", 0)])
def test_unsupported_configs_are_rejected(field, value):
    cfg = kie.make_config(TINY, 64)
    setattr(cfg, field, value)
    with pytest.raises(kie.KieError) as e:
        kie.kie_query_buffers(cfg, 152)
    assert e.value.code == kie.KIE_ERR_INVALID


def test_product_path_fails_loudly_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError):
        kie.Decoder(TINY, {}, 16)
