// Batched prefill (kie_prefill.cu): buffers and entry point shared with the C ABI.
#pragma once
#include <cuda_runtime.h>

#include "kie_decode.cuh"

namespace kie {

constexpr int PF_TOKENS = 128;  // prompt tokens per chunk

// fp32 activations of one chunk (device): x, h [PF_TOKENS][d]; q, o [PF_TOKENS][Hq*dh]; a [PF_TOKENS][F];
// scale [PF_TOKENS] (per-token RMS scale); part [splits][PF_TOKENS][M] (the raw sums of a projection's K splits,
// kie_tc_splits). Tensor-core operands: layer l's projection j (QKV, WO, GU, DOWN) is stored as canonical tiles
// at tc_w + l * tc_layer_stride + tc_off[j] (kie_tcgemm.cuh); tc_b holds one chunk's activation tiles.
struct PrefillBufs {
  float *x, *h, *q, *o, *a, *scale, *part;
  float *att_o, *att_ml;  // attention partials: [pieces][PF_TOKENS][Hq][dh] and [pieces][PF_TOKENS][Hq][2]
  const uint8_t *tc_w;
  long long tc_layer_stride, tc_off[4];
  uint8_t *tc_b;
  int *status;  // raised if a tensor-core GEMM's wait runs out
  unsigned long long timeout_ns;
};

// K tiles (of 64 columns) per split and the number of splits for a projection of Mt 128-row tiles and KT K tiles
// on an n_cta-SM GPU: enough splits to give every SM one (tile, split) block, none of them empty.
inline void kie_tc_splits(int Mt, int KT, int n_cta, int *kt_per_split, int *splits) {
  int ns = n_cta / (Mt > 0 ? Mt : 1);
  ns = ns < 1 ? 1 : (ns > KT ? KT : ns);
  const int kps = (KT + ns - 1) / ns;
  *kt_per_split = kps;
  *splits = (KT + kps - 1) / kps;
}

// Attention pieces a prompt position can span: positions per piece, and pieces for max_seq positions.
constexpr int PF_ATT_PIECE = 512;
inline int kie_pf_att_pieces(int max_seq) { return (max_seq + PF_ATT_PIECE - 1) / PF_ATT_PIECE; }

// Byte offset of element (r, k) in a canonical 128 x 64 tensor-core tile (8 x 8 fp16 core matrices of 128
// contiguous bytes; core matrix (i, j) at i * 1024 + j * 128). The device code's tc_tile_offset is the same map.
inline int kie_tc_offset_in_tile(int r, int k) { return (r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2; }

// Bytes of the canonical tensor-core tiles of an [M, K] matrix (rows padded to 128, columns to 64).
inline size_t kie_tc_tile_bytes(int M, int K) { return (size_t)((M + 127) / 128) * ((K + 63) / 64) * 128 * 64 * 2; }

}  // namespace kie

// Pack a row-major fp16 [M, K] matrix (device) into canonical tensor-core tiles at dst, folding gain (or null)
// into the columns like the decode's pack kernel. Asynchronous on `st`.
cudaError_t kie_launch_tc_pack(const uint16_t *src, int M, int K, const uint16_t *gain, uint8_t *dst, cudaStream_t st);

// Enqueue the prefill of n tokens (device ids) at positions pos0 .. pos0+n-1 on `st`: the K/V cache rows, the
// logits of the last token (p.logits) and the next token to emit (p.persist->next_token).
cudaError_t kie_run_prefill(const kie::DecodeParams &p, const kie::PrefillBufs &b, const int *tok_dev, int pos0,
                            int n, cudaStream_t st);
