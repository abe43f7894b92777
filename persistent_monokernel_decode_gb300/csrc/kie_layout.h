// Per-CTA tiled weight layout, shared by the host packer and the device streams.
//
// Every projection W [M, K] is split by rows over the n CTAs of the persistent grid, in pairs of rows
// (pairs are never split: they carry the two halves of a RoPE rotation, or a gate/up pair). CTA i owns
// rows [r0, r1) with r0 = 2*floor(i*P/n), P = M/2. Its rows occupy the contiguous element range
// [r0*K, r1*K) of the packed matrix, re-tiled as
//     for each row group g of up to TILE_ROWS rows:  for each column block b of up to TILE_COLS columns:
//         tile[rows_in_group][cols_in_block], row-major,
// so that every tile is one contiguous run of bytes that a single 1-D bulk copy moves into shared memory.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define KIE_HD __host__ __device__ __forceinline__
#else
#define KIE_HD inline
#endif

namespace kie {

constexpr int TILE_ROWS = 32;
constexpr int TILE_COLS = 256;
constexpr int SLOT_BYTES = TILE_ROWS * TILE_COLS * 2;  // 16 KB: one ring slot holds one full tile

struct RowRange {
  int r0, r1;
};

KIE_HD RowRange rows_of_cta(int M, int n, int i) {
  const long long P = M / 2;
  return {(int)(2 * ((long long)i * P / n)), (int)(2 * ((long long)(i + 1) * P / n))};
}

// CTA owning row r.
KIE_HD int owner_of_row(int M, int n, int r) {
  const long long P = M / 2;
  int i = P > 0 ? (int)(((long long)(r / 2) * n) / P) : 0;
  if (i >= n) i = n - 1;
  while (i + 1 < n && rows_of_cta(M, n, i + 1).r0 <= r) ++i;
  while (i > 0 && rows_of_cta(M, n, i).r0 > r) --i;
  return i;
}

// FP8 (one-byte) matrices use column blocks of FP8_TILE_COLS, so a full tile is again SLOT_BYTES.
constexpr int FP8_TILE_COLS = 2 * TILE_COLS;

// Element offset of W[r][c] in the packed matrix whose column blocks are bw columns wide.
KIE_HD long long packed_offset_bw(int M, int K, int n, int r, int c, int bw) {
  const RowRange rr = rows_of_cta(M, n, owner_of_row(M, n, r));
  const int lr = r - rr.r0;
  const int g = lr / TILE_ROWS;
  const int rows_g = (rr.r1 - rr.r0 - g * TILE_ROWS) < TILE_ROWS ? (rr.r1 - rr.r0 - g * TILE_ROWS) : TILE_ROWS;
  const int b = c / bw;
  const int w = (K - b * bw) < bw ? (K - b * bw) : bw;
  return (long long)rr.r0 * K + (long long)g * TILE_ROWS * K + (long long)rows_g * bw * b +
         (long long)(lr - g * TILE_ROWS) * w + (c - b * bw);
}

// Element offset of W[r][c] in a packed fp16 matrix (column blocks of TILE_COLS).
KIE_HD long long packed_offset(int M, int K, int n, int r, int c) { return packed_offset_bw(M, K, n, r, c, TILE_COLS); }

// Byte offset of code Q[r][c] in a packed FP8 matrix: column blocks of FP8_TILE_COLS codes; within a full block
// the 16-code chunk q of row r sits at chunk q ^ 4 when r is odd (row-major otherwise). Rows are split over
// CTAs in pairs, so a row's parity is also its parity within its tile, and within two tiles of the same rows
// copied back to back. The swizzle lets the tensor-core consumer's lanes of two neighbouring rows read the
// same chunk columns from different halves of a 128-byte line (no shared-memory bank conflict).
KIE_HD long long packed_offset_fp8(int M, int K, int n, int r, int c) {
  const long long o = packed_offset_bw(M, K, n, r, c, FP8_TILE_COLS);
  const int b = c / FP8_TILE_COLS;
  if (K - b * FP8_TILE_COLS < FP8_TILE_COLS || !(r & 1)) return o;
  const int q = (c - b * FP8_TILE_COLS) >> 4;
  return o + (long long)(((q ^ 4) - q) * 16);
}

}  // namespace kie
