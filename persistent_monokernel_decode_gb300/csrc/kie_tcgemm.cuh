// Tensor-core (tcgen05) GEMM of the batched prefill: Y = W' X for a chunk of up to PF_TOKENS prompt tokens.
//
// The prefill projections are real dense contractions (128 tokens share every weight), so they run on the
// 5th-generation tensor cores: one elected thread issues tcgen05.mma with both operands in shared memory and
// the fp32 accumulator in tensor memory (TMEM), a producer thread feeds a 4-stage shared-memory ring with 1-D
// bulk copies, and four warps read the accumulator back with tcgen05.ld.
//
// Precision: the activations are fp32. Each input x is split into two fp16 values, hi = fp16(x) and
// lo = fp16(x - hi): hi + lo is within 2^-21 |x| of x while lo is a normal fp16 (|x| >= 2^-3) and within 2^-25
// absolute below; the tensor core forms W'·hi and W'·lo (fp16 products are exact in fp32) and accumulates in
// fp32, and the epilogue adds the two, so a projection stays within about 1e-5 of sum |W' x| of the exact one.
// The B operand of one MMA is therefore 256 columns: the chunk's 128 tokens' high parts, then their low parts.
//
// Operand layout (both K-major, no swizzle): a tile is made of 8 x 8 fp16 "core matrices" of 128 contiguous
// bytes; core matrix (i, j) of rows 8i..8i+7 and columns 8j..8j+7 of a 64-column tile sits at i * 1024 + j * 128.
// In the matrix descriptor the leading-dimension byte offset (next core matrix along K) is 128 and the
// stride-dimension byte offset (next 8-row group) is 1,024. Weights are stored in HBM already in this layout,
// tile by tile (a 128 x 64 tile is one 16 KB bulk copy); the activations are converted into it per chunk.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kie_device.cuh"
#include "kie_prefill.cuh"

namespace kie {

constexpr int TC_M = 128;                     // rows per tile = TMEM lanes
constexpr int TC_N = 2 * PF_TOKENS;           // accumulator columns: tokens' high parts, then low parts
constexpr int TC_KT = 64;                     // columns per stage (four MMAs of K = 16)
constexpr int TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_M * TC_KT * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_N * TC_KT * 2;  // 32 KB
constexpr int TC_THREADS = 128;               // 4 warps: producer lane, MMA lane, then all four read TMEM
constexpr int TC_TMEM_COLS = TC_N;            // fp32 accumulator columns
constexpr size_t TC_SMEM = (size_t)TC_STAGES * (TC_A_BYTES + TC_B_BYTES);
static_assert(TC_N <= 256 && TC_N % 16 == 0, "one MMA covers the whole accumulator");

// Byte offset of element (r, k) in a canonical 64-column tile (r < rows of the tile, k < 64).
__host__ __device__ __forceinline__ int tc_tile_offset(int r, int k) {
  return (r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Shared-memory matrix descriptor: start address, LBO 128 B (along K), SBO 1,024 B (8-row groups), the
// descriptor version of the sm_100 family (bit 46), no swizzle.
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: D fp32, A and B fp16, both K-major, N = TC_N, M = TC_M.
constexpr uint32_t TC_IDESC = (1u << 4) | ((uint32_t)(TC_N >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24);

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// The mbarrier receives one arrival once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// The warp's 32 TMEM lanes (lane field of taddr = 32 * (warp % 4)), 16 consecutive fp32 columns from taddr.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcArgs {
  const uint8_t *A;   // weights: [M tiles][KT][16 KB] canonical tiles (rows past M and columns past K are zero)
  const uint8_t *B;   // activations: [KT][32 KB] canonical tiles of the chunk's hi/lo parts
  int KT;             // 64-column tiles along K
  int kt_per_split;   // K tiles summed by one block (blockIdx.y = split)
  float *part;        // raw sums hi + lo: [split][PF_TOKENS][M]
  int M, T;           // rows, tokens of the chunk
  int *status;        // raised (ST_TIMEOUT) if a wait runs out
  unsigned long long timeout_ns;
};

// One 128-row tile (blockIdx.x) over one K split (blockIdx.y): part[split][t][r] = sum_k W'[r][k] x[t][k].
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm_kernel(const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  __shared__ __align__(8) uint64_t full[TC_STAGES], empty[TC_STAGES], done;
  __shared__ uint32_t tmem_base;
  uint8_t *sA = tc_smem, *sB = tc_smem + (size_t)TC_STAGES * TC_A_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, split = blockIdx.y;
  const int kt0 = split * a.kt_per_split, kt1 = min(a.KT, kt0 + a.kt_per_split), nk = kt1 - kt0;
  const Guard g{a.status, a.timeout_ns};
  if (threadIdx.x == 0) {
    for (int i = 0; i < TC_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (threadIdx.x == 0) {  // producer: weight tile + activation tile per stage
    const uint64_t policy = l2_evict_first_policy();
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int st = i % TC_STAGES;
      if (i >= TC_STAGES && !wait_mbar(&empty[st], (uint32_t)((i / TC_STAGES - 1) & 1), g)) break;
      mbar_arrive_expect_tx(&full[st], TC_A_BYTES + TC_B_BYTES);
      bulk_g2s(sA + (size_t)st * TC_A_BYTES, a.A + ((size_t)mt * a.KT + kt0 + i) * TC_A_BYTES, TC_A_BYTES, &full[st],
               policy);
      bulk_g2s(sB + (size_t)st * TC_B_BYTES, a.B + (size_t)(kt0 + i) * TC_B_BYTES, TC_B_BYTES, &full[st], policy);
      ++issued;
    }
    // every copy must have landed before the block may exit (a bounded wait; the MMA thread normally saw them)
    for (int i = issued - TC_STAGES > 0 ? issued - TC_STAGES : 0; i < issued; ++i) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[i % TC_STAGES], (uint32_t)((i / TC_STAGES) & 1)))
        if (globaltimer() - t0 > g.timeout_ns) {
          raise_status(g, ST_TIMEOUT);
          break;
        }
    }
  } else if (threadIdx.x == 32) {  // MMA issuer
    for (int i = 0; i < nk; ++i) {
      const int st = i % TC_STAGES;
      if (!wait_mbar(&full[st], (uint32_t)((i / TC_STAGES) & 1), g)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + (size_t)st * TC_A_BYTES), b0 = smem_u32(sB + (size_t)st * TC_B_BYTES);
#pragma unroll
      for (int s = 0; s < TC_KT / 16; ++s)  // K = 16 per MMA: two core matrices along K
        tc_mma(tmem, tc_smem_desc(a0 + 256 * s), tc_smem_desc(b0 + 256 * s), TC_IDESC, (i > 0 || s > 0) ? 1u : 0u);
      tc_commit(&empty[st]);  // the stage is free once these MMAs have read it
    }
    tc_commit(&done);  // completes when every MMA above has
  }
  __syncwarp();

  // epilogue: warp w reads TMEM lanes 32w .. 32w+31 = tile rows; hi + lo per token
  const bool have = wait_mbar(&done, 0u, g);
  tc_fence_after();
  const int r = mt * TC_M + warp * 32 + lane;
  float *dst = a.part + (size_t)split * PF_TOKENS * a.M;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  for (int t0 = 0; t0 < a.T; t0 += 16) {
    float hi[16], lo[16];
    tmem_ld16(lane_base + (uint32_t)t0, hi);
    tmem_ld16(lane_base + (uint32_t)(PF_TOKENS + t0), lo);
    if (have && r < a.M) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (t0 + j < a.T) dst[(size_t)(t0 + j) * a.M + r] = hi[j] + lo[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TC_TMEM_COLS);
}

// B tiles of one chunk: element (n, k) of the [2 * PF_TOKENS][KT * 64] operand is hi(x[n][k]) for n < PF_TOKENS
// and lo(x[n - PF_TOKENS][k]) after, zero past T tokens or K columns. One thread writes 8 columns (16 bytes).
__global__ void tc_split_kernel(const float *x, int T, int K, int KT, uint8_t *B) {
  const int groups = KT * (TC_KT / 8);
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)TC_N * groups) return;
  const int n = (int)(idx / groups), kg = (int)(idx % groups), k0 = kg * 8;
  const int t = n % PF_TOKENS;
  const bool low = n >= PF_TOKENS;
  __align__(16) __half h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float v = (t < T && k0 + e < K) ? x[(size_t)t * K + k0 + e] : 0.f;
    const __half hv = __float2half_rn(v);
    h[e] = low ? __float2half_rn(v - __half2float(hv)) : hv;
  }
  *reinterpret_cast<uint4 *>(B + (size_t)(k0 / TC_KT) * TC_B_BYTES + tc_tile_offset(n, k0 % TC_KT)) =
      *reinterpret_cast<const uint4 *>(h);
}

// A tiles of a row-major fp16 [M, K] matrix: rows padded to a multiple of 128 and columns to KT * 64 with
// zeros; if gain is not null every column c is first multiplied by gain[c] in fp32 and rounded back to fp16
// (round to nearest even), the same fold as the decode's packed weights. One thread writes 8 columns.
__global__ void tc_pack_kernel(const uint16_t *src, int M, int K, int KT, const uint16_t *gain, uint8_t *A) {
  const int groups = KT * (TC_KT / 8), Mp = (M + TC_M - 1) / TC_M * TC_M;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)Mp * groups) return;
  const int m = (int)(idx / groups), kg = (int)(idx % groups), k0 = kg * 8;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (m < M && k0 < K) {  // K is a multiple of 8: a group is all inside or all outside
    v = *reinterpret_cast<const uint4 *>(src + (size_t)m * K + k0);
    if (gain) {
      __half2 *h = reinterpret_cast<__half2 *>(&v);
      const __half2 *gh = reinterpret_cast<const __half2 *>(gain + k0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 w = __half22float2(h[e]), gg = __half22float2(gh[e]);
        h[e] = __floats2half2_rn(w.x * gg.x, w.y * gg.y);
      }
    }
  }
  *reinterpret_cast<uint4 *>(A + ((size_t)(m / TC_M) * KT + k0 / TC_KT) * TC_A_BYTES + tc_tile_offset(m % TC_M, k0 % TC_KT)) = v;
}

}  // namespace kie
