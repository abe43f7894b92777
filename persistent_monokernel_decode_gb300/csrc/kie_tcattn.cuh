// Tensor-core (tcgen05) causal attention of the batched prefill.
//
// A block is one query head h and one piece z of the cached positions [z * PF_ATT_PIECE, (z + 1) * PF_ATT_PIECE)
// for the chunk's T <= 128 tokens (one token per accumulator row / TMEM lane). Per 128-position key tile:
//   S = Q K^T on the tensor cores (Q fp32 split into fp16 hi + lo, two MMAs into one fp32 TMEM accumulator;
//   K fp16 from the cache), the causal mask and 1/sqrt(dh) applied when each thread reads its row of S back.
// Two passes over the piece: the first keeps the row maxima m, the second forms P = exp(S - m) (fp32, summed
// into l), writes P as fp16 hi + lo, and accumulates O += P V on the tensor cores (V transposed into the K-major
// operand layout while it is staged), so O never needs rescaling. A token whose positions fit in one piece
// writes o = O / l; otherwise the piece's partial (m, l, O) goes to the same buffers as the CUDA-core kernel's,
// and pf_attn_merge combines the pieces in order.
//
// Operands use the canonical K-major layout without swizzle (kie_tcgemm.cuh) with K tiles of width KW:
// element (r, k) at (r / 8) * KW * 16 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2, descriptor LBO 128 B,
// SBO KW * 16 B.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kie_tcgemm.cuh"

namespace kie {

constexpr int TA_M = 128;  // query rows (tokens) per block
constexpr int TA_N = 128;  // key positions per tile
constexpr int TA_THREADS = 128;

__host__ __device__ __forceinline__ int ta_offset(int r, int k, int kw) {
  return (r >> 3) * kw * 16 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ uint64_t ta_desc(uint32_t saddr, int kw) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)((kw * 16) >> 4) << 32) |
         ((uint64_t)1 << 46);
}

__host__ __device__ constexpr uint32_t ta_idesc(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TA_M >> 4) << 24);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte asynchronous global -> shared copy; bytes past src_bytes (0 or 16) are zero-filled.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

template <int DH>
constexpr size_t ta_smem_bytes() {
  return (size_t)2 * TA_M * DH * 2    // Q hi, lo
         + (size_t)TA_N * DH * 2      // K tile
         + (size_t)2 * TA_M * TA_N * 2  // P hi, lo
         + (size_t)DH * TA_N * 2;     // V^T tile
}

struct TaArgs {
  const float *q;       // [T][Hq][DH] fp32 (RoPE applied), this chunk
  const __half *kvl;    // this layer's cache: K planes [Hkv][max_seq][DH], then V planes
  float *o;             // [T][Hq][DH]
  float *po, *pml;      // partials [piece][T][Hq][DH], [piece][T][Hq][2]
  int T, pos0, Hq, Hkv, max_seq;
  int *status;
  unsigned long long timeout_ns;
};

template <int DH>
__global__ void __launch_bounds__(TA_THREADS, 1) ta_attn_kernel(const TaArgs a) {
  extern __shared__ __align__(1024) uint8_t ta_smem[];
  __shared__ __align__(8) uint64_t mbar;
  __shared__ uint32_t tmem_base;
  uint8_t *sQh = ta_smem, *sQl = sQh + TA_M * DH * 2, *sK = sQl + TA_M * DH * 2;
  uint8_t *sPh = sK + TA_N * DH * 2, *sPl = sPh + TA_M * TA_N * 2, *sV = sPl + TA_M * TA_N * 2;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x, z = blockIdx.y, G = a.Hq / a.Hkv, kh = h / G;
  const int jlo = z * PF_ATT_PIECE;
  const int jhi = min(jlo + PF_ATT_PIECE, a.pos0 + a.T);  // exclusive: no token attends past its own position
  if (jlo >= jhi) return;
  const Guard g{a.status, a.timeout_ns};
  const size_t plane = (size_t)a.max_seq * DH;
  const __half *Kb = a.kvl + (size_t)kh * plane, *Vb = a.kvl + (size_t)(a.Hkv + kh) * plane;

  if (tid == 0) {
    mbar_init(&mbar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);  // S: columns [0, 128); O: [128, 128 + DH)
    tmem_relinquish();
  }
  // Q of the chunk's tokens for head h, split into hi / lo (rows past T are zero)
  for (int i = tid; i < TA_M * (DH / 8); i += TA_THREADS) {
    const int t = i / (DH / 8), k0 = (i % (DH / 8)) * 8;
    __align__(16) __half hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float v = t < a.T ? a.q[((size_t)t * a.Hq + h) * DH + k0 + e] : 0.f;
      hi[e] = __float2half_rn(v);
      lo[e] = __float2half_rn(v - __half2float(hi[e]));
    }
    *reinterpret_cast<uint4 *>(sQh + ta_offset(t, k0, DH)) = *reinterpret_cast<const uint4 *>(hi);
    *reinterpret_cast<uint4 *>(sQl + ta_offset(t, k0, DH)) = *reinterpret_cast<const uint4 *>(lo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base, tS = tmem, tO = tmem + TA_N;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const int row = tid;  // this thread's token = TMEM lane
  const int pos = a.pos0 + row;
  const bool live = row < a.T && pos >= jlo;
  const float scale = rsqrtf((float)DH);
  uint32_t nmma = 0;  // completions of mbar so far
  bool ok = true;

  // stage K (and, if with_v, V transposed) for positions [kt, kt + TA_N) (zero past jhi). K moves by
  // asynchronous copies; the thread's V loads are all issued before the transposing stores, so every load of
  // the tile is in flight at once.
  constexpr int PER = TA_N * (DH / 8) / TA_THREADS;  // 16-byte pieces per thread per tile
  static_assert(TA_N * (DH / 8) % TA_THREADS == 0, "tile pieces split evenly over the block");
  auto stage = [&](int kt, bool with_v) {
    uint4 vv[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + u * TA_THREADS, p = i / (DH / 8), k0 = (i % (DH / 8)) * 8, j = kt + p;
      const bool in = j < jhi;
      cp_async16(sK + ta_offset(p, k0, DH), Kb + (in ? (size_t)j * DH + k0 : 0), in ? 16u : 0u);
      if (with_v) vv[u] = in ? *reinterpret_cast<const uint4 *>(Vb + (size_t)j * DH + k0) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (with_v) {
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = tid + u * TA_THREADS, p = i / (DH / 8), k0 = (i % (DH / 8)) * 8;
        const __half *vh = reinterpret_cast<const __half *>(&vv[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) *reinterpret_cast<__half *>(sV + ta_offset(k0 + e, p, TA_N)) = vh[e];
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();
  };
  // S = Q K^T into TMEM columns [0, 128), then wait for it
  auto mma_s = [&]() {
    if (tid == 0) {
      tc_fence_after();
      const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl), kb = smem_u32(sK);
#pragma unroll
      for (int s = 0; s < DH / 16; ++s)
        tc_mma(tS, ta_desc(qh + 256 * s, DH), ta_desc(kb + 256 * s, DH), ta_idesc(TA_N), s > 0 ? 1u : 0u);
#pragma unroll
      for (int s = 0; s < DH / 16; ++s)
        tc_mma(tS, ta_desc(ql + 256 * s, DH), ta_desc(kb + 256 * s, DH), ta_idesc(TA_N), 1u);
      tc_commit(&mbar);
    }
    __syncwarp();
    ok = wait_mbar(&mbar, nmma++ & 1u, g) && ok;
    tc_fence_after();
  };
  // this thread's row of S for columns [c0, c0 + 16), masked and scaled (-inf where not attended)
  auto s_chunk = [&](int kt, int c0, float (&v)[16]) {
    tmem_ld16(tS + lane_base + (uint32_t)c0, v);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int j = kt + c0 + e;
      v[e] = (live && j <= pos && j < jhi) ? v[e] * scale : -INFINITY;
    }
  };

  // pass 1: row maxima over the piece
  float m = -INFINITY;
  for (int kt = jlo; kt < jhi; kt += TA_N) {
    stage(kt, false);
    mma_s();
    for (int c0 = 0; c0 < TA_N; c0 += 16) {
      float v[16];
      s_chunk(kt, c0, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) m = fmaxf(m, v[e]);
    }
    tc_fence_before();
    __syncthreads();  // every row read before the next tile's MMAs overwrite S
  }
  // pass 2: P = exp(S - m), l = sum P, O += P V
  float l = 0.f;
  bool first = true;
  for (int kt = jlo; kt < jhi; kt += TA_N) {
    stage(kt, true);
    mma_s();
    for (int c0 = 0; c0 < TA_N; c0 += 16) {
      float v[16];
      s_chunk(kt, c0, v);
      __align__(16) __half ph[16], pl[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float p = v[e] == -INFINITY ? 0.f : expf(v[e] - m);
        l += p;
        ph[e] = __float2half_rn(p);
        pl[e] = __float2half_rn(p - __half2float(ph[e]));
      }
      *reinterpret_cast<uint4 *>(sPh + ta_offset(row, c0, TA_N)) = *reinterpret_cast<const uint4 *>(ph);
      *reinterpret_cast<uint4 *>(sPh + ta_offset(row, c0 + 8, TA_N)) = *reinterpret_cast<const uint4 *>(ph + 8);
      *reinterpret_cast<uint4 *>(sPl + ta_offset(row, c0, TA_N)) = *reinterpret_cast<const uint4 *>(pl);
      *reinterpret_cast<uint4 *>(sPl + ta_offset(row, c0 + 8, TA_N)) = *reinterpret_cast<const uint4 *>(pl + 8);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ph = smem_u32(sPh), pl = smem_u32(sPl), vb = smem_u32(sV);
#pragma unroll
      for (int s = 0; s < TA_N / 16; ++s)
        tc_mma(tO, ta_desc(ph + 256 * s, TA_N), ta_desc(vb + 256 * s, TA_N), ta_idesc(DH), (!first || s > 0) ? 1u : 0u);
#pragma unroll
      for (int s = 0; s < TA_N / 16; ++s)
        tc_mma(tO, ta_desc(pl + 256 * s, TA_N), ta_desc(vb + 256 * s, TA_N), ta_idesc(DH), 1u);
      tc_commit(&mbar);
    }
    __syncwarp();
    ok = wait_mbar(&mbar, nmma++ & 1u, g) && ok;  // P, V and K smem are free again
    tc_fence_after();
    first = false;
  }
  // O / l, or the piece's partial
  const bool single = pos < PF_ATT_PIECE;
  const size_t oi = (size_t)row * a.Hq + h;
  for (int c0 = 0; c0 < DH; c0 += 16) {
    float v[16];
    tmem_ld16(tO + lane_base + (uint32_t)c0, v);
    if (ok && live) {
      if (single) {
        const float inv = 1.0f / l;
#pragma unroll
        for (int e = 0; e < 16; ++e) a.o[oi * DH + c0 + e] = v[e] * inv;
      } else {
        const size_t pi = (size_t)z * a.T * a.Hq + oi;
#pragma unroll
        for (int e = 0; e < 16; ++e) a.po[pi * DH + c0 + e] = v[e];
      }
    }
  }
  if (ok && live && !single) {
    const size_t pi = (size_t)z * a.T * a.Hq + oi;
    a.pml[pi * 2] = m;
    a.pml[pi * 2 + 1] = l;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace kie
