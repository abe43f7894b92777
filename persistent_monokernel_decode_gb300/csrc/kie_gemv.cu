// Standalone batch-1 GEMV (y = W x, fp16 weights, fp32 accumulation) built from the same producer ring and
// tile consumer as the decode kernel, plus the kernel that packs a row-major matrix into the per-CTA tile
// layout (kie_layout.h). The pages' GEMV is the batch-1 workhorse ("math kernels are rewritten for batch 1":
// every matmul is a GEMV, matrix cores stay idle); on GB300 it runs on the CUDA cores with weights moved by
// the bulk-copy engine.
#include <cuda_runtime.h>

#include "kie_device.cuh"

namespace kie {

struct GemvParams {
  const uint8_t *packed;
  const __half *x;
  float *y;
  int M, K, n_cta, nslot, vec_floats, out_floats;
  unsigned long long timeout_ns;
};

// Status word of the standalone GEMV's bounded waits (set only if a wait runs out).
__device__ int g_gemv_status;

__global__ void __launch_bounds__(BLOCK, 1) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem s = carve_smem(smem_raw, p.nslot, p.vec_floats, p.out_floats);
  init_ring(s, p.nslot);
  const Guard g{&g_gemv_status, p.timeout_ns};
  const RowRange rr = rows_of_cta(p.M, p.n_cta, blockIdx.x);
  if (threadIdx.x >= NCT) {
    if (threadIdx.x == NCT) {
      RingPos rp{0, 0u, 0};
      produce_region(p.packed + (size_t)rr.r0 * p.K * 2, rr.r1 - rr.r0, p.K, s, p.nslot, rp,
                     l2_evict_first_policy(), g);
      drain_ring(s, p.nslot, rp, g);
    }
    return;
  }
  RingPos rp{0, 0u, 0};
  stage_f16(s, p.x, p.K, false);
  consume_region(s, p.nslot, rp, rr.r1 - rr.r0, p.K, 1.0f, g);
  consumer_sync();
  for (int i = threadIdx.x; i < rr.r1 - rr.r0; i += NCT) p.y[rr.r0 + i] = s.out[i];
}

// dst = packed(src) for a row-major [M, K] fp16 matrix; if gain is not null, every column c is first
// multiplied by gain[c] in fp32 and rounded back to fp16 (round to nearest even): the RMSNorm gain fold.
// One thread moves 8 consecutive elements (16 bytes) of one row.
__global__ void pack_kernel(const uint16_t *src, uint16_t *dst, int M, int K, int n, const uint16_t *gain) {
  const long long chunks = (long long)M * (K / 8);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < chunks;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / (K / 8));
    const int c = (int)(idx % (K / 8)) * 8;
    uint4 v = *reinterpret_cast<const uint4 *>(src + (size_t)r * K + c);
    if (gain) {
      __half2 *h = reinterpret_cast<__half2 *>(&v);
      const __half2 *gh = reinterpret_cast<const __half2 *>(gain + c);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 w = __half22float2(h[e]), gg = __half22float2(gh[e]);
        h[e] = __floats2half2_rn(w.x * gg.x, w.y * gg.y);
      }
    }
    *reinterpret_cast<uint4 *>(dst + packed_offset(M, K, n, r, c)) = v;
  }
}

// dst = packed(src) for FP8 codes [M, K] (packed_offset_fp8: column blocks of FP8_TILE_COLS codes, chunks of
// odd rows swizzled in full blocks). With b == null row r is
// a[r]; otherwise rows interleave two [M/2, K] matrices: row 2i = a[i], row 2i + 1 = b[i] (gate/up pairs).
// One thread moves 16 consecutive codes of one row; K is a multiple of 16.
__global__ void pack_fp8_kernel(const uint8_t *a, const uint8_t *b, uint8_t *dst, int M, int K, int n) {
  const long long chunks = (long long)M * (K / 16);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < chunks;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / (K / 16));
    const int c = (int)(idx % (K / 16)) * 16;
    const uint8_t *src = b ? ((r & 1) ? b : a) + (size_t)(r >> 1) * K + c : a + (size_t)r * K + c;
    *reinterpret_cast<uint4 *>(dst + packed_offset_fp8(M, K, n, r, c)) = *reinterpret_cast<const uint4 *>(src);
  }
}

// The sparse-MoE router folded through the WO projection: out[e][k] = sum_j rg[e][j] * wo[j][k] for an fp32
// [E, d] matrix rg (the router with the FFN RMSNorm gain applied) and the fp16 [d, dq] matrix Wo, accumulated in
// fp64 in index order and rounded to fp32. One thread per output; a warp's threads share e, so rg is a
// broadcast and Wo is read in coalesced rows.
__global__ void fold_router_kernel(const float *rg, const uint16_t *wo, float *out, int E, int d, int dq) {
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)E * dq) return;
  const int e = (int)(idx / dq), k = (int)(idx % dq);
  double acc = 0.0;
  for (int j = 0; j < d; ++j) {
    __half_raw r;
    r.x = wo[(size_t)j * dq + k];
    acc = fma((double)rg[(size_t)e * d + j], (double)__half2float(__half(r)), acc);
  }
  out[idx] = (float)acc;
}

}  // namespace kie

cudaError_t kie_launch_fold_router(const float *rg, const uint16_t *wo, float *out, int E, int d, int dq,
                                   cudaStream_t stream) {
  const long long n = (long long)E * dq;
  kie::fold_router_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(rg, wo, out, E, d, dq);
  return cudaGetLastError();
}

cudaError_t kie_launch_pack_fp8(const uint8_t *a, const uint8_t *b, uint8_t *dst, int M, int K, int n_cta,
                                cudaStream_t stream) {
  const long long chunks = (long long)M * (K / 16);
  int blocks = (int)((chunks + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  kie::pack_fp8_kernel<<<blocks, 256, 0, stream>>>(a, b, dst, M, K, n_cta);
  return cudaGetLastError();
}

cudaError_t kie_launch_gemv(const uint8_t *packed, const __half *x, float *y, int M, int K, int n_cta, int nslot,
                            unsigned long long timeout_ns, cudaStream_t stream) {
  kie::GemvParams p;
  p.packed = packed;
  p.x = x;
  p.y = y;
  p.M = M;
  p.K = K;
  p.n_cta = n_cta;
  p.nslot = nslot;
  p.vec_floats = K;
  p.out_floats = (M / 2 + n_cta - 1) / n_cta * 2 + 2;
  p.timeout_ns = timeout_ns;
  const size_t smem = kie::smem_bytes(nslot, p.vec_floats, p.out_floats);
  cudaError_t e = cudaFuncSetAttribute(kie::gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kie::gemv_kernel<<<n_cta, kie::BLOCK, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t kie_launch_pack(const uint16_t *src, uint16_t *dst, int M, int K, int n_cta, const uint16_t *gain,
                            cudaStream_t stream) {
  const long long chunks = (long long)M * (K / 8);
  int blocks = (int)((chunks + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  kie::pack_kernel<<<blocks, 256, 0, stream>>>(src, dst, M, K, n_cta, gain);
  return cudaGetLastError();
}
