// Batched prefill: a prompt's tokens go through each layer together, in chunks of up to PF_TOKENS, so every
// weight is read once per chunk instead of once per token. Same arithmetic as the decode kernel (fp16 weights
// with the RMSNorm gains folded, fp32 activations and accumulation, RoPE from the fp32 table, fp16 K/V cache,
// max-subtracted softmax), on the same packed weights; the prompt is part of the decode problem (the pages' 2B
// workload has a 4,096-token sequence), not a different model path.
//
// Kernels, per chunk of T tokens:
//   pf_embed  X[t] = fp32(E[tok[t]])
//   per layer: pf_rms(X) -> projection QKV (RoPE, K/V append, q) -> ta_attn (causal, over the cache) ->
//              projection WO (H = X + Wo o) -> pf_rms(H) -> projection GU (A = silu(g) u) -> projection DOWN
//              (X = H + Wd a)
//   after the last chunk: pf_rms(last X) -> pf_gemm LM head (one token, CUDA cores) -> pf_argmax (next token)
// A projection is a tensor-core GEMM (kie_tcgemm.cuh: the chunk's activations split into fp16 high and low
// parts, tcgen05.mma into TMEM, K split over blocks so that every SM has one) followed by pf_reduce, which adds
// the K splits in order and applies the epilogue. The attention is a tensor-core kernel too (kie_tcattn.cuh:
// one block per query head and 512-position piece; pf_attn_merge combines the pieces of long contexts). No sum's order depends on how the prompt is cut into chunks
// (a token's column of the MMA is computed like any other), so a prompt prefilled in pieces leaves bit-identical
// logits and cache.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kie.h"
#include "kie_decode.cuh"
#include "kie_layout.h"
#include "kie_prefill.cuh"
#include "kie_tcattn.cuh"
#include "kie_tcgemm.cuh"

namespace kie {
namespace {

constexpr int PF_THREADS = 256;
constexpr int PA_PIECE = PF_ATT_PIECE;  // positions per attention piece (fixed boundaries 0, 512, 1024, ...)
constexpr int GR = TILE_ROWS;    // output rows per block pass (a row group of the packed layout)
constexpr int KC = 32;           // columns per shared-memory stage
constexpr int XS = PF_TOKENS + 4;  // padded token stride of the staged input (bank spread)

enum Epi { EPI_QKV = 0, EPI_WO = 1, EPI_GU = 2, EPI_DOWN = 3, EPI_LM = 4 };

struct GemmArgs {
  const uint8_t *w;      // LM head: packed [M, K] (all CTAs' regions)
  int M, K, n_cta;       // rows, columns, CTAs the layout was packed for
  const float *in;       // [T][K] token-major input rows
  const float *scale;    // [T] per-token RMS scale, or null (1)
  int T;
  // epilogues
  float *out;            // WO/DOWN: [T][M]; GU: [T][M/2]; QKV: q [T][Hq*dh]; LM: [M]
  const float *resid;    // WO/DOWN: [T][M]
  __half *kv;            // QKV: this layer's K plane base ([2][Hkv][max_seq][dh])
  const float2 *rope;    // QKV: [max_seq][dh/2]
  int pos0, Hq, Hkv, dh, max_seq;
  // pf_reduce input: the raw sums of ksplit K splits, part[ksplit][PF_TOKENS][M], added in order
  int ksplit;
  float *part;
};

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Epilogue of the row pair (r, r + 1) of token t from their raw sums s0, s1 (QKV: RoPE, then q to out or k/v
// to the fp16 cache; GU: SwiGLU). Pairs are RoPE halves or gate/up rows, adjacent in the packed order.
template <int EPI>
__device__ __forceinline__ void epi_pair(const GemmArgs &a, int t, int r, float s0, float s1) {
  const float sc = a.scale ? a.scale[t] : 1.0f;
  const float y0 = s0 * sc, y1 = s1 * sc;
  if (EPI == EPI_GU) {
    a.out[(size_t)t * (a.M / 2) + r / 2] = silu_mul(y0, y1);
  } else {
    const int dh = a.dh, qrows = a.Hq * dh, krows = a.Hkv * dh, pos = a.pos0 + t;
    const size_t plane = (size_t)a.max_seq * dh;
    if (r < qrows + krows) {
      const int rq = r < qrows ? r : r - qrows;
      const float2 cs = a.rope[(size_t)pos * (dh / 2) + (rq % dh) / 2];
      const float a2 = y0 * cs.x - y1 * cs.y, b2 = y1 * cs.x + y0 * cs.y;
      if (r < qrows) {
        *reinterpret_cast<float2 *>(a.out + (size_t)t * qrows + r) = make_float2(a2, b2);
      } else {
        *reinterpret_cast<__half2 *>(a.kv + (size_t)(rq / dh) * plane + (size_t)pos * dh + rq % dh) =
            __floats2half2_rn(a2, b2);
      }
    } else {
      const int rv = r - qrows - krows;
      *reinterpret_cast<__half2 *>(a.kv + (size_t)a.Hkv * plane + (size_t)(rv / dh) * plane + (size_t)pos * dh +
                                   rv % dh) = __floats2half2_rn(y0, y1);
    }
  }
}

// Epilogue of row r of token t from its raw sum s (WO/DOWN: residual add; LM: logits of the one token).
template <int EPI>
__device__ __forceinline__ void epi_one(const GemmArgs &a, int t, int r, float s) {
  const float y = s * (a.scale ? a.scale[t] : 1.0f);
  if (EPI == EPI_LM) a.out[r] = y;
  else a.out[(size_t)t * a.M + r] = a.resid[(size_t)t * a.M + r] + y;
}

// out rows of row group blockIdx.y of CTA region blockIdx.x (rows [r0, r1) of the decode's row split), for
// T <= PF_TOKENS tokens. Thread (ty, tx) owns rows 4ty .. 4ty+3 of the group and tokens 4tx .. 4tx+3; every
// output is one fp32 FMA chain over k in ascending order.
template <int EPI>
__global__ void __launch_bounds__(PF_THREADS) pf_gemm(const GemmArgs a) {
  __shared__ __align__(16) float Ws[KC][GR];       // W chunk, transposed: [k][row]
  __shared__ __align__(16) float Xs[KC][XS];       // input chunk, transposed: [k][token]
  const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
  const RowRange rr = rows_of_cta(a.M, a.n_cta, blockIdx.x);
  const int R = rr.r1 - rr.r0, K = a.K;
  const __half *region = reinterpret_cast<const __half *>(a.w) + (size_t)rr.r0 * K;
  {
    const int g0 = (int)blockIdx.y * GR;
    if (g0 >= R) return;
    const int k_lo = 0, k_hi = K;
    const int rows = min(GR, R - g0);
    const int bw = TILE_COLS;  // the packed layout's column blocks
    const __half *gbase = region + (size_t)g0 * K;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    // 32-column stages over k = 0 .. K in order; the next stage's W and input values are loaded into registers
    // while this stage's products run (the packed tile of column kcol is the one of block kcol / bw)
    float f[4];
    float4 v[PF_TOKENS * KC / 4 / PF_THREADS];
    auto load = [&](int kcol) {
      const int b0 = kcol / bw * bw, w = min(bw, K - b0), kc = kcol - b0;
      const __half *tile = gbase + (size_t)rows * b0;  // [rows][w] row-major
      const int r = tid >> 3, c = (tid & 7) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) f[e] = 0.f;
      if (r < rows && kc + c < w) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(tile + (size_t)r * w + kc + c);
        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
        f[0] = lo.x;
        f[1] = lo.y;
        f[2] = hi.x;
        f[3] = hi.y;
      }
#pragma unroll
      for (int i = 0; i < PF_TOKENS * KC / 4 / PF_THREADS; ++i) {
        const int idx = tid + i * PF_THREADS, t = idx >> 3, cc = (idx & 7) * 4;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < a.T && kc + cc < w) v[i] = *reinterpret_cast<const float4 *>(a.in + (size_t)t * K + kcol + cc);
      }
    };
    load(k_lo);
    for (int kcol = k_lo; kcol < k_hi; kcol += KC) {
      {
        const int r = tid >> 3, c = (tid & 7) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) Ws[c + e][r] = f[e];
#pragma unroll
        for (int i = 0; i < PF_TOKENS * KC / 4 / PF_THREADS; ++i) {
          const int idx = tid + i * PF_THREADS, t = idx >> 3, cc = (idx & 7) * 4;
          Xs[cc][t] = v[i].x;
          Xs[cc + 1][t] = v[i].y;
          Xs[cc + 2][t] = v[i].z;
          Xs[cc + 3][t] = v[i].w;
        }
      }
      __syncthreads();
      if (kcol + KC < k_hi) load(kcol + KC);
#pragma unroll 8
      for (int k = 0; k < KC; ++k) {
        const float4 wv = *reinterpret_cast<const float4 *>(&Ws[k][4 * ty]);
        const float4 xv = *reinterpret_cast<const float4 *>(&Xs[k][4 * tx]);
        const float wr[4] = {wv.x, wv.y, wv.z, wv.w}, xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(wr[i], xr[jj], acc[i][jj]);
      }
      __syncthreads();
    }
    // epilogue (or the raw sums of this K slice): rows g0 + 4ty + i (< R), tokens 4tx + j (< T)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 4 * tx + j;
      if (t >= a.T) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int lr = g0 + 4 * ty + i;
        if (lr >= R) continue;
        const int r = rr.r0 + lr;
        if (EPI == EPI_QKV || EPI == EPI_GU) {
          if ((i & 1) == 0) epi_pair<EPI>(a, t, r, acc[i][j], acc[i + 1][j]);  // R and g0 even: pairs whole
        } else {
          epi_one<EPI>(a, t, r, acc[i][j]);
        }
      }
    }
  }
}

// The split-K sums: slices added in order (a fixed order, whatever the chunking), then the epilogue.
template <int EPI>
__global__ void pf_reduce(const GemmArgs a) {
  const int per_t = (EPI == EPI_QKV || EPI == EPI_GU) ? a.M / 2 : a.M;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)a.T * per_t) return;
  const int t = (int)(idx / per_t), u = (int)(idx % per_t);
  auto sum = [&](int r) {
    float v = a.part[(size_t)t * a.M + r];
    for (int k = 1; k < a.ksplit; ++k) v += a.part[((size_t)k * PF_TOKENS + t) * a.M + r];
    return v;
  };
  if (EPI == EPI_QKV || EPI == EPI_GU) epi_pair<EPI>(a, t, 2 * u, sum(2 * u), sum(2 * u + 1));
  else epi_one<EPI>(a, t, u, sum(u));
}

// scale[t] = 1 / sqrt(mean(x_t^2) + eps), one warp per token, lane-strided sums then a fixed tree.
__global__ void pf_rms(const float *x, int T, int d, float eps, float *scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float *row = x + (size_t)warp * d;
  float s = 0.f;
  for (int i = lane; i < d; i += 32) s = fmaf(row[i], row[i], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) scale[warp] = 1.0f / sqrtf(s / (float)d + eps);
}

__global__ void pf_embed(const int *tok, int T, const __half *E, int d, float *x) {
  const int t = blockIdx.x;
  if (t >= T) return;
  const __half *row = E + (size_t)tok[t] * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) x[(size_t)t * d + i] = __half2float(row[i]);
}

// o of the tokens whose positions span several pieces: pieces in ascending order, w_z = exp(m_z - M),
// o = sum_z w_z o_z / sum_z w_z l_z. Block: one token and one query head, a thread per dimension.
__global__ void pf_attn_merge(int T, int pos0, int Hq, int DH, const float *po, const float *pml, float *o) {
  const int t = blockIdx.x, hq = blockIdx.y, e = threadIdx.x, pos = pos0 + t;
  if (pos < PA_PIECE || e >= DH) return;
  const int S = pos / PA_PIECE + 1;
  const size_t oi = (size_t)t * Hq + hq, stride = (size_t)T * Hq;
  float M = -INFINITY;
  for (int zz = 0; zz < S; ++zz) M = fmaxf(M, pml[(zz * stride + oi) * 2]);
  float num = 0.f, den = 0.f;
  for (int zz = 0; zz < S; ++zz) {
    const float w = expf(pml[(zz * stride + oi) * 2] - M);
    den += w * pml[(zz * stride + oi) * 2 + 1];
    num += w * po[(zz * stride + oi) * DH + e];
  }
  o[oi * DH + e] = num / den;
}

// argmax over the logits (lowest index on ties), written as the next token to emit.
__global__ void pf_argmax(const float *logits, int V, Persist *persist) {
  __shared__ unsigned long long best[32];
  unsigned long long b = 0ull;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const unsigned u = __float_as_uint(logits[i]);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const unsigned long long key = ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
    b = key > b ? key : b;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, b, o);
    b = other > b ? other : b;
  }
  if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = best[w] > m ? best[w] : m;
    persist->next_token = (int)(0xFFFFFFFFu - (unsigned)(m & 0xFFFFFFFFull));
  }
}

// The LM head of the last prompt token (a GEMV: T = 1) on the decode's packed weights.
cudaError_t lm_head(GemmArgs a, cudaStream_t st) {
  const int groups = (2 * ((a.M / 2 + a.n_cta - 1) / a.n_cta) + GR - 1) / GR;  // row groups of the largest region
  a.ksplit = 1;
  a.part = nullptr;
  pf_gemm<EPI_LM><<<dim3(a.n_cta, groups), PF_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

// One projection of the chunk on the tensor cores: split a.in into hi/lo tiles, the GEMM of the K splits into
// b.part, then pf_reduce (splits in order + epilogue).
template <int EPI>
cudaError_t tc_project(GemmArgs a, const uint8_t *w_tiles, const PrefillBufs &b, cudaStream_t st) {
  const int KT = (a.K + TC_KT - 1) / TC_KT, Mt = (a.M + TC_M - 1) / TC_M;
  int kps, ns;
  kie_tc_splits(Mt, KT, a.n_cta, &kps, &ns);
  const long long nb = (long long)TC_N * KT * (TC_KT / 8);
  tc_split_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(a.in, a.T, a.K, KT, b.tc_b);
  const TcArgs t{w_tiles, b.tc_b, KT, kps, b.part, a.M, a.T, b.status, b.timeout_ns};
  tc_gemm_kernel<<<dim3(Mt, ns), TC_THREADS, TC_SMEM, st>>>(t);
  a.ksplit = ns;
  a.part = b.part;
  const long long n = (long long)a.T * ((EPI == EPI_QKV || EPI == EPI_GU) ? a.M / 2 : a.M);
  pf_reduce<EPI><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace kie

cudaError_t kie_run_prefill(const kie::DecodeParams &p, const kie::PrefillBufs &b, const int *tok_dev, int pos0,
                            int n, cudaStream_t st) {
  using namespace kie;
  const int d = p.d, dq = p.Hq * p.dh, F = p.F, qkv = (p.Hq + 2 * p.Hkv) * p.dh;
  const size_t plane = (size_t)p.max_seq * p.dh;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ta_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ta_smem_bytes<128>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ta_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ta_smem_bytes<64>());
  if (e != cudaSuccess) return e;
  int last_t = 0;
  for (int c0 = 0; c0 < n; c0 += PF_TOKENS) {
    const int T = n - c0 < PF_TOKENS ? n - c0 : PF_TOKENS, pos = pos0 + c0;
    last_t = T - 1;
    pf_embed<<<T, 256, 0, st>>>(tok_dev + c0, T, p.embed, d, b.x);
    const int rms_blocks = (T * 32 + 255) / 256;
    for (int l = 0; l < p.L; ++l) {
      const uint8_t *tw = b.tc_w + (size_t)l * b.tc_layer_stride;
      __half *kvl = p.kv + (size_t)l * 2 * p.Hkv * plane;
      pf_rms<<<rms_blocks, 256, 0, st>>>(b.x, T, d, p.eps, b.scale);
      GemmArgs a{};
      a.n_cta = p.n_cta;
      a.T = T;
      a.pos0 = pos;
      a.Hq = p.Hq;
      a.Hkv = p.Hkv;
      a.dh = p.dh;
      a.max_seq = p.max_seq;
      a.rope = p.rope;
      a.kv = kvl;
      // QKV (+ RoPE, K/V append, q)
      a.M = qkv;
      a.K = d;
      a.in = b.x;
      a.scale = b.scale;
      a.out = b.q;
      if ((e = tc_project<EPI_QKV>(a, tw + b.tc_off[0], b, st)) != cudaSuccess) return e;
      // attention over positions 0 .. pos0 + t on the tensor cores, split into pieces of PA_PIECE positions
      const int pieces = (pos + T - 1) / PA_PIECE + 1;
      const TaArgs ta{b.q, kvl, b.o, b.att_o, b.att_ml, T, pos, p.Hq, p.Hkv, p.max_seq, b.status, b.timeout_ns};
      if (p.dh == 128)
        ta_attn_kernel<128><<<dim3(p.Hq, pieces), TA_THREADS, ta_smem_bytes<128>(), st>>>(ta);
      else
        ta_attn_kernel<64><<<dim3(p.Hq, pieces), TA_THREADS, ta_smem_bytes<64>(), st>>>(ta);
      if (pieces > 1) pf_attn_merge<<<dim3(T, p.Hq), p.dh, 0, st>>>(T, pos, p.Hq, p.dh, b.att_o, b.att_ml, b.o);
      // WO + residual
      a.M = d;
      a.K = dq;
      a.in = b.o;
      a.scale = nullptr;
      a.out = b.h;
      a.resid = b.x;
      if ((e = tc_project<EPI_WO>(a, tw + b.tc_off[1], b, st)) != cudaSuccess) return e;
      // gate/up + SwiGLU
      pf_rms<<<rms_blocks, 256, 0, st>>>(b.h, T, d, p.eps, b.scale);
      a.M = 2 * F;
      a.K = d;
      a.in = b.h;
      a.scale = b.scale;
      a.out = b.a;
      if ((e = tc_project<EPI_GU>(a, tw + b.tc_off[2], b, st)) != cudaSuccess) return e;
      // down + residual
      a.M = d;
      a.K = F;
      a.in = b.a;
      a.scale = nullptr;
      a.out = b.x;
      a.resid = b.h;
      if ((e = tc_project<EPI_DOWN>(a, tw + b.tc_off[3], b, st)) != cudaSuccess) return e;
    }
  }
  // logits of the last prompt token and the next token to emit
  const float *xl = b.x + (size_t)last_t * d;
  pf_rms<<<1, 32, 0, st>>>(xl, 1, d, p.eps, b.scale);
  kie::GemmArgs a{};
  a.w = p.w_lm;
  a.M = p.V;
  a.K = d;
  a.n_cta = p.n_cta;
  a.in = xl;
  a.scale = b.scale;
  a.T = 1;
  a.out = p.logits;
  if ((e = kie::lm_head(a, st)) != cudaSuccess) return e;
  kie::pf_argmax<<<1, 1024, 0, st>>>(p.logits, p.V, p.persist);
  return cudaGetLastError();
}

cudaError_t kie_launch_tc_pack(const uint16_t *src, int M, int K, const uint16_t *gain, uint8_t *dst, cudaStream_t st) {
  const int KT = (K + kie::TC_KT - 1) / kie::TC_KT, Mp = (M + kie::TC_M - 1) / kie::TC_M * kie::TC_M;
  const long long n = (long long)Mp * KT * (kie::TC_KT / 8);
  kie::tc_pack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(src, M, K, KT, gain, dst);
  return cudaGetLastError();
}

// Host-side layout query of include/kie.h: byte offset of W[r][c] in the tensor-core copy of an [M, K] matrix.
extern "C" int64_t kie_tc_tile_offset(int M, int K, int r, int c) {
  if (M < 1 || K < 8 || K % 8 || r < 0 || r >= M || c < 0 || c >= K) return -1;
  const int KT = (K + 63) / 64;
  return ((int64_t)(r / 128) * KT + c / 64) * (128 * 64 * 2) + kie::kie_tc_offset_in_tile(r % 128, c % 64);
}
