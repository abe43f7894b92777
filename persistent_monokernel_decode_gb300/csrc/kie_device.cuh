// Device building blocks shared by the persistent decode kernel and the standalone GEMV kernel.
//
// Every CTA runs NCW consumer warps and one producer warpgroup, whose first lane is the producer and whose
// registers mostly go to the consumers (setmaxnreg). The producer walks the CTA's
// static sequence of weight tiles (it does not depend on any activation) and moves each tile from HBM
// into a shared-memory ring slot with one 1-D bulk copy (cp.async.bulk, completion counted on the slot's
// "full" mbarrier, L2 evict-first policy). Consumers wait on "full", run their part of the dot products
// from shared memory, and release the slot on its "empty" mbarrier. Because the producer never waits for
// a grid barrier, weight loads stay in flight while the consumers synchronise with the rest of the grid:
// the in-kernel weight prefetch of the monokernel pages ("inside the monokernel": FFN weights are
// prefetched while attention runs), done here by the GB300's bulk-copy engine.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>
#include <stdint.h>

#include "kie_layout.h"

namespace kie {

constexpr int NCW = 8;                          // consumer warps
constexpr int NCT = NCW * 32;                   // consumer threads
constexpr int BLOCK = NCT + 128;                // + one producer warpgroup (one lane streams the weights)
// Register split of the decode kernel (setmaxnreg): the block launches with LAUNCH_REGS per thread, the producer
// warpgroup drops to PRODUCER_REGS and hands the rest to the two consumer warpgroups, which rise to
// CONSUMER_REGS. The counts must balance exactly against the launch, or the consumers' increase would wait for
// registers that never come: the launch path checks the compiled count before every launch.
constexpr int LAUNCH_REGS = 168, PRODUCER_REGS = 40, CONSUMER_REGS = 232;
static_assert(NCT * CONSUMER_REGS + (BLOCK - NCT) * PRODUCER_REGS <= BLOCK * LAUNCH_REGS,
              "the register split must fit in the launch allocation");
static_assert(BLOCK * LAUNCH_REGS <= 65536, "one block per SM");
constexpr int ROWS_PER_WARP = TILE_ROWS / NCW;  // rows of a tile each consumer warp owns
constexpr int FP8_RED_FLOATS = (NCW + 1) * TILE_ROWS;  // partial sums of one FP8 row group
static_assert(TILE_ROWS % NCW == 0, "tile rows must split evenly over consumer warps");

constexpr int ST_OK = 0;
constexpr int ST_TIMEOUT = 1;

// ---- PTX wrappers --------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One contiguous global -> shared bulk copy; bytes and both addresses are multiples of 16.
// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned address and size); no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release add at GPU scope, no reply: the thread's earlier accesses, and those ordered before them by a CTA
// barrier, happen before the increment for any thread that observes it with an acquire load.
__device__ __forceinline__ void red_release_gpu_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_gpu(const int *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Register reallocation between warpgroups (all threads of a warpgroup execute the same one).
template <int N>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void regs_acquire() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}

// Named barrier 1: the NCT consumer threads of this CTA (the producer warpgroup never joins it).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---- warp-level tensor-core fragments (mma.sync m16n8k16, fp16 inputs, fp32 accumulators) -----------------
//
// Fragment ownership (g = lane / 4, t = lane % 4): A (16 x 16, row-major) a0 = rows g, cols 2t..2t+1;
// a1 = row g + 8; a2 = row g, cols + 8; a3 = row g + 8, cols + 8. B (16 x 8, k x n) b0 = k 2t..2t+1, n g;
// b1 = k + 8. C/D (16 x 8) c0, c1 = row g, cols 2t, 2t + 1; c2, c3 = row g + 8, same cols.

// Four 8x8 fp16 matrices from shared memory; lanes 8i..8i+7 give the row addresses of matrix i (16-byte rows).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row))
               : "memory");
}

// Two 8x8 fp16 matrices (lanes 0..15 give the row addresses; the others' are not used).
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(row))
               : "memory");
}

// As ldsm_x2, each matrix transposed on the way (row-major k x n storage -> the B fragment).
__device__ __forceinline__ void ldsm_x2_trans(uint32_t (&r)[2], const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(row))
               : "memory");
}

// d += A B on one 16x8x16 tile (registers only: the compiler may schedule it freely).
__device__ __forceinline__ void mma_f16_f32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- shared memory ---------------------------------------------------------------------------------------

struct Smem {
  uint8_t *ring;           // nslot * SLOT_BYTES
  float *vec;              // the phase's input vector (fp32), also attention scratch
  float *out;              // per-CTA row results of the current projection
  uint64_t *full, *empty;  // ring mbarriers
  float *red;              // NCW floats of cross-warp reduction scratch
  unsigned long long *kred;  // NCW keys of cross-warp argmax scratch
  volatile int *flags;     // [0] abort, [1] last-arriver flag
  float *scal;             // [0] inv_rms
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte size of the dynamic shared memory for a ring of nslot slots, vec_floats input-vector floats and
// out_floats row results.
__host__ __device__ inline size_t smem_bytes(int nslot, int vec_floats, int out_floats) {
  size_t o = (size_t)nslot * SLOT_BYTES;
  o += align_up((size_t)vec_floats * 4, 128);
  o += align_up((size_t)out_floats * 4, 128);
  o += 2 * (size_t)nslot * 8;
  o += NCW * 4 + NCW * 8 + 16 + 16;
  return align_up(o, 128);
}

__device__ inline Smem carve_smem(uint8_t *base, int nslot, int vec_floats, int out_floats) {
  Smem s;
  size_t o = 0;
  s.ring = base;
  o += (size_t)nslot * SLOT_BYTES;
  s.vec = (float *)(base + o);
  o += align_up((size_t)vec_floats * 4, 128);
  s.out = (float *)(base + o);
  o += align_up((size_t)out_floats * 4, 128);
  s.full = (uint64_t *)(base + o);
  o += (size_t)nslot * 8;
  s.empty = (uint64_t *)(base + o);
  o += (size_t)nslot * 8;
  s.kred = (unsigned long long *)(base + o);
  o += NCW * 8;
  s.red = (float *)(base + o);
  o += NCW * 4;
  s.flags = (volatile int *)(base + o);
  o += 16;
  s.scal = (float *)(base + o);
  return s;
}

// Thread 0 initialises the ring barriers; every thread of the block (producer warpgroup included) must call.
__device__ inline void init_ring(Smem &s, int nslot) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nslot; ++i) {
      mbar_init(&s.full[i], 1);      // the producer's arrive.expect_tx (+ the copy's bytes)
      mbar_init(&s.empty[i], NCW);   // one arrival per consumer warp
    }
    s.flags[0] = 0;
    s.flags[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();
}

// ---- bounded waits ---------------------------------------------------------------------------------------

// Everything a wait needs to give up cleanly: the launch-wide status word (any CTA may set it) and the
// wait limit.
struct Guard {
  int *status;
  unsigned long long timeout_ns;
};

__device__ inline void raise_status(const Guard &g, int code) { atomicCAS(g.status, ST_OK, code); }

// Wait for phase `parity` of an mbarrier. Gives up (returns false) when another CTA has raised the status
// word or when the wait exceeds the limit, in which case it raises ST_TIMEOUT itself.
__device__ inline bool wait_mbar(uint64_t *bar, uint32_t parity, const Guard &g) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (int spins = 1;; ++spins) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spins & 63) == 0) {
      if (ld_relaxed_gpu(g.status) != ST_OK) return false;
      if (globaltimer() - t0 > g.timeout_ns) {
        raise_status(g, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// ---- ring ------------------------------------------------------------------------------------------------

struct RingPos {
  int slot;
  uint32_t phase;
  long long issued;  // producer only: tiles issued so far
};

__device__ __forceinline__ void ring_advance(RingPos &r, int nslot) {
  if (++r.slot == nslot) {
    r.slot = 0;
    r.phase ^= 1u;
  }
}

// Producer: stream the tiles of rows [0, R) of one CTA region (R rows of K columns, packed) into the ring.
// Returns false if it had to give up (status raised).
// eb: bytes per element (2 for fp16, 1 for FP8), bw: column-block width of the packed layout.
__device__ inline bool produce_region(const uint8_t *region, int R, int K, Smem &s, int nslot, RingPos &rp,
                                      uint64_t policy, const Guard &g, int eb = 2, int bw = TILE_COLS) {
  const uint8_t *src = region;
  for (int g0 = 0; g0 < R; g0 += TILE_ROWS) {
    const int rows = min(TILE_ROWS, R - g0);
    for (int k0 = 0; k0 < K; k0 += bw) {
      const uint32_t bytes = (uint32_t)rows * (uint32_t)min(bw, K - k0) * (uint32_t)eb;
      if (!wait_mbar(&s.empty[rp.slot], rp.phase ^ 1u, g)) return false;
      mbar_arrive_expect_tx(&s.full[rp.slot], bytes);
      bulk_g2s(s.ring + (size_t)rp.slot * SLOT_BYTES, src, bytes, &s.full[rp.slot], policy);
      src += bytes;
      ++rp.issued;
      ring_advance(rp, nslot);
    }
  }
  return true;
}

// Producer: the same R rows of two FP8 regions (two experts) as ONE region of 2R rows (2R <= TILE_ROWS): for
// each column block, A's R-row tile then B's, back to back in one slot, i.e. the [2R][w] tile that
// consume_region_fp8 reads for a 2R-row region. B null: A alone (R rows).
__device__ inline bool produce_stacked_fp8(const uint8_t *A, const uint8_t *B, int R, int K, Smem &s, int nslot,
                                           RingPos &rp, uint64_t policy, const Guard &g) {
  for (int k0 = 0; k0 < K; k0 += FP8_TILE_COLS) {
    const uint32_t bytes = (uint32_t)R * (uint32_t)min(FP8_TILE_COLS, K - k0);
    if (!wait_mbar(&s.empty[rp.slot], rp.phase ^ 1u, g)) return false;
    uint8_t *dst = s.ring + (size_t)rp.slot * SLOT_BYTES;
    mbar_arrive_expect_tx(&s.full[rp.slot], B ? 2 * bytes : bytes);
    bulk_g2s(dst, A + (size_t)R * k0, bytes, &s.full[rp.slot], policy);
    if (B) bulk_g2s(dst + bytes, B + (size_t)R * k0, bytes, &s.full[rp.slot], policy);
    ++rp.issued;
    ring_advance(rp, nslot);
  }
  return true;
}

// Producer, before the CTA may exit: wait until every bulk copy it issued has landed (bounded), so no copy
// writes into the shared memory of a finished CTA.
__device__ inline void drain_ring(Smem &s, int nslot, const RingPos &rp, const Guard &g) {
  Guard local = g;
  for (int i = 0; i < nslot; ++i) {
    const long long uses = rp.issued > i ? (rp.issued - i + nslot - 1) / nslot : 0;
    if (uses == 0) continue;
    const uint32_t parity = (uint32_t)((uses - 1) & 1);
    // A landed copy completes its phase whether or not a consumer read it; the limit only guards a fault.
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&s.full[i], parity))
      if (globaltimer() - t0 > local.timeout_ns) {
        raise_status(local, ST_TIMEOUT);
        break;
      }
  }
}

// ---- consumer: one projection over the CTA's rows ------------------------------------------------------

__device__ __forceinline__ float dot8(const uint4 w, const float4 xa, const float4 xb) {
  const float2 w0 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
  const float2 w1 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
  const float2 w2 = __half22float2(*reinterpret_cast<const __half2 *>(&w.z));
  const float2 w3 = __half22float2(*reinterpret_cast<const __half2 *>(&w.w));
  float a = w0.x * xa.x;
  a = fmaf(w0.y, xa.y, a);
  a = fmaf(w1.x, xa.z, a);
  a = fmaf(w1.y, xa.w, a);
  float b = w2.x * xb.x;
  b = fmaf(w2.y, xb.y, b);
  b = fmaf(w3.x, xb.z, b);
  b = fmaf(w3.y, xb.w, b);
  return a + b;
}

// The column blocks [k_begin, k_end) (full 256-column blocks) of one row group, for a warp that owns NJ rows of
// the group (rows warp, warp + NCW, ...). Every warp waits for and releases every tile, whatever its NJ: the
// ring's empty barriers count NCW arrivals. The warp copies its rows to registers and hands the slot back
// before the math, so a slot is held only for the shared-memory reads. This loop is kept free of per-row
// guards and runtime strides: it is the hot loop of the whole decode.
template <int NJ>
__device__ __forceinline__ void tile_loop(const uint8_t *ring, uint64_t *full, uint64_t *empty, const float *vec,
                                          float (&acc)[ROWS_PER_WARP], int nslot, int &slot, uint32_t &phase,
                                          int k_begin, int k_end, bool &ok, volatile int *flags, const Guard &g) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k0 = k_begin; k0 < k_end; k0 += TILE_COLS) {
    if (ok && !wait_mbar(&full[slot], phase, g)) {
      ok = false;
      flags[0] = 1;
    }
    // no branch on `ok` here: after an abort the reads below still stay inside the slot and the results are
    // discarded, and a branch-free body is what lets the compiler overlap one tile's reads with the math
    uint4 wv[NJ > 0 ? NJ : 1];
    const uint8_t *t = ring + (size_t)slot * SLOT_BYTES + (size_t)warp * (TILE_COLS * 2) + lane * 16;
#pragma unroll
    for (int j = 0; j < NJ; ++j) wv[j] = *reinterpret_cast<const uint4 *>(t + (size_t)j * NCW * TILE_COLS * 2);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == nslot) {
      slot = 0;
      phase ^= 1u;
    }
    if (NJ > 0) {
      const float4 xa = *reinterpret_cast<const float4 *>(vec + k0 + lane * 8);
      const float4 xb = *reinterpret_cast<const float4 *>(vec + k0 + lane * 8 + 4);
#pragma unroll
      for (int j = 0; j < NJ; ++j) acc[j] += dot8(wv[j], xa, xb);
    }
  }
}

// out[i] = scale * sum_k W[r0 + i][k] * vec[k] for the R rows of this CTA, consuming the tiles the producer
// streams for this region (row group by row group, each group column block by column block). Warp w owns rows
// w, w + NCW, ... of each group and reduces them across lanes at the end of the group.
//
// A thread whose wait gives up raises the CTA abort flag and skips the remaining waits but walks the same tile
// sequence, so every consumer thread reaches the same named barriers; callers test the flag only after a
// consumer_sync.
static __device__ __noinline__ void consume_region(Smem &s, int nslot, RingPos &rp, int R, int K, float scale,
                                                   const Guard &g) {
  bool ok = s.flags[0] == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // register copies of the shared-memory layout (the struct itself may live in local memory here)
  const float *vec = s.vec;
  const uint8_t *const ring = s.ring;
  uint64_t *const full = s.full, *const empty = s.empty;
  float *const out = s.out;
  volatile int *const flags = s.flags;
  int slot = rp.slot;
  uint32_t phase = rp.phase;
  const int kfull = K / TILE_COLS * TILE_COLS;  // columns covered by full 256-column blocks
  for (int g0 = 0; g0 < R; g0 += TILE_ROWS) {
    const int rows = min(TILE_ROWS, R - g0);
    const int nj = min(ROWS_PER_WARP, (rows - warp + NCW - 1) / NCW);  // rows of this group owned by the warp
    float acc[ROWS_PER_WARP];
#pragma unroll
    for (int j = 0; j < ROWS_PER_WARP; ++j) acc[j] = 0.f;
    switch (nj) {
      case 4: tile_loop<4>(ring, full, empty, vec, acc, nslot, slot, phase, 0, kfull, ok, flags, g); break;
      case 3: tile_loop<3>(ring, full, empty, vec, acc, nslot, slot, phase, 0, kfull, ok, flags, g); break;
      case 2: tile_loop<2>(ring, full, empty, vec, acc, nslot, slot, phase, 0, kfull, ok, flags, g); break;
      case 1: tile_loop<1>(ring, full, empty, vec, acc, nslot, slot, phase, 0, kfull, ok, flags, g); break;
      default: tile_loop<0>(ring, full, empty, vec, acc, nslot, slot, phase, 0, kfull, ok, flags, g); break;
    }
    if (kfull < K) {  // a last, narrower column block (K not a multiple of 256): the guarded path
      const int k0 = kfull, w = K - kfull;
      if (ok && !wait_mbar(&full[slot], phase, g)) {
        ok = false;
        flags[0] = 1;
      }
      const bool active = ok && lane * 8 < w;
      uint4 wv[ROWS_PER_WARP];
      if (active) {
        const uint8_t *tile = ring + (size_t)slot * SLOT_BYTES;
#pragma unroll
        for (int j = 0; j < ROWS_PER_WARP; ++j)
          if (j < nj) wv[j] = *reinterpret_cast<const uint4 *>(tile + ((size_t)(warp + NCW * j) * w + lane * 8) * 2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == nslot) {
        slot = 0;
        phase ^= 1u;
      }
      if (active) {
        const float4 xa = *reinterpret_cast<const float4 *>(vec + k0 + lane * 8);
        const float4 xb = *reinterpret_cast<const float4 *>(vec + k0 + lane * 8 + 4);
#pragma unroll
        for (int j = 0; j < ROWS_PER_WARP; ++j)
          if (j < nj) acc[j] += dot8(wv[j], xa, xb);
      }
    }
#pragma unroll
    for (int j = 0; j < ROWS_PER_WARP; ++j) {
      if (j < nj) {
        const float v = warp_sum(acc[j]);
        if (lane == 0) out[g0 + warp + NCW * j] = v * scale;
      }
    }
  }
  rp.slot = slot;
  rp.phase = phase;
}

// ---- consumer: one FP8 (E4M3) projection -----------------------------------------------------------------

// Sixteen E4M3 codes (one 16-byte chunk of a tile row, column order = byte order) times x[0..16). Each code
// pair goes through the hardware E4M3x2 -> f16x2 conversion, which is exact (every E4M3 value is an fp16
// value), then fp32 FMAs.
__device__ __forceinline__ float dot16_e4m3(const uint4 w, const float4 x0, const float4 x1, const float4 x2,
                                            const float4 x3) {
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
  const float4 xs[4] = {x0, x1, x2, x3};
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wd[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wd[i] >> 16), __NV_E4M3);
    const float2 f0 = __half22float2(__half2(lo)), f1 = __half22float2(__half2(hi));
    a = fmaf(f0.x, xs[i].x, a);
    a = fmaf(f0.y, xs[i].y, a);
    b = fmaf(f1.x, xs[i].z, b);
    b = fmaf(f1.y, xs[i].w, b);
  }
  return a + b;
}

// Two E4M3 codes (the low and high byte of v) -> f16x2 (low half = low byte); exact, every E4M3 value is an
// fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// x (fp32, 16 values from an fp16 high part and an fp16 low part) for the scalar path of ragged blocks.
__device__ __forceinline__ void load_split16(const __half *xh, const __half *xl, float4 (&x)[4]) {
  const uint4 h0 = *reinterpret_cast<const uint4 *>(xh), h1 = *reinterpret_cast<const uint4 *>(xh + 8);
  const uint4 l0 = *reinterpret_cast<const uint4 *>(xl), l1 = *reinterpret_cast<const uint4 *>(xl + 8);
  const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  const uint32_t lw[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
  float f[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&hw[i]));
    const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&lw[i]));
    f[2 * i] = a.x + c.x;
    f[2 * i + 1] = a.y + c.y;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
}

// One full 512-code FP8 block of a row group on the tensor cores (mma.sync m16n8k16, fp32 accumulation).
// A = the weights (E4M3 -> fp16, exact); B = x as two columns, its fp16 high part (column 0) and the fp16
// rounding of the remainder (column 1); the other six columns are zero. The k order inside a 16-wide MMA step
// is permuted so that a lane's four A values of a row are four consecutive codes: in step j of 64-code group q,
// lane (g = lane / 4, t = lane % 4) holds codes 64q + 16t + 4j + {0, 1} (the fragment's k = 2t, 2t + 1) and
// + {2, 3} (k = 2t + 8, 2t + 9), and B is read in the same order. NMB row blocks of 16: with NMB = 2 warp w
// takes rows 16 (w % 2) + [0, 16) and groups w / 2, w / 2 + 4; with NMB = 1 every warp takes rows [0, 16) and
// group w. `wa`, `wb`: the lane's 16-byte chunks of rows g and g + 8 of its row block, per group.
template <int NMB>
__device__ __forceinline__ void fp8_block_mma(const uint4 (&wa)[NMB], const uint4 (&wb)[NMB], const __half *xh,
                                              const __half *xl, int k0, float (&acc)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, fg = lane >> 2, ft = lane & 3;
#pragma unroll
  for (int i = 0; i < NMB; ++i) {
    const int grp = NMB == 2 ? (warp >> 1) + 4 * i : warp;
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
    if (fg < 2) {
      const __half *xs = (fg == 0 ? xh : xl) + k0 + grp * 64 + ft * 16;
      x0 = *reinterpret_cast<const uint4 *>(xs);
      x1 = *reinterpret_cast<const uint4 *>(xs + 8);
    }
    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const uint32_t ww[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
    const uint32_t vw[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a[4] = {e4m3x2_to_f16x2(ww[j]), e4m3x2_to_f16x2(vw[j]), e4m3x2_to_f16x2(ww[j] >> 16),
                             e4m3x2_to_f16x2(vw[j] >> 16)};
      const uint32_t b[2] = {xw[2 * j], xw[2 * j + 1]};
      mma_f16_f32(acc, a, b);
    }
  }
}

// The full blocks of one row group (rows <= TILE_ROWS) for NMB row blocks of 16; every warp waits for and
// releases every tile (the ring's empty barriers count NCW arrivals), after copying its chunks to registers.
template <int NMB>
__device__ __forceinline__ void tile_loop_fp8_mma(const uint8_t *ring, uint64_t *full, uint64_t *empty,
                                                  const __half *xh, const __half *xl, float (&acc)[4], int nslot,
                                                  int &slot, uint32_t &phase, int k_end, bool &ok,
                                                  volatile int *flags, const Guard &g) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, fg = lane >> 2, ft = lane & 3;
  const int ra = (NMB == 2 ? 16 * (warp & 1) : 0) + fg;  // rows ra and ra + 8 (same parity)
  const uint32_t swz = (uint32_t)(ra & 1) << 6;          // chunk q of an odd row is stored at q ^ 4
  for (int k0 = 0; k0 < k_end; k0 += FP8_TILE_COLS) {
    if (ok && !wait_mbar(&full[slot], phase, g)) {
      ok = false;
      flags[0] = 1;
    }
    const uint8_t *tile = ring + (size_t)slot * SLOT_BYTES;
    uint4 wa[NMB], wb[NMB];
#pragma unroll
    for (int i = 0; i < NMB; ++i) {
      const int grp = NMB == 2 ? (warp >> 1) + 4 * i : warp;
      const uint32_t cb = ((uint32_t)(grp * 64 + ft * 16)) ^ swz;
      wa[i] = *reinterpret_cast<const uint4 *>(tile + (size_t)ra * FP8_TILE_COLS + cb);
      wb[i] = *reinterpret_cast<const uint4 *>(tile + (size_t)(ra + 8) * FP8_TILE_COLS + cb);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == nslot) {
      slot = 0;
      phase ^= 1u;
    }
    fp8_block_mma<NMB>(wa, wb, xh, xl, k0, acc);
  }
}

// Row r (< rows) of an FP8 row group from the partial sums its warps left in `red`, in a fixed order: the
// tensor-core warps that own the row (all of them for <= 16 rows, every other one otherwise), then the ragged
// block's sum.
__device__ __forceinline__ float fp8_group_sum(const float *red, int r, int rows, bool ragged) {
  const int nmb = rows > 16 ? 2 : 1;
  float v = 0.f;
  for (int w = 0; w < NCW; ++w)
    if (nmb == 1 || (w & 1) == (r >> 4)) v += red[w * TILE_ROWS + r];
  if (ragged) v += red[NCW * TILE_ROWS + r];
  return v;
}

// out[i] = scale * sum_k Q[r0 + i][k] * x[k] over the R rows of this CTA in one packed FP8 region (codes taken at
// their E4M3 value; the caller applies the row scales). x is given as its fp16 high part xh and low part xl
// (K values each). Full 512-code blocks run on the tensor cores (fp8_block_mma); a ragged last block takes the
// CUDA-core path with x = xh + xl, one 16-code chunk per lane and row, rows warp, warp + NCW, ... Per row group
// the partial sums meet in `red` (9 x TILE_ROWS floats) and are added in a fixed order (fp8_group_sum). With
// `defer` (R <= TILE_ROWS only) the region stops there: no consumer_sync, `out` untouched, the partial sums left
// in `red` for the caller, who syncs once after several regions (each with its own `red`) and adds them itself.
// A thread whose wait gives up raises the CTA abort flag and walks the same tile sequence, like consume_region.
static __device__ __noinline__ void consume_region_fp8(Smem &s, int nslot, RingPos &rp, int R, int K,
                                                       const __half *xh, const __half *xl, float scale,
                                                       float *out, float *red, const Guard &g,
                                                       bool defer = false) {
  bool ok = s.flags[0] == 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, fg = lane >> 2, ft = lane & 3;
  const uint8_t *const ring = s.ring;
  uint64_t *const full = s.full, *const empty = s.empty;
  volatile int *const flags = s.flags;
  int slot = rp.slot;
  uint32_t phase = rp.phase;
  const int kfull = K / FP8_TILE_COLS * FP8_TILE_COLS;
  for (int g0 = 0; g0 < R; g0 += TILE_ROWS) {
    const int rows = min(TILE_ROWS, R - g0);
    const int nmb = rows > 16 ? 2 : 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (nmb == 2)
      tile_loop_fp8_mma<2>(ring, full, empty, xh, xl, acc, nslot, slot, phase, kfull, ok, flags, g);
    else
      tile_loop_fp8_mma<1>(ring, full, empty, xh, xl, acc, nslot, slot, phase, kfull, ok, flags, g);
    // column 0 of D is W x_hi, column 1 W x_lo: lane t = 0 of each quad holds both for rows g and g + 8
    if (ft == 0) {
      const int r = (nmb == 2 ? 16 * (warp & 1) : 0) + fg;
      red[warp * TILE_ROWS + r] = acc[0] + acc[1];
      red[warp * TILE_ROWS + r + 8] = acc[2] + acc[3];
    }
    const bool ragged = kfull < K;
    if (ragged) {  // the last, narrower column block (w codes per row, a multiple of 16): CUDA cores
      const int w = K - kfull;
      const int nj = min(ROWS_PER_WARP, (rows - warp + NCW - 1) / NCW);
      if (ok && !wait_mbar(&full[slot], phase, g)) {
        ok = false;
        flags[0] = 1;
      }
      const bool active = ok && lane * 16 < w;
      uint4 wv[ROWS_PER_WARP];
      if (active) {
        const uint8_t *tile = ring + (size_t)slot * SLOT_BYTES;
#pragma unroll
        for (int j = 0; j < ROWS_PER_WARP; ++j)
          if (j < nj) wv[j] = *reinterpret_cast<const uint4 *>(tile + (size_t)(warp + NCW * j) * w + lane * 16);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == nslot) {
        slot = 0;
        phase ^= 1u;
      }
      float tacc[ROWS_PER_WARP] = {0.f, 0.f, 0.f, 0.f};
      if (active) {
        float4 x[4];
        load_split16(xh + kfull + lane * 16, xl + kfull + lane * 16, x);
#pragma unroll
        for (int j = 0; j < ROWS_PER_WARP; ++j)
          if (j < nj) tacc[j] = dot16_e4m3(wv[j], x[0], x[1], x[2], x[3]);
      }
#pragma unroll
      for (int j = 0; j < ROWS_PER_WARP; ++j) {
        if (j < nj) {
          const float v = warp_sum(tacc[j]);
          if (lane == 0) red[NCW * TILE_ROWS + warp + NCW * j] = v;
        }
      }
    }
    if (defer) break;  // R <= TILE_ROWS: this was the only row group
    consumer_sync();
    for (int r = tid; r < rows; r += NCT) out[g0 + r] = fp8_group_sum(red, r, rows, ragged) * scale;
    consumer_sync();  // red is reused by the next row group
  }
  rp.slot = slot;
  rp.phase = phase;
}

// 4-byte asynchronous global -> shared copy (completion: cp_async_wait_all by the issuing thread).
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- staging the input vector ---------------------------------------------------------------------------

// vec[0..K) = src (fp32, written by other CTAs earlier in the launch: read through L2). If want_ss, returns
// the CTA-uniform sum of squares (ends with a consumer_sync either way).
__device__ inline float stage_f32(Smem &s, const float *src, int K, bool want_ss) {
  const int tid = threadIdx.x;
  float ss = 0.f;
  for (int i = tid * 4; i < K; i += NCT * 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + i));
    *reinterpret_cast<float4 *>(s.vec + i) = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (!want_ss) {
    consumer_sync();
    return 0.f;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) s.red[tid >> 5] = ss;
  consumer_sync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) t += s.red[w];
  consumer_sync();  // s.red may be reused right after
  return t;
}

// Four fp32 values as their fp16 high parts hi = fp16(v) (to hi[0..4)) and the fp16 roundings of the
// remainders v - hi (to lo[0..4)): the two-column B operand of the tensor-core FP8 GEMV.
__device__ __forceinline__ void split4(const float4 v, __half *hi, __half *lo) {
  const __half2 h0 = __floats2half2_rn(v.x, v.y), h1 = __floats2half2_rn(v.z, v.w);
  const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
  const __half2 l0 = __floats2half2_rn(v.x - f0.x, v.y - f0.y), l1 = __floats2half2_rn(v.z - f1.x, v.w - f1.y);
  uint2 hw, lw;
  hw.x = *reinterpret_cast<const uint32_t *>(&h0);
  hw.y = *reinterpret_cast<const uint32_t *>(&h1);
  lw.x = *reinterpret_cast<const uint32_t *>(&l0);
  lw.y = *reinterpret_cast<const uint32_t *>(&l1);
  *reinterpret_cast<uint2 *>(hi) = hw;
  *reinterpret_cast<uint2 *>(lo) = lw;
}

// vec[0..K) = src * gain (src fp32 written by other CTAs, read through L2; gain read-only) and the CTA-uniform
// sum of squares of src (the RMSNorm of src with its gain applied to the staged copy). K a multiple of 4.
// With `split` the staged values are also written as fp16 high parts split[0..K) and low parts split[K..2K).
__device__ inline float stage_f32_gain(Smem &s, const float *src, const float *gain, int K, __half *split) {
  const int tid = threadIdx.x;
  float ss = 0.f;
  for (int i = tid * 4; i < K; i += NCT * 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + i));
    const float4 w = __ldg(reinterpret_cast<const float4 *>(gain + i));
    const float4 u = make_float4(v.x * w.x, v.y * w.y, v.z * w.z, v.w * w.w);
    *reinterpret_cast<float4 *>(s.vec + i) = u;
    if (split) split4(u, split + i, split + K + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) s.red[tid >> 5] = ss;
  consumer_sync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) t += s.red[w];
  consumer_sync();
  return t;
}

// split[0..K) = fp16 high parts and split[K..2K) = fp16 low parts of src (fp32 written by other CTAs, read
// through L2); nothing else is staged. K a multiple of 4.
__device__ inline void stage_split(const float *src, int K, __half *split) {
  for (int i = threadIdx.x * 4; i < K; i += NCT * 4)
    split4(__ldcg(reinterpret_cast<const float4 *>(src + i)), split + i, split + K + i);
  consumer_sync();
}

// vec[0..K) = fp32(src) for an fp16 vector that is read-only during the launch.
__device__ inline float stage_f16(Smem &s, const __half *src, int K, bool want_ss) {
  const int tid = threadIdx.x;
  float ss = 0.f;
  for (int i = tid * 8; i < K; i += NCT * 8) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src + i));
    const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h[e]);
      s.vec[i + 2 * e] = f.x;
      s.vec[i + 2 * e + 1] = f.y;
      ss += f.x * f.x + f.y * f.y;
    }
  }
  if (!want_ss) {
    consumer_sync();
    return 0.f;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) s.red[tid >> 5] = ss;
  consumer_sync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) t += s.red[w];
  consumer_sync();
  return t;
}

}  // namespace kie
