// The persistent decode monokernel for sm_103a.
//
// One cooperative launch of n_cta CTAs (one per SM) runs n whole decode steps, as the monokernel pages
// describe it ("inside the monokernel": one resident grid runs the token loop, sampling included, and never
// hands control back to the host between tokens). Per token:
//
//   embed -> for each layer:
//     [QKV]   q,k,v = inv_rms(x) * (W'qkv x); RoPE from the table; K,V appended (fp16) ........ barrier
//     [ATT]   split-KV attention over the cached positions; the pieces of a KV head merge it ...... barrier
//     [WO]    h = x + Wo o ........................................................................ barrier
//     [GU]    a = silu(gate) * up,  [gate; up] = inv_rms(h) * (W'gu h), rows interleaved ........ barrier
//     [DOWN]  x = h + Wd a ........................................................................ barrier
//   [LM] logits = inv_rms(x) * (W'lm x); per-CTA argmax folded with one 64-bit atomicMax ........... barrier
//
// W' are the repacked weights with the RMSNorm gain folded into their columns (the "RMSNorm folding" and
// "offline QKV repacking" items of the pages), so a norm is just one scalar computed redundantly by every
// CTA from the full vector. Weights stream through each CTA's shared-memory ring (kie_device.cuh) without
// ever waiting for a barrier; consumers wait at the grid barrier, which is one global counter polled with
// acquire loads and bounded by a %globaltimer limit.
#include <cuda_runtime.h>

#include "kie_decode.cuh"
#include "kie_device.cuh"

namespace kie {

// ---- grid barrier -----------------------------------------------------------------------------------------

// All consumer threads of every CTA call this together. Returns false (uniformly within the CTA) when the
// launch is being abandoned: a wait ran out here or anywhere else.
__device__ inline bool grid_barrier(const DecodeParams &p, Smem &s, uint32_t &gen, const Guard &g,
                                    unsigned long long &wait_ns) {
  consumer_sync();
  const uint32_t idx = gen++;
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    bool ok = s.flags[0] == 0;
    if (ok) {
      // Release add, acquire polls, then the CTA barrier: together they order every write made before any
      // CTA's arrival before every read made after this CTA leaves. Data other CTAs wrote is always read
      // through L2 (ld.global.cg), so no stale L1 line can be hit.
      if (!((int)blockIdx.x == p.skip_cta && (int)idx == p.skip_barrier)) red_release_gpu_add(&p.ctl->bar_count, 1u);
      const unsigned target = (idx + 1u) * (unsigned)p.n_cta;
      for (int spins = 1;; ++spins) {
        const unsigned cur = ld_acquire_gpu(&p.ctl->bar_count);
        if ((int)(cur - target) >= 0) break;
        if ((spins & 15) == 0) {
          if (ld_relaxed_gpu(&p.ctl->status) != ST_OK) {
            ok = false;
            break;
          }
          if (globaltimer() - t0 > p.timeout_ns) {
            raise_status(g, ST_TIMEOUT);
            atomicCAS(&p.ctl->where, 0, (int)idx + 1);
            ok = false;
            break;
          }
        }
      }
    }
    const uint64_t dt = globaltimer() - t0;
    wait_ns += dt;
    if (idx < (uint32_t)TRACE_CAP) {
      p.trace[(size_t)idx * p.n_cta + blockIdx.x] = (uint32_t)min(dt, (uint64_t)0xFFFFFFFFu);
      p.trace_arrive[(size_t)idx * p.n_cta + blockIdx.x] = t0;
    }
    if (!ok) s.flags[0] = 1;
  }
  consumer_sync();
  return s.flags[0] == 0;
}

// ---- epilogues ------------------------------------------------------------------------------------------

// Fused QKV rows of this CTA, [r0, r1): rows come in pairs. Query and key pairs hold the two halves
// (i, i + dh/2) of one RoPE rotation, rotated here with the table row of `pos`; keys and values go to the
// cache as fp16, queries to p.q (fp32, same pair-adjacent order as the cached keys).
__device__ inline void epilogue_qkv(const DecodeParams &p, const Smem &s, int l, int pos, int r0, int r1) {
  const int dh = p.dh, qrows = p.Hq * dh, krows = p.Hkv * dh;
  const size_t plane = (size_t)p.max_seq * dh;
  __half *Kl = p.kv + (size_t)l * 2 * p.Hkv * plane;
  __half *Vl = Kl + (size_t)p.Hkv * plane;
  const float2 *tab = reinterpret_cast<const float2 *>(s.out + p.out_rope);  // RoPE row of pos, staged per token
  for (int pr = threadIdx.x; pr < (r1 - r0) / 2; pr += NCT) {
    const int r = r0 + 2 * pr;
    float a = s.out[2 * pr], b = s.out[2 * pr + 1];
    if (r < qrows + krows) {
      const int rr = r < qrows ? r : r - qrows;
      const float2 cs = tab[(rr % dh) / 2];
      const float a2 = a * cs.x - b * cs.y, b2 = b * cs.x + a * cs.y;
      if (r < qrows) {
        *reinterpret_cast<float2 *>(p.q + r) = make_float2(a2, b2);
      } else {
        __half2 kv2 = __floats2half2_rn(a2, b2);
        *reinterpret_cast<__half2 *>(Kl + (size_t)(rr / dh) * plane + (size_t)pos * dh + rr % dh) = kv2;
      }
    } else {
      const int rr = r - qrows - krows;
      *reinterpret_cast<__half2 *>(Vl + (size_t)(rr / dh) * plane + (size_t)pos * dh + rr % dh) =
          __floats2half2_rn(a, b);
    }
  }
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  const unsigned u = __float_as_uint(v);
  const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

__device__ __forceinline__ int key_index(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
}

// The float a key was made from (argmax_key's order-preserving map inverted, bit for bit).
__device__ __forceinline__ float key_value(unsigned long long key) {
  const unsigned ord = (unsigned)(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

// ---- split-KV attention -----------------------------------------------------------------------------------

// Piece `sp` of KV head `kh`: positions [j0, j1) of the c cached ones. Emits the unnormalised partial (m, l, o)
// of each of the `group` query heads; once all S pieces of the head are in, each piece merges a 1/S slice of
// the head's outputs (log-sum-exp rescaling) into p.o. This is the pages' "attention recompute" idea in GB300 form: each SM recomputes exactly
// its slice from the cache instead of exchanging intermediate attention state.
//
// Latency matters more than bandwidth here (a piece reads <= 16 KB of K/V per sub-chunk), so every sub-chunk's
// K and V rows are requested together with q in one round trip, the next sub-chunk is prefetched into registers
// while the current one is used from shared memory, and no step waits on a dependent global load.
//
// Both products of a sub-chunk run on the tensor cores (mma.sync m16n8k16, fp32 accumulation): the scores as
// Q K^T with the group's query heads as the rows of A, then O += P V. K and V are fp16 already, so they are
// exact operands; q and the softmax weights p are fp32, and each is split into an fp16 high part and the fp16
// rounding of the remainder, which fill rows h and 8 + h of A. The two rows' products are summed in fp32, so
// the result carries about 22 significant bits of q and p instead of fp16's 11.
template <int DPL>
__device__ inline void attention_piece(const DecodeParams &p, Smem &s, int l, int kh, int sp, int S, int j0,
                                       int j1, unsigned target, const Guard &g) {
  constexpr int DH = DPL * 32;
  constexpr int U = DH / 8;                          // 16-byte units per K or V row
  constexpr int UPT = (ATT_SUB * U + NCT - 1) / NCT;  // units per thread per sub-chunk
  constexpr int RS = DH + 8;                         // row stride (halfs) of q, K and V: 16-byte rows that
                                                     // ldmatrix reads from eight different bank groups
  constexpr int PS = ATT_SUB + 8;                    // row stride (halfs) of P
  constexpr int NTILE = DH / 8;                      // 8-column tiles of the output
  constexpr int TPW = (NTILE + NCW - 1) / NCW;       // output tiles per consumer warp
  static_assert(ATT_SUB == 32, "four 8-position score tiles, two 16-position P V steps per sub-chunk");
  static_assert(MAX_GROUP <= 8, "a group's high parts fill rows 0..7 of A, the low parts rows 8..15");
  static_assert(MAX_GROUP <= NCW, "one consumer warp per query head in the softmax");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int fg = lane >> 2, ft = lane & 3;           // fragment row group and column pair of this lane
  const int G = p.Hq / p.Hkv;
  __half *qA = reinterpret_cast<__half *>(s.vec);    // [16][RS] q / sqrt(dh): high parts, low parts
  __half *Ks = qA + 16 * RS;                         // [ATT_SUB][RS]
  __half *Vs = Ks + ATT_SUB * RS;                    // [ATT_SUB][RS]
  float *ps = reinterpret_cast<float *>(Vs + ATT_SUB * RS);  // [MAX_GROUP][ATT_SUB] softmax scratch:
  float *pmax = ps, *psum = ps + 4 * 8, *mnew = ps + 8 * 8;  // [4 warps][8 heads] partial maxima and sums
  __half *PA = reinterpret_cast<__half *>(ps + MAX_GROUP * ATT_SUB);  // [16][PS] p: high parts, low parts
  float *corr = reinterpret_cast<float *>(PA + 16 * PS);  // [MAX_GROUP]
  float *mrun = corr + MAX_GROUP;
  float *lrun = mrun + MAX_GROUP;
  float *mw = lrun + MAX_GROUP;                        // merge: [smax][G] m, then weights
  float *ml = mw + p.smax * G;                         // merge: [smax][G] l
  const float scale = 1.4426950408889634f / sqrtf((float)DH);  // log2(e) / sqrt(dh): scores in log2 units
  const size_t plane = (size_t)p.max_seq * DH;
  const __half *Kb = p.kv + ((size_t)l * 2 * p.Hkv + kh) * plane;
  const __half *Vb = p.kv + ((size_t)l * 2 * p.Hkv + p.Hkv + kh) * plane;

  uint4 kreg[UPT], vreg[UPT];
  auto fetch = [&](int jb) {  // registers <- K, V rows [jb, jb + ATT_SUB) that exist
    const int nb = min(ATT_SUB, j1 - jb);
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const int u = tid + k * NCT;
      if (u < nb * U) {
        const size_t off = (size_t)(jb + u / U) * DH + (u % U) * 8;
        kreg[k] = __ldcg(reinterpret_cast<const uint4 *>(Kb + off));
        vreg[k] = __ldcg(reinterpret_cast<const uint4 *>(Vb + off));
      }
    }
  };
  // shared memory <- the registers fetched for jb; rows past the end are zero, so that both products below
  // always run over ATT_SUB positions (a zero V row times a zero weight adds nothing)
  auto stash = [&](int jb) {
    const int nb = min(ATT_SUB, j1 - jb);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const int u = tid + k * NCT;
      if (u < ATT_SUB * U) {
        const bool in = u < nb * U;
        const size_t at = (size_t)(u / U) * RS + (u % U) * 8;
        *reinterpret_cast<uint4 *>(Ks + at) = in ? kreg[k] : zero;
        *reinterpret_cast<uint4 *>(Vs + at) = in ? vreg[k] : zero;
      }
    }
  };

  if (j0 < j1) fetch(j0);
  // A of the scores: row h = fp16(q_h), row 8 + h = fp16(q_h - row h); rows of heads past the group are zero
  for (int i = tid; i < 16 * DH; i += NCT) {
    const int r = i / DH, d = i % DH, h = r & 7;
    float v = 0.f;
    if (h < G) {
      const float qv = __ldcg(p.q + ((size_t)kh * G + h) * DH + d) * scale;
      const float hi = __half2float(__float2half_rn(qv));
      v = r < 8 ? hi : qv - hi;
    }
    qA[r * RS + d] = __float2half_rn(v);
  }
  for (int i = tid; i < 16 * PS; i += NCT) PA[i] = __float2half_rn(0.f);
  if (tid < MAX_GROUP) {
    mrun[tid] = -INFINITY;
    lrun[tid] = 0.f;
  }
  // output accumulators: warp w owns column tiles w, w + NCW, ...; rows fg (high) and fg + 8 (low) of each
  // belong to query head fg and are summed when the piece is published
  float acc[TPW][4];
#pragma unroll
  for (int i = 0; i < TPW; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  // ldmatrix row addresses: lane l points at row (l % 8) + 8 * ((l / 8) % 2), column half l / 16 of A
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);

  for (int jb = j0; jb < j1; jb += ATT_SUB) {
    const int nb = min(ATT_SUB, j1 - jb);
    stash(jb);
    consumer_sync();                               // Ks, Vs (and qA, PA) ready; ps free
    if (jb + ATT_SUB < j1) fetch(jb + ATT_SUB);    // next sub-chunk in flight while this one is used
    // scores S = Q K^T in log2 units: warp w < 4 takes positions [8w, 8w + 8) of the sub-chunk (two accumulator
    // chains over the DH / 16 steps of 16). Lane (g, t) holds head g's scores at positions 8w + 2t, 8w + 2t + 1
    // (rows g and 8 + g of D, the q high and low parts, summed); positions past nb weigh 0. The warp's maximum
    // per head comes from the lane's quad (two shuffles), and the four warps' maxima meet in shared memory.
    float s0 = -INFINITY, s1 = -INFINITY;
    if (warp < ATT_SUB / 8) {
      const int n0 = warp * 8, p0 = n0 + 2 * ft;
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        uint32_t a[4], b[2];
        ldsm_x4(a, qA + arow * RS + ks * 16 + acol);
        ldsm_x2(b, Ks + (n0 + (lane & 7)) * RS + ks * 16 + 8 * ((lane >> 3) & 1));
        mma_f16_f32(c[ks & 1], a, b);
      }
      if (p0 < nb) s0 = (c[0][0] + c[0][2]) + (c[1][0] + c[1][2]);
      if (p0 + 1 < nb) s1 = (c[0][1] + c[0][3]) + (c[1][1] + c[1][3]);
      float m8 = fmaxf(s0, s1);
      m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 1));
      m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 2));
      if (ft == 0) pmax[warp * 8 + fg] = m8;
    }
    consumer_sync();
    // online softmax, in the same lanes: m_new = max(m_run, the four warps' maxima), p = 2^(s - m_new) into rows
    // h (fp16 high part) and 8 + h (fp16 remainder) of the P operand, the warp's partial sums per head; warp 0
    // also leaves m_new and the rescale factor 2^(m_run - m_new) for the P V step. Lanes of heads past the group
    // compute on zero rows and store nothing.
    if (warp < ATT_SUB / 8) {
      const int p0 = warp * 8 + 2 * ft;
      const float mo = mrun[fg];
      const float mn = fmaxf(fmaxf(mo, fmaxf(pmax[fg], pmax[8 + fg])), fmaxf(pmax[16 + fg], pmax[24 + fg]));
      const float e0 = exp2f(s0 - mn), e1 = exp2f(s1 - mn);
      float sm = e0 + e1;
      sm += __shfl_xor_sync(0xffffffffu, sm, 1);
      sm += __shfl_xor_sync(0xffffffffu, sm, 2);
      if (fg < G) {
        const __half2 hi = __floats2half2_rn(e0, e1);
        const float2 hf = __half22float2(hi);
        *reinterpret_cast<__half2 *>(PA + fg * PS + p0) = hi;
        *reinterpret_cast<__half2 *>(PA + (8 + fg) * PS + p0) = __floats2half2_rn(e0 - hf.x, e1 - hf.y);
        if (ft == 0) {
          psum[warp * 8 + fg] = sm;
          if (warp == 0) {
            mnew[fg] = mn;
            corr[fg] = exp2f(mo - mn);
          }
        }
      }
    }
    consumer_sync();
    // o = o * corr + P V: two steps of 16 positions per column tile
    {
      const float cg = fg < G ? corr[fg] : 0.f;
      uint32_t a0[4], a1[4];
      ldsm_x4(a0, PA + arow * PS + acol);
      ldsm_x4(a1, PA + arow * PS + 16 + acol);
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        const int nt = warp + i * NCW;
        if (nt < NTILE) {
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][e] *= cg;
          uint32_t b0[2], b1[2];
          ldsm_x2_trans(b0, Vs + (lane & 15) * RS + nt * 8);
          ldsm_x2_trans(b1, Vs + (16 + (lane & 15)) * RS + nt * 8);
          mma_f16_f32(acc[i], a0, b0);
          mma_f16_f32(acc[i], a1, b1);
        }
      }
    }
    if (tid < G) {  // the running sum and maximum of head tid (every reader of the old values is past)
      lrun[tid] = lrun[tid] * corr[tid] + ((psum[tid] + psum[8 + tid]) + (psum[16 + tid] + psum[24 + tid]));
      mrun[tid] = mnew[tid];
    }
    consumer_sync();                               // Ks, Vs, PA and the softmax scratch reused next
  }

  // publish (m, l, o) of this piece
  const int E = G * DH;  // outputs of this KV head's query group
  const size_t piece = (size_t)kh * p.smax + sp;
  if (fg < G) {
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      const int nt = warp + i * NCW;
      if (nt < NTILE)
        *reinterpret_cast<float2 *>(p.part_o + piece * E + (size_t)fg * DH + nt * 8 + 2 * ft) =
            make_float2(acc[i][0] + acc[i][2], acc[i][1] + acc[i][3]);
    }
  }
  if (tid < G) *reinterpret_cast<float2 *>(p.part_ml + (piece * G + tid) * 2) = make_float2(mrun[tid], lrun[tid]);
  consumer_sync();
  // count this piece in (no reply needed), then wait for the other pieces of head kh: the counter only grows
  // during a launch, and `target` is the running total of pieces up to this layer's attention step
  if (tid == 0) {
    red_release_gpu_add(&p.ctl->att_cnt[kh], 1u);
    const uint64_t t0 = globaltimer();
    bool ok = true;
    for (int spins = 1;; ++spins) {
      if ((int)(ld_acquire_gpu(&p.ctl->att_cnt[kh]) - target) >= 0) break;
      if ((spins & 15) == 0) {
        if (ld_relaxed_gpu(&p.ctl->status) != ST_OK) {
          ok = false;
          break;
        }
        if (globaltimer() - t0 > p.timeout_ns) {
          raise_status(g, ST_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    if (!ok) s.flags[0] = 1;
  }
  consumer_sync();
  if (s.flags[0]) return;

  // Merge, split across the S pieces of the head: this CTA produces outputs [e0, e1) of the E,
  //   o_e = sum_q w_q o_q,e   with   w_q = 2^(m_q - M) / sum_r 2^(m_r - M) l_r,   M = max_r m_r
  // (the maxima m are in log2 units, like the scores)
  // for the query head of e. Every value it needs (all (m, l) of the head, and its slice of every piece's o)
  // is requested before any is used: one round trip.
  const int sl = (E + S - 1) / S;
  const int e0 = min(E, sp * sl), e1 = min(E, e0 + sl), w = e1 - e0;
  if (w == 0) return;
  float *mo = reinterpret_cast<float *>(Ks);  // [S][w] in the K half of the staging area (free now)
  constexpr int LPT = (MAX_GROUP * DH + NCT - 1) / NCT + 1;  // o loads per thread per round
  for (int r = 0; r * LPT * NCT < S * w || r * NCT < S * G; ++r) {  // one round unless S * G > NCT
    const int base = r * LPT * NCT;
    float rv[LPT];
    float2 rml;
#pragma unroll
    for (int k = 0; k < LPT; ++k) {
      const int i = base + tid + k * NCT;
      if (i < S * w) rv[k] = __ldcg(p.part_o + ((size_t)kh * p.smax + i / w) * E + e0 + i % w);
    }
    const int im = r * NCT + tid;  // (m, l) pairs: one per thread and round
    if (im < S * G) rml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml) + (size_t)kh * p.smax * G + im);
#pragma unroll
    for (int k = 0; k < LPT; ++k) {
      const int i = base + tid + k * NCT;
      if (i < S * w) mo[i] = rv[k];
    }
    if (im < S * G) {
      mw[im] = rml.x;
      ml[im] = rml.y;
    }
  }
  consumer_sync();
  if (S <= 16) {  // few pieces: each output's thread takes its head's maximum and normaliser itself (no
                  // cross-lane reduction, no further barrier), then sums the pieces in order
    for (int i = tid; i < w; i += NCT) {
      const int h = (e0 + i) / DH;
      float mx = -INFINITY;
      for (int q = 0; q < S; ++q) mx = fmaxf(mx, mw[q * G + h]);
      float den = 0.f, a = 0.f;
      for (int q = 0; q < S; ++q) {
        const float wq = exp2f(mw[q * G + h] - mx);
        den = fmaf(wq, ml[q * G + h], den);
        a = fmaf(wq, mo[q * w + i], a);
      }
      p.o[(size_t)kh * E + e0 + i] = a / den;
    }
    return;
  }
  if (warp < G) {  // warp h: the weights of query head h, lane per piece
    const int h = warp;
    float mx = -INFINITY;
    for (int q = lane; q < S; q += 32) mx = fmaxf(mx, mw[q * G + h]);
    mx = warp_max(mx);
    float den = 0.f;
    for (int q = lane; q < S; q += 32) den = fmaf(exp2f(mw[q * G + h] - mx), ml[q * G + h], den);
    den = warp_sum(den);
    const float inv = 1.0f / den;
    for (int q = lane; q < S; q += 32) mw[q * G + h] = exp2f(mw[q * G + h] - mx) * inv;
  }
  consumer_sync();
  // many pieces: P threads per output, each over every P-th piece, then a sum over the P partials
  float *red = reinterpret_cast<float *>(Vs);  // [P][w]; mo ends before the V half of the staging area
  const int P = max(1, NCT / w);
  for (int idx = tid; idx < P * w; idx += NCT) {
    const int i = idx % w, part = idx / w, h = (e0 + i) / DH;
    float a = 0.f;
    for (int q = part; q < S; q += P) a = fmaf(mw[q * G + h], mo[q * w + i], a);
    red[idx] = a;
  }
  consumer_sync();
  for (int i = tid; i < w; i += NCT) {
    float a = 0.f;
    for (int part = 0; part < P; ++part) a += red[part * w + i];
    p.o[(size_t)kh * E + e0 + i] = a;
  }
}

// ---- the kernel -------------------------------------------------------------------------------------------

// Pieces per KV head for c attended positions: one sub-chunk (ATT_SUB positions) per piece while there are
// enough CTAs, at most smax so that every piece has its own CTA (longer contexts then give each piece several
// sub-chunks). Fewer, longer pieces measured slower: the sub-chunks of a piece run one after the other.
__device__ __forceinline__ int split_pieces(const DecodeParams &p, int c) {
  const int s = (c + ATT_SUB - 1) / ATT_SUB;
  return s < p.smax ? s : p.smax;
}

// ---- sparse-MoE FFN steps ---------------------------------------------------------------------------------
//
// Shared-memory selection area (s.out + p.out_moe): an mbarrier that completes once per (token, layer) when the
// consumers publish the routed experts, then top_k expert ids and top_k routing weights.
struct MoeSel {
  uint64_t *bar;
  int *ids;
  float *wts;
};

__device__ __forceinline__ MoeSel moe_sel(const DecodeParams &p, const Smem &s) {
  float *b = s.out + p.out_moe;
  return {reinterpret_cast<uint64_t *>(b), reinterpret_cast<int *>(b + 2), b + 2 + MAX_TOP_K};
}

// The router by linearity. Its logits are inv_rms(h) * (R (g o h)) with h = x + Wo o, so with rg = R diag(g)
// and rgwo = rg Wo (folded at creation) they are inv_rms(h) * (rg x + rgwo o): rg x is taken in the QKV phase
// (x is staged there), rgwo o in the WO phase (o is staged there), and the logits need no phase and no grid
// barrier of their own. This CTA's rows e = CTA, CTA + n_cta, ... of the K-column fp32 matrix M times the staged
// vector, into out[e]: the first row is requested into registers when the phase starts (RouterRow), so its L2
// round trip overlaps the phase's GEMV (staging it in shared memory with cp.async instead measured slower); any
// further rows (more experts than CTAs) are read afterwards. A CTA-wide dot product per row, summed in a fixed
// order.
constexpr int ROUTER_V4 = 4;  // float4 per thread held for the first row: rows of up to 4 * 4 * NCT columns

struct RouterRow {
  float4 v[ROUTER_V4];
};

__device__ __forceinline__ RouterRow moe_router_fetch(const DecodeParams &p, const float *M, int K) {
  RouterRow r;
  const int e = blockIdx.x;
#pragma unroll
  for (int i = 0; i < ROUTER_V4; ++i) {
    const int k = (threadIdx.x + i * NCT) * 4;
    r.v[i] = (e < p.E && k < K) ? __ldg(reinterpret_cast<const float4 *>(M + (size_t)e * K + k))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  return r;
}

__device__ inline void moe_router_part(const DecodeParams &p, Smem &s, const RouterRow &first, const float *M, int K,
                                       float *out) {
  const int tid = threadIdx.x;
  for (int e = blockIdx.x; e < p.E; e += p.n_cta) {
    float a0 = 0.f, a1 = 0.f;
    if (e == (int)blockIdx.x && K <= ROUTER_V4 * NCT * 4) {
#pragma unroll
      for (int i = 0; i < ROUTER_V4; ++i) {
        const int k = (tid + i * NCT) * 4;
        if (k < K) {
          const float4 w = first.v[i], v = *reinterpret_cast<const float4 *>(s.vec + k);
          a0 = fmaf(w.x, v.x, a0);
          a1 = fmaf(w.y, v.y, a1);
          a0 = fmaf(w.z, v.z, a0);
          a1 = fmaf(w.w, v.w, a1);
        }
      }
    } else {
      for (int k = tid * 4; k < K; k += NCT * 4) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(M + (size_t)e * K + k));
        const float4 v = *reinterpret_cast<const float4 *>(s.vec + k);
        a0 = fmaf(w.x, v.x, a0);
        a1 = fmaf(w.y, v.y, a1);
        a0 = fmaf(w.z, v.z, a0);
        a1 = fmaf(w.w, v.w, a1);
      }
    }
    const float acc = warp_sum(a0 + a1);
    if ((tid & 31) == 0) s.red[tid >> 5] = acc;
    consumer_sync();
    if (tid == 0) {
      float t = 0.f;
      for (int w8 = 0; w8 < NCW; ++w8) t += s.red[w8];
      out[e] = t;
    }
    consumer_sync();
  }
}

// Warp 0 of every CTA, right after the WO barrier: the top_k experts, chosen on the unnormalised router sums
// rg x + rgwo o (the logits are these times inv_rms(h), one positive factor for all experts, so the order is the
// logits' order; only sums whose scaled values would round to the same float can rank differently, and such
// ties either side may break), in descending order, the lowest id first among equal ones. All CTAs get identical
// results from identical inputs. The ids go to the producer through the selection mbarrier at once, before the
// staging of g o h, so the routed experts' first tiles are on their way while the CTA stages. With
// p.forced_experts the given experts of (token t, layer l) are used instead of the own selection (which still
// goes to p.out_experts). Returns in lane j < top_k the sum of the j-th selected expert.
__device__ __forceinline__ float moe_sum(const DecodeParams &p, int e) {
  return __ldcg(p.rlog + e) + __ldcg(p.rlog + p.E + e);
}

__device__ inline float moe_select_ids(const DecodeParams &p, const MoeSel &sel, int t, int l) {
  const int lane = threadIdx.x & 31;
  constexpr int PER = MAX_EXPERTS / 32;
  unsigned long long key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < p.E ? argmax_key(moe_sum(p, e), e) : 0ull;
  }
  int mine = 0;
  unsigned long long mkey = 0ull;  // lane j: the key of the j-th largest sum
  for (int j = 0; j < p.top_k; ++j) {
    unsigned long long b = 0ull;
#pragma unroll
    for (int i = 0; i < PER; ++i) b = key[i] > b ? key[i] : b;
    // the warp's largest 64-bit key from two 32-bit reductions: the largest high half, then the largest low half
    // among the lanes whose own largest key has that high half (a lane's largest key is its largest low half
    // for its largest high half)
    const unsigned bh = (unsigned)(b >> 32);
    const unsigned mh = __reduce_max_sync(0xffffffffu, bh);
    const unsigned ml = __reduce_max_sync(0xffffffffu, bh == mh ? (unsigned)b : 0u);
    b = ((unsigned long long)mh << 32) | ml;
    const int id = key_index(b);
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i == id) key[i] = 0ull;
    if (lane == j) {
      mine = id;
      mkey = b;
    }
  }
  const size_t at = ((size_t)t * p.L + l) * p.top_k + lane;
  if (p.out_experts && blockIdx.x == 0 && lane < p.top_k) p.out_experts[at] = mine;
  // the selected sums come back out of their keys (no second read); forced ids read theirs
  float v = lane < p.top_k ? key_value(mkey) : 0.f;
  if (p.forced_experts && lane < p.top_k) {
    mine = p.forced_experts[at];  // ids checked on the host
    v = moe_sum(p, mine);
  }
  if (lane < p.top_k) sel.ids[lane] = mine;
  __syncwarp();
  if (lane == 0) mbar_arrive(sel.bar);
  return v;
}

// Warp 0, once inv_rms(h) is known: the routing weights, the softmax over the selected logits v_j * inv (read by
// the consumers after the expert gate/up phase).
__device__ inline void moe_select_weights(const DecodeParams &p, const MoeSel &sel, float v, float inv) {
  const int lane = threadIdx.x & 31;
  const float x = lane < p.top_k ? v * inv : -INFINITY;
  const float mx = warp_max(x);
  const float ev = lane < p.top_k ? expf(x - mx) : 0.f;
  const float sum = warp_sum(ev);
  if (lane < p.top_k) sel.wts[lane] = ev / sum;
}

__device__ inline void producer_main(const DecodeParams &p, Smem &s, const Guard &g, bool moe) {
  const uint64_t policy = l2_evict_first_policy();
  RingPos rp{0, 0u, 0};
  const RowRange rq = rows_of_cta((p.Hq + 2 * p.Hkv) * p.dh, p.n_cta, blockIdx.x);
  const RowRange ro = rows_of_cta(p.d, p.n_cta, blockIdx.x);
  const RowRange rg = rows_of_cta(2 * p.F, p.n_cta, blockIdx.x);  // gate/up rows (of each expert, for MoE)
  const RowRange rl = rows_of_cta(p.V, p.n_cta, blockIdx.x);
  const int dq = p.Hq * p.dh;
  const MoeSel sel = moe_sel(p, s);
  uint32_t nsel = 0;  // selections consumed so far (completions of the selection mbarrier)
  bool ok = true;
  for (int t = 0; t < p.n && ok; ++t) {
    for (int l = 0; l < p.L && ok; ++l) {
      const uint8_t *lw = p.wbase + (size_t)l * p.layer_stride;
      ok = ok && produce_region(lw + p.off_qkv + (size_t)rq.r0 * p.d * 2, rq.r1 - rq.r0, p.d, s, p.nslot, rp, policy, g);
      ok = ok && produce_region(lw + p.off_wo + (size_t)ro.r0 * dq * 2, ro.r1 - ro.r0, dq, s, p.nslot, rp, policy, g);
      if (moe) {
        // the routed experts are known only once the router has run: wait for the consumers' selection
        ok = ok && wait_mbar(sel.bar, nsel++ & 1u, g);
        // gate/up: two experts' rows stacked into one tile when each gives at most half a tile of rows
        const int Re = rg.r1 - rg.r0;
        const uint8_t *gub = lw + p.off_egu + (size_t)rg.r0 * p.d;
        if (Re > 0 && 2 * Re <= TILE_ROWS) {
          for (int j = 0; j < p.top_k && ok; j += 2)
            ok = produce_stacked_fp8(gub + (size_t)sel.ids[j] * p.egu_bytes,
                                     j + 1 < p.top_k ? gub + (size_t)sel.ids[j + 1] * p.egu_bytes : nullptr, Re, p.d, s,
                                     p.nslot, rp, policy, g);
        } else {
          for (int j = 0; j < p.top_k && ok; ++j)
            ok = produce_region(gub + (size_t)sel.ids[j] * p.egu_bytes, Re, p.d, s, p.nslot, rp, policy, g, 1,
                                FP8_TILE_COLS);
        }
        // the down tiles only once the last gate/up tile has landed: issued with them, they share HBM with the
        // gate/up burst that the phase waits for, while they are needed only after the next barrier
        if (ok && Re > 0) {
          const bool wrap = rp.slot == 0;
          ok = wait_mbar(&s.full[wrap ? p.nslot - 1 : rp.slot - 1], wrap ? rp.phase ^ 1u : rp.phase, g);
        }
        for (int j = 0; j < p.top_k && ok; ++j)
          ok = produce_region(lw + p.off_edn + (size_t)sel.ids[j] * p.edn_bytes + (size_t)ro.r0 * p.F, ro.r1 - ro.r0,
                              p.F, s, p.nslot, rp, policy, g, 1, FP8_TILE_COLS);
        continue;
      }
      ok = ok && produce_region(lw + p.off_gu + (size_t)rg.r0 * p.d * 2, rg.r1 - rg.r0, p.d, s, p.nslot, rp, policy, g);
      ok = ok && produce_region(lw + p.off_down + (size_t)ro.r0 * p.F * 2, ro.r1 - ro.r0, p.F, s, p.nslot, rp, policy, g);
    }
    if (ok && (!p.lm_last_only || t == p.n - 1))
      ok = produce_region(p.w_lm + (size_t)rl.r0 * p.d * 2, rl.r1 - rl.r0, p.d, s, p.nslot, rp, policy, g);
  }
  drain_ring(s, p.nslot, rp, g);
}

template <bool MOE>
__device__ inline void consumer_main(const DecodeParams &p, Smem &s, const Guard &g) {
  const int tid = threadIdx.x;
  const RowRange rq = rows_of_cta((p.Hq + 2 * p.Hkv) * p.dh, p.n_cta, blockIdx.x);
  const RowRange ro = rows_of_cta(p.d, p.n_cta, blockIdx.x);
  const RowRange rg = rows_of_cta(2 * p.F, p.n_cta, blockIdx.x);
  const RowRange rl = rows_of_cta(p.V, p.n_cta, blockIdx.x);
  const int dq = p.Hq * p.dh;
  // this CTA's rows of x and h, kept in shared memory as well as in global memory (where the other CTAs read
  // them), so the residual adds read nothing back
  float *const xs = s.out + p.out_res;
  float *const hs = xs + (ro.r1 - ro.r0);
  RingPos rp{0, 0u, 0};
  uint32_t gen = 0;
  unsigned att_target = 0;  // split-KV pieces per KV head counted so far in this launch
  unsigned long long wait_ns = 0;
  bool ok = true;
  const uint64_t t_start = globaltimer();

  for (int t = 0; t < p.n && ok; ++t) {
    const int pos = p.pos0 + t;
    // the token this step consumes, and the token greedy decode emits here
    const int predicted = t == 0 ? p.persist->next_token : key_index(__ldcg(&p.ctl->amax[(t - 1) & 1]));
    int token = p.mode == MODE_FORCED ? p.forced[t] : predicted;
    token = token < 0 ? 0 : (token >= p.V ? p.V - 1 : token);  // ids are checked on the host; never read outside E
    if (blockIdx.x == 0 && tid == 0 && p.out_tokens) p.out_tokens[t] = predicted;

    // embed: stage E[token], keep this CTA's residual slice in x; stage the RoPE row of pos
    float ss = stage_f16(s, p.embed + (size_t)token * p.d, p.d, true);
    for (int i = ro.r0 + tid; i < ro.r1; i += NCT) p.x[i] = xs[i - ro.r0] = s.vec[i];
    for (int i = tid; i < p.dh; i += NCT) s.out[p.out_rope + i] = __ldg(reinterpret_cast<const float *>(p.rope) + (size_t)pos * p.dh + i);

    for (int l = 0; l < p.L; ++l) {
      // [QKV] + RoPE + K/V append
      {  // L2 prefetch of the cached K/V rows this CTA's attention piece will read (positions before pos)
        const int c = pos + 1, S = split_pieces(p, c), C = (c + S - 1) / S;
        if (tid == 0 && (int)blockIdx.x < p.Hkv * S) {
          const int kh = blockIdx.x / S, sp = blockIdx.x % S;
          const int j0 = min(pos, sp * C), j1 = min(pos, j0 + C);
          if (j1 > j0) {
            const size_t plane = (size_t)p.max_seq * p.dh;
            const __half *Kb = p.kv + ((size_t)l * 2 * p.Hkv + kh) * plane + (size_t)j0 * p.dh;
            const __half *Vb = p.kv + ((size_t)l * 2 * p.Hkv + p.Hkv + kh) * plane + (size_t)j0 * p.dh;
            bulk_prefetch_l2(Kb, (uint32_t)((j1 - j0) * p.dh * 2));
            bulk_prefetch_l2(Vb, (uint32_t)((j1 - j0) * p.dh * 2));
          }
        }
        if (MOE && tid == 0)  // this CTA's rows of the folded router, used at the end of the QKV and WO phases
          for (int e = blockIdx.x; e < p.E; e += p.n_cta) {
            const uint8_t *lw = p.wbase + (size_t)l * p.layer_stride;
            bulk_prefetch_l2(lw + p.off_rg + (size_t)e * p.d * 4, (uint32_t)p.d * 4);
            bulk_prefetch_l2(lw + p.off_rgwo + (size_t)e * dq * 4, (uint32_t)dq * 4);
          }
      }
      const float *const rgl = reinterpret_cast<const float *>(p.wbase + (size_t)l * p.layer_stride + p.off_rg);
      RouterRow rrow;
      if constexpr (MOE) rrow = moe_router_fetch(p, rgl, p.d);
      if (l > 0) ss = stage_f32(s, p.x, p.d, true);
      consume_region(s, p.nslot, rp, rq.r1 - rq.r0, p.d, 1.0f / sqrtf(ss / (float)p.d + p.eps), g);
      consumer_sync();
      if constexpr (MOE) moe_router_part(p, s, rrow, rgl, p.d, p.rlog);  // rg x, on the staged x
      epilogue_qkv(p, s, l, pos, rq.r0, rq.r1);
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;
      if (l == 0 && blockIdx.x == 0 && tid == 0) p.ctl->amax[(t + 1) & 1] = 0ull;  // every CTA has read it

      // [ATT] split-KV attention over c = pos + 1 positions
      {
        const int c = pos + 1;
        const int S = split_pieces(p, c);
        const int C = (c + S - 1) / S;
        const int item = blockIdx.x;
        att_target += (unsigned)S;
        if (item < p.Hkv * S) {
          const int kh = item / S, sp = item % S;
          const int j0 = min(c, sp * C), j1 = min(c, j0 + C);
          if (p.dh == 128)
            attention_piece<4>(p, s, l, kh, sp, S, j0, j1, att_target, g);
          else
            attention_piece<2>(p, s, l, kh, sp, S, j0, j1, att_target, g);
        }
      }
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;

      // [WO] h = x + Wo o
      const float *const rgwol = reinterpret_cast<const float *>(p.wbase + (size_t)l * p.layer_stride + p.off_rgwo);
      if constexpr (MOE) rrow = moe_router_fetch(p, rgwol, dq);
      stage_f32(s, p.o, dq, false);
      consume_region(s, p.nslot, rp, ro.r1 - ro.r0, dq, 1.0f, g);
      consumer_sync();
      if constexpr (MOE) moe_router_part(p, s, rrow, rgwol, dq, p.rlog + p.E);  // rgwo o, on the staged o
      for (int i = tid; i < ro.r1 - ro.r0; i += NCT) p.h[ro.r0 + i] = hs[i] = xs[i] + s.out[i];
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;

      if constexpr (MOE) {
        // [SELECT] the routed experts from rg x + rgwo o (both already summed), published to the producer by warp
        // 0 while the others stage g o h for the experts, also split into fp16 high and low parts for their
        // tensor-core GEMVs, and inv_rms(h); then the routing weights from the logits inv_rms(h) * (rg x + rgwo o)
        __half *const xgu = reinterpret_cast<__half *>(s.vec + p.d);
        const MoeSel sel = moe_sel(p, s);
        float vsel = 0.f;
        if (tid < 32) vsel = moe_select_ids(p, sel, t, l);
        ss = stage_f32_gain(s, p.h, p.gffn + (size_t)l * p.d, p.d, xgu);  // ends with consumer_sync: ids visible
        const float inv = 1.0f / sqrtf(ss / (float)p.d + p.eps);
        if (tid < 32) moe_select_weights(p, sel, vsel, inv);
        // row scales of this CTA's rows of the routed experts, copied while the first tiles are in flight
        const int Re = rg.r1 - rg.r0, Rd = ro.r1 - ro.r0;
        float *const scg = s.out + p.out_moe + MOE_SEL_FLOATS, *const scd = scg + p.top_k * Re;
        {
          const float *esg = reinterpret_cast<const float *>(p.wbase + (size_t)l * p.layer_stride + p.off_esgu);
          const float *esd = reinterpret_cast<const float *>(p.wbase + (size_t)l * p.layer_stride + p.off_esdn);
          for (int i = tid; i < p.top_k * Re; i += NCT)
            cp_async4(scg + i, esg + (size_t)sel.ids[i / Re] * 2 * p.F + rg.r0 + i % Re);
          for (int i = tid; i < p.top_k * Rd; i += NCT)
            cp_async4(scd + i, esd + (size_t)sel.ids[i / Rd] * p.d + ro.r0 + i % Rd);
        }
        // [EXPERT GATE/UP] a_j = silu(gate_j) * up_j for each routed expert j, rows interleaved
        // two experts per tile when stacked (see the producer): their rows land side by side in s.out
        const int step = (Re > 0 && 2 * Re <= TILE_ROWS) ? 2 : 1;
        for (int j = 0; j < p.top_k; j += step)
          consume_region_fp8(s, p.nslot, rp, min(step, p.top_k - j) * Re, p.d, xgu, xgu + p.d, inv, s.out + j * Re,
                             s.vec + 2 * p.d, g);
        cp_async_wait_all();
        consumer_sync();
        for (int i = tid; i < p.top_k * (Re / 2); i += NCT) {
          const int j = i / (Re / 2), pr = i % (Re / 2);
          const float gt = s.out[j * Re + 2 * pr] * scg[j * Re + 2 * pr];
          const float up = s.out[j * Re + 2 * pr + 1] * scg[j * Re + 2 * pr + 1];
          p.a[(size_t)j * p.F + rg.r0 / 2 + pr] = gt / (1.0f + expf(-gt)) * up;
        }
        if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;

        // [EXPERT DOWN] x = h + sum_j w_j * (Wd_j a_j)
        // (a_j staged as fp16 high parts [top_k][F] then low parts [top_k][F])
        __half *const xdn = reinterpret_cast<__half *>(s.vec);
        const int KA = p.top_k * p.F;
        stage_split(p.a, KA, xdn);
        // one row group per expert (the usual case): each expert's partial sums stay in their own area of s.vec
        // and all are added after one consumer_sync, when s.vec has room for the top_k areas after a
        const bool dfr = Rd <= TILE_ROWS && p.vec_floats >= KA + p.top_k * FP8_RED_FLOATS;
        for (int j = 0; j < p.top_k; ++j)
          consume_region_fp8(s, p.nslot, rp, Rd, p.F, xdn + (size_t)j * p.F, xdn + KA + (size_t)j * p.F, 1.0f,
                             s.out + j * Rd, s.vec + KA + (dfr ? j * FP8_RED_FLOATS : 0), g, dfr);
        consumer_sync();
        const bool rag = p.F % FP8_TILE_COLS != 0;
        for (int i = tid; i < Rd; i += NCT) {
          float acc = 0.f;
          for (int j = 0; j < p.top_k; ++j) {
            const float v = dfr ? fp8_group_sum(s.vec + KA + j * FP8_RED_FLOATS, i, Rd, rag) * 1.0f : s.out[j * Rd + i];
            acc += sel.wts[j] * (scd[j * Rd + i] * v);
          }
          p.x[ro.r0 + i] = xs[i] = hs[i] + acc;
        }
        if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;
        continue;
      }

      // [GU] a = silu(gate) * up
      ss = stage_f32(s, p.h, p.d, true);
      consume_region(s, p.nslot, rp, rg.r1 - rg.r0, p.d, 1.0f / sqrtf(ss / (float)p.d + p.eps), g);
      consumer_sync();
      for (int pr = tid; pr < (rg.r1 - rg.r0) / 2; pr += NCT) {
        const float gt = s.out[2 * pr], up = s.out[2 * pr + 1];
        p.a[rg.r0 / 2 + pr] = gt / (1.0f + expf(-gt)) * up;
      }
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;

      // [DOWN] x = h + Wd a
      stage_f32(s, p.a, p.F, false);
      consume_region(s, p.nslot, rp, ro.r1 - ro.r0, p.F, 1.0f, g);
      consumer_sync();
      for (int i = tid; i < ro.r1 - ro.r0; i += NCT) p.x[ro.r0 + i] = xs[i] = hs[i] + s.out[i];
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;
    }
    if (!ok) break;

    // [LM] logits and greedy argmax
    if (!p.lm_last_only || t == p.n - 1) {
      ss = stage_f32(s, p.x, p.d, true);
      consume_region(s, p.nslot, rp, rl.r1 - rl.r0, p.d, 1.0f / sqrtf(ss / (float)p.d + p.eps), g);
      consumer_sync();
      float *dst = p.out_logits ? p.out_logits + (size_t)t * p.V : nullptr;
      unsigned long long best = 0ull;
      for (int i = tid; i < rl.r1 - rl.r0; i += NCT) {
        const float v = s.out[i];
        p.logits[rl.r0 + i] = v;
        if (dst) dst[rl.r0 + i] = v;
        const unsigned long long k = argmax_key(v, rl.r0 + i);
        best = k > best ? k : best;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if ((tid & 31) == 0) s.kred[tid >> 5] = best;
      consumer_sync();
      if (tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < NCW; ++w) b = s.kred[w] > b ? s.kred[w] : b;
        if (b) atomicMax(&p.ctl->amax[t & 1], b);
      }
      if (!(ok = grid_barrier(p, s, gen, g, wait_ns))) break;
      if (t == p.n - 1 && blockIdx.x == 0 && tid == 0)
        p.persist->next_token = key_index(__ldcg(&p.ctl->amax[t & 1]));
    }
  }
  if (tid == 0) {
    unsigned long long *st = p.cta_stats + (size_t)blockIdx.x * 4;
    st[0] = wait_ns;
    st[1] = gen;
    st[2] = t_start;
    st[3] = globaltimer();
  }
}

// MOE selects the sparse-MoE FFN (p.E > 0); the dense instantiation carries none of its code.
template <bool MOE>
__global__ void __launch_bounds__(BLOCK, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem s = carve_smem(smem_raw, p.nslot, p.vec_floats, p.out_floats);
  if (MOE && threadIdx.x == 0) mbar_init(moe_sel(p, s).bar, 1);  // made visible by init_ring's fence and sync
  init_ring(s, p.nslot);
  const Guard g{&p.ctl->status, p.timeout_ns};
  if (threadIdx.x >= NCT) {
    regs_release<PRODUCER_REGS>();
    if (threadIdx.x == NCT) producer_main(p, s, g, MOE);
    return;
  }
  regs_acquire<CONSUMER_REGS>();
  consumer_main<MOE>(p, s, g);
}

// The split-KV attention step alone (profiling): layers [0, n_layers) over c cached positions, with whatever q and
// cache the workspace holds, through the same device function, register split and grid barrier as decode_kernel.
// The producer warpgroup has nothing to stream and leaves after the ring set-up.
__global__ void __launch_bounds__(BLOCK, 1) attention_kernel(const DecodeParams p, int c, int n_layers) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem s = carve_smem(smem_raw, p.nslot, p.vec_floats, p.out_floats);
  init_ring(s, p.nslot);
  const Guard g{&p.ctl->status, p.timeout_ns};
  if (threadIdx.x >= NCT) {
    regs_release<PRODUCER_REGS>();
    return;
  }
  regs_acquire<CONSUMER_REGS>();
  uint32_t gen = 0;
  unsigned att_target = 0;
  unsigned long long wait_ns = 0;
  const uint64_t t_start = globaltimer();
  for (int l = 0; l < n_layers; ++l) {
    const int S = split_pieces(p, c), C = (c + S - 1) / S;
    att_target += (unsigned)S;
    if ((int)blockIdx.x < p.Hkv * S) {
      const int kh = blockIdx.x / S, sp = blockIdx.x % S;
      const int j0 = min(c, sp * C), j1 = min(c, j0 + C);
      if (p.dh == 128)
        attention_piece<4>(p, s, l, kh, sp, S, j0, j1, att_target, g);
      else
        attention_piece<2>(p, s, l, kh, sp, S, j0, j1, att_target, g);
    }
    if (!grid_barrier(p, s, gen, g, wait_ns)) break;
  }
  if (threadIdx.x == 0) {
    unsigned long long *st = p.cta_stats + (size_t)blockIdx.x * 4;
    st[0] = wait_ns;
    st[1] = gen;
    st[2] = t_start;
    st[3] = globaltimer();
  }
}

}  // namespace kie

// The register split inside the kernel is sized for LAUNCH_REGS per thread at launch; a build that compiled the
// kernel to fewer would leave the consumers' register increase waiting forever, so it is never launched.
static cudaError_t check_register_split(const void *fn) {
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, fn);
  if (e != cudaSuccess) return e;
  return a.numRegs >= kie::LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t kie_launch_attention(const kie::DecodeParams &p, size_t smem, int c, int n_layers, cudaStream_t stream) {
  const void *fn = (const void *)kie::attention_kernel;
  cudaError_t e = check_register_split(fn);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void *args[] = {(void *)&p, (void *)&c, (void *)&n_layers};
  return cudaLaunchCooperativeKernel(fn, dim3(p.n_cta), dim3(kie::BLOCK), args, smem, stream);
}

// Launch helper used by the C ABI (kie_api.cu).
cudaError_t kie_launch_decode(const kie::DecodeParams &p, size_t smem, cudaStream_t stream) {
  const void *fn = p.E > 0 ? (const void *)kie::decode_kernel<true> : (const void *)kie::decode_kernel<false>;
  cudaError_t e = check_register_split(fn);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void *args[] = {(void *)&p};
  return cudaLaunchCooperativeKernel(fn, dim3(p.n_cta), dim3(kie::BLOCK), args, smem, stream);
}

// Blocks per SM that both instantiations can keep resident with `smem` bytes of dynamic shared memory.
int kie_decode_max_blocks_per_sm(size_t smem) {
  int best = 1 << 30;
  for (const void *fn : {(const void *)kie::decode_kernel<false>, (const void *)kie::decode_kernel<true>}) {
    int nb = 0;
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kie::BLOCK, smem) != cudaSuccess) return -1;
    best = nb < best ? nb : best;
  }
  return best;
}
