// C ABI of the decode library (declared in include/kie.h): configuration checks, device buffer planning,
// the offline weight repack, and the host side of every launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kie.h"
#include "kie_decode.cuh"
#include "kie_prefill.cuh"
#include "kie_device.cuh"

cudaError_t kie_launch_decode(const kie::DecodeParams &p, size_t smem, cudaStream_t stream);
int kie_decode_max_blocks_per_sm(size_t smem);
cudaError_t kie_launch_attention(const kie::DecodeParams &p, size_t smem, int c, int n_layers, cudaStream_t stream);
cudaError_t kie_launch_gemv(const uint8_t *packed, const __half *x, float *y, int M, int K, int n_cta, int nslot,
                            unsigned long long timeout_ns, cudaStream_t stream);
cudaError_t kie_launch_pack(const uint16_t *src, uint16_t *dst, int M, int K, int n_cta, const uint16_t *gain,
                            cudaStream_t stream);
cudaError_t kie_launch_fold_router(const float *rg, const uint16_t *wo, float *out, int E, int d, int dq,
                                   cudaStream_t stream);
cudaError_t kie_launch_pack_fp8(const uint8_t *a, const uint8_t *b, uint8_t *dst, int M, int K, int n_cta,
                                cudaStream_t stream);

namespace {

constexpr int LOGIT_CHUNK = 64;  // forced-decode steps per launch when per-step logits are returned
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 1000000000ull;
constexpr size_t ALIGN = 256;

thread_local std::string g_create_error;

size_t al(size_t v) { return kie::align_up(v, ALIGN); }

// Byte offsets of the device weight buffer. Per layer (layer_stride apart): qkv, wo, then the dense FFN (gu,
// down) or the sparse-MoE FFN (the router folded by linearity: rg = router o g_ffn [E][d] and rgwo = rg Wo
// [E][dq], both fp32; egu/edn: n_experts packed FP8 matrices egu_bytes/edn_bytes apart, esgu/esdn: their row
// scales). Then the LM head, the embedding and (MoE) the fp32 FFN gains [L][d].
// Dense models also keep each layer's four projections as canonical tensor-core tiles for the batched prefill
// (tc, tc_layer_stride apart, tc_off[QKV, WO, GU, DOWN] within a layer).
struct WeightLayout {
  size_t qkv, wo, gu, down, rg, rgwo, egu, edn, esgu, esdn, egu_bytes, edn_bytes, layer_stride, lm, embed, gffn, tc,
      tc_layer_stride, tc_off[4], total;
};

// The per-launch scratch of the decode kernel: activations, router logits, split-KV partials and the control
// block. It opens the ctx workspace; kie_decode_noalloc places the same layout in its static array instead.
struct ScratchLayout {
  size_t x, h, q, o, a, rlog, part_o, part_ml, ctl, total;
};

struct WsLayout {
  ScratchLayout scr;  // at offset 0
  size_t logits, rope, persist, trace, trace_arrive, stats, tok_in, tok_out, chunk, route_in, route_out, pf_x, pf_h,
      pf_q, pf_o, pf_a,
      pf_scale, pf_part, pf_tcb, pf_att_o, pf_att_ml, total;
  int smax;
};

struct Plan {
  int n_cta, nslot, vec_floats, out_floats, out_res, out_rope, out_moe;
  size_t smem;
  WeightLayout w;
  WsLayout ws;
  size_t kv_bytes;
};

int max_rows_per_cta(int M, int n) { return 2 * ((M / 2 + n - 1) / n); }

// Split-KV pieces per KV head at most: one CTA each.
int split_kv_max(const kie_config *c, int n_cta) { return std::max(1, n_cta / c->n_kv_heads); }

ScratchLayout scratch_layout(const kie_config *c, const kie_moe_config *moe, int n_cta) {
  const int dq = c->n_heads * c->head_dim, G = c->n_heads / c->n_kv_heads, smax = split_kv_max(c, n_cta);
  const int topk = moe ? moe->top_k : 0, E = moe ? moe->n_experts : 0;
  ScratchLayout s;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  s.x = take((size_t)c->d_model * 4);
  s.h = take((size_t)c->d_model * 4);
  s.q = take((size_t)dq * 4);
  s.o = take((size_t)dq * 4);
  s.a = take((size_t)c->ffn_dim * std::max(1, topk) * 4);
  s.rlog = take((size_t)2 * E * 4);  // the two partial router logits (from x and from o) of each expert
  s.part_o = take((size_t)c->n_kv_heads * smax * G * c->head_dim * 4);
  s.part_ml = take((size_t)c->n_kv_heads * smax * G * 2 * 4);
  s.ctl = take(sizeof(kie::Ctl));
  s.total = o;
  return s;
}

const char *check_moe(const kie_config *c, const kie_moe_config *m) {
  if (!m) return nullptr;
  if (m->n_experts < 1 || m->n_experts > kie::MAX_EXPERTS) return "n_experts must be in [1, 256]";
  if (m->top_k < 1 || m->top_k > kie::MAX_TOP_K || m->top_k > m->n_experts) return "top_k must be in [1, min(8, n_experts)]";
  if (c->d_model % 16 || c->ffn_dim % 16) return "a sparse-MoE model needs d_model and ffn_dim multiples of 16";
  return nullptr;
}

const char *check_config(const kie_config *c) {
  if (!c) return "config is NULL";
  if (c->n_layers < 1) return "n_layers must be >= 1";
  if (c->d_model < 8 || c->d_model % 8) return "d_model must be a positive multiple of 8";
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (c->n_heads / c->n_kv_heads > kie::MAX_GROUP) return "more than 8 query heads per KV head";
  if (c->n_kv_heads > kie::MAX_KV_HEADS) return "more than 64 KV heads";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  if (c->ffn_dim < 8 || c->ffn_dim % 8) return "ffn_dim must be a positive multiple of 8";
  if (c->vocab < 2 || c->vocab % 2) return "vocab must be even and >= 2";
  if (c->max_seq < 1) return "max_seq must be >= 1";
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return "rms_eps must be >= 0 and rope_theta > 0";
  return nullptr;
}

// moe: null for a dense model.
const char *make_plan(const kie_config *c, const kie_moe_config *moe, int n_cta, int smem_optin, Plan *pl) {
  const int d = c->d_model, dh = c->head_dim, dq = c->n_heads * dh, G = c->n_heads / c->n_kv_heads;
  const size_t L = (size_t)c->n_layers;
  const int E = moe ? moe->n_experts : 0, topk = moe ? moe->top_k : 0, F = c->ffn_dim;
  pl->n_cta = n_cta;
  if (n_cta < c->n_kv_heads) return "the grid needs at least one CTA per KV head";
  // shared memory: ring + input vector (largest of d, F, Hq*dh, attention scratch) + row results
  // attention scratch (floats): the q operand [16][dh + 8] f16, K and V sub-chunks [ATT_SUB][dh + 8] f16,
  // scores [MAX_GROUP][ATT_SUB], the P operand [16][ATT_SUB + 8] f16, 3 x MAX_GROUP running values, and the
  // merge's [smax][G] m/weight and l arrays
  const int smax = std::max(1, n_cta / c->n_kv_heads);
  const int att = 8 * (dh + 8) + kie::ATT_SUB * (dh + 8) + kie::MAX_GROUP * kie::ATT_SUB +
                  8 * (kie::ATT_SUB + 8) + 3 * kie::MAX_GROUP + 2 * smax * G + 64;
  pl->vec_floats = std::max(std::max(std::max(d, c->ffn_dim), std::max(dq, att)), topk * F);
  // sparse MoE: the expert GEMVs' fp16 split of their input (g o h after its fp32 copy: 2d floats in all;
  // a: top_k F floats) and their cross-warp partial sums (9 x TILE_ROWS floats)
  if (moe) pl->vec_floats = std::max(pl->vec_floats, std::max(2 * d, topk * F) + kie::FP8_RED_FLOATS);
  // row results of the widest projection (for MoE also top_k experts' rows side by side), then this CTA's slices
  // of x and h, then the token's RoPE row, then (MoE) the expert selection and the routed experts' row scales
  const int rows_gu = max_rows_per_cta(2 * F, n_cta), rows_d = max_rows_per_cta(d, n_cta);
  const int rows = std::max({max_rows_per_cta((c->n_heads + 2 * c->n_kv_heads) * dh, n_cta), rows_d, rows_gu,
                             max_rows_per_cta(c->vocab, n_cta), topk * rows_gu, topk * rows_d});
  pl->out_res = (int)kie::align_up((size_t)rows, 4);
  pl->out_rope = pl->out_res + (int)kie::align_up((size_t)2 * rows_d, 4);
  pl->out_moe = pl->out_rope + (int)kie::align_up((size_t)dh, 4);
  pl->out_floats = moe ? pl->out_moe + kie::MOE_SEL_FLOATS + topk * (rows_gu + rows_d) : pl->out_rope + dh;
  const size_t fixed = kie::smem_bytes(0, pl->vec_floats, pl->out_floats);
  const long long room = (long long)smem_optin - (long long)fixed - 1024;
  int nslot = room > 0 ? (int)(room / (kie::SLOT_BYTES + 16)) : 0;
  nslot = std::min(nslot, 16);
  if (nslot < 4) return "model too wide: shared memory leaves fewer than 4 ring slots";
  pl->nslot = nslot;
  pl->smem = kie::smem_bytes(nslot, pl->vec_floats, pl->out_floats);
  // weights
  WeightLayout &w = pl->w;
  const size_t qkv = (size_t)(c->n_heads + 2 * c->n_kv_heads) * dh * d * 2;
  w = WeightLayout{};
  w.qkv = 0;
  w.wo = al(qkv);
  if (!moe) {
    w.gu = w.wo + al((size_t)d * dq * 2);
    w.down = w.gu + al((size_t)2 * F * d * 2);
    w.layer_stride = w.down + al((size_t)d * F * 2);
  } else {
    w.rg = w.wo + al((size_t)d * dq * 2);
    w.rgwo = w.rg + al((size_t)E * d * 4);
    w.egu = w.rgwo + al((size_t)E * dq * 4);
    w.egu_bytes = al((size_t)2 * F * d);
    w.edn = w.egu + E * w.egu_bytes;
    w.edn_bytes = al((size_t)d * F);
    w.esgu = w.edn + E * w.edn_bytes;
    w.esdn = w.esgu + al((size_t)E * 2 * F * 4);
    w.layer_stride = w.esdn + al((size_t)E * d * 4);
  }
  w.lm = L * w.layer_stride;
  w.embed = w.lm + al((size_t)c->vocab * d * 2);
  w.gffn = w.embed + al((size_t)c->vocab * d * 2);
  w.tc = w.gffn + (moe ? al(L * d * 4) : 0);
  const int qkv_rows = (c->n_heads + 2 * c->n_kv_heads) * dh;
  const int tcM[4] = {qkv_rows, d, 2 * F, d}, tcK[4] = {d, dq, d, F};
  if (!moe) {
    size_t o = 0;
    for (int j = 0; j < 4; ++j) {
      w.tc_off[j] = o;
      o += al(kie::kie_tc_tile_bytes(tcM[j], tcK[j]));
    }
    w.tc_layer_stride = o;
  }
  w.total = w.tc + L * w.tc_layer_stride;
  // K/V cache
  pl->kv_bytes = al(L * 2 * c->n_kv_heads * (size_t)c->max_seq * dh * 2);
  // workspace
  WsLayout &s = pl->ws;
  s.smax = split_kv_max(c, n_cta);
  s.scr = scratch_layout(c, moe, n_cta);
  size_t o = s.scr.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  s.logits = take((size_t)c->vocab * 4);
  s.rope = take((size_t)c->max_seq * (dh / 2) * 8);
  s.persist = take(sizeof(kie::Persist));
  s.trace = take((size_t)kie::TRACE_CAP * n_cta * 4);
  s.trace_arrive = take((size_t)kie::TRACE_CAP * n_cta * 8);
  s.stats = take((size_t)n_cta * 4 * 8);
  s.tok_in = take((size_t)c->max_seq * 4);
  s.tok_out = take((size_t)c->max_seq * 4);
  s.chunk = take((size_t)LOGIT_CHUNK * c->vocab * 4);
  // forced and returned expert selections of one forced-decode launch (sparse MoE)
  s.route_in = take((size_t)LOGIT_CHUNK * L * topk * 4);
  s.route_out = take((size_t)LOGIT_CHUNK * L * topk * 4);
  // batched prefill: fp32 activations of one chunk of prompt tokens
  s.pf_x = take((size_t)kie::PF_TOKENS * d * 4);
  s.pf_h = take((size_t)kie::PF_TOKENS * d * 4);
  s.pf_q = take((size_t)kie::PF_TOKENS * dq * 4);
  s.pf_o = take((size_t)kie::PF_TOKENS * dq * 4);
  s.pf_a = take((size_t)kie::PF_TOKENS * c->ffn_dim * 4);
  s.pf_scale = take((size_t)kie::PF_TOKENS * 4);
  size_t part_rows = 0, kt_max = 0;  // the K splits of each tensor-core projection, side by side
  for (int j = 0; j < 4 && !moe; ++j) {
    int kps, ns;
    kie::kie_tc_splits((tcM[j] + 127) / 128, (tcK[j] + 63) / 64, n_cta, &kps, &ns);
    part_rows = std::max(part_rows, (size_t)ns * tcM[j]);
    kt_max = std::max(kt_max, (size_t)(tcK[j] + 63) / 64);
  }
  s.pf_part = take((size_t)kie::PF_TOKENS * part_rows * 4);
  s.pf_tcb = take(kt_max * 2 * kie::PF_TOKENS * 64 * 2);
  const size_t att_parts = moe ? 0 : (size_t)kie::kie_pf_att_pieces(c->max_seq) * kie::PF_TOKENS * c->n_heads;
  s.pf_att_o = take(att_parts * dh * 4);
  s.pf_att_ml = take(att_parts * 2 * 4);
  s.total = o;
  return nullptr;
}

struct DeviceInfo {
  int dev, sms, smem_optin;
};

bool device_info(DeviceInfo *di, std::string *err) {
  cudaError_t e = cudaGetDevice(&di->dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&di->sms, cudaDevAttrMultiProcessorCount, di->dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&di->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, di->dev);
  if (e != cudaSuccess) {
    *err = std::string("CUDA device query failed: ") + cudaGetErrorString(e);
    return false;
  }
  return true;
}

}  // namespace

struct kie_ctx {
  int device = -1;  // the CUDA device the ctx was created on (current at creation)
  kie_config cfg{};
  kie_moe_config moe{};  // n_experts == 0: dense FFN
  cudaStream_t stream = nullptr;
  Plan plan{};
  bool owns = false;
  uint8_t *wbuf = nullptr, *kvbuf = nullptr, *wsbuf = nullptr;
  kie::DecodeParams base{};
  int pos = 0;
  bool has_logits = false;
  unsigned long long timeout_ns = DEFAULT_TIMEOUT_NS;
  int skip_cta = -1, skip_barrier = -1;
  int32_t *pinned = nullptr;  // host staging: [max_seq] tokens + status words
  std::string err;
};

namespace {

int fail(kie_ctx *ctx, int code, const std::string &msg) {
  if (ctx)
    ctx->err = msg;
  else
    g_create_error = msg;
  return code;
}

int cuda_fail(kie_ctx *ctx, cudaError_t e, const char *what) {
  return fail(ctx, KIE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define KIE_CUDA(ctx, call)                                  \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
  } while (0)

// Host copy of the fused QKV matrix: every query and key head becomes dh/2 row pairs (i, i + dh/2), so that
// one CTA holds both inputs of each RoPE rotation; value heads are copied as they are.
void fuse_qkv(const kie_config &c, const uint16_t *wq, const uint16_t *wk, const uint16_t *wv, uint16_t *dst) {
  const int d = c.d_model, dh = c.head_dim, half = dh / 2;
  const size_t row = (size_t)d;
  auto pairs = [&](const uint16_t *src, int heads) {
    for (int h = 0; h < heads; ++h)
      for (int i = 0; i < half; ++i) {
        std::memcpy(dst, src + ((size_t)h * dh + i) * row, row * 2);
        dst += row;
        std::memcpy(dst, src + ((size_t)h * dh + i + half) * row, row * 2);
        dst += row;
      }
  };
  pairs(wq, c.n_heads);
  pairs(wk, c.n_kv_heads);
  std::memcpy(dst, wv, (size_t)c.n_kv_heads * dh * row * 2);
}

// Host copy of the gate/up matrix with rows interleaved: row 2j = gate_j, row 2j+1 = up_j.
void fuse_gate_up(const kie_config &c, const uint16_t *wg, const uint16_t *wu, uint16_t *dst) {
  const size_t row = (size_t)c.d_model;
  for (int j = 0; j < c.ffn_dim; ++j) {
    std::memcpy(dst + (2 * (size_t)j) * row, wg + (size_t)j * row, row * 2);
    std::memcpy(dst + (2 * (size_t)j + 1) * row, wu + (size_t)j * row, row * 2);
  }
}

// Upload a row-major fp16 [M, K] matrix and pack it for the decode (dst) and, if tc_dst is not null, as
// canonical tensor-core tiles for the prefill; gain_host (or null) is folded into the columns of both.
int upload_and_pack(kie_ctx *ctx, const uint16_t *host, int M, int K, uint8_t *dst, const uint16_t *gain_host,
                    uint16_t *stage, uint16_t *gain_dev, uint8_t *tc_dst = nullptr) {
  const size_t bytes = (size_t)M * K * 2;
  KIE_CUDA(ctx, cudaMemcpyAsync(stage, host, bytes, cudaMemcpyHostToDevice, ctx->stream));
  const uint16_t *g = nullptr;
  if (gain_host) {
    KIE_CUDA(ctx, cudaMemcpyAsync(gain_dev, gain_host, (size_t)K * 2, cudaMemcpyHostToDevice, ctx->stream));
    g = gain_dev;
  }
  KIE_CUDA(ctx, kie_launch_pack(stage, (uint16_t *)dst, M, K, ctx->plan.n_cta, g, ctx->stream));
  if (tc_dst) KIE_CUDA(ctx, kie_launch_tc_pack(stage, M, K, g, tc_dst, ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  return KIE_OK;
}

int upload(kie_ctx *ctx, uint8_t *dst, const void *host, size_t bytes) {
  KIE_CUDA(ctx, cudaMemcpyAsync(dst, host, bytes, cudaMemcpyHostToDevice, ctx->stream));
  return KIE_OK;
}

// The sparse-MoE FFN of layer l: the router folded by linearity (rg = router o g_ffn, exact in fp32, and
// rgwo = rg Wo in fp64 on the device, rounded to fp32), each expert's FP8 gate/up (rows interleaved) and down
// matrices packed through `stage` (>= 2 * max(F, dq) * d bytes), row scales interleaved like the rows, FFN gain
// as fp32.
int repack_moe_layer(kie_ctx *ctx, const kie_weights *w, const kie_moe_weights *mw, int l, uint8_t *stage) {
  const kie_config &c = ctx->cfg;
  const Plan &pl = ctx->plan;
  const int d = c.d_model, F = c.ffn_dim, E = ctx->moe.n_experts, dq = c.n_heads * c.head_dim;
  uint8_t *lw = ctx->wbuf + (size_t)l * pl.w.layer_stride;
  std::vector<float> rg((size_t)E * d);
  for (int e = 0; e < E; ++e)
    for (int j = 0; j < d; ++j) {
      __half_raw r, g;
      r.x = mw->router[l][(size_t)e * d + j];
      g.x = w->ffn_norm[l][j];
      rg[(size_t)e * d + j] = __half2float(__half(r)) * __half2float(__half(g));  // exact: 11 x 11 bits
    }
  int rc = upload(ctx, lw + pl.w.rg, rg.data(), rg.size() * 4);
  if (rc == KIE_OK) rc = upload(ctx, stage, w->wo[l], (size_t)d * dq * 2);
  if (rc == KIE_OK) {
    KIE_CUDA(ctx, kie_launch_fold_router(reinterpret_cast<const float *>(lw + pl.w.rg),
                                         reinterpret_cast<const uint16_t *>(stage),
                                         reinterpret_cast<float *>(lw + pl.w.rgwo), E, d, dq, ctx->stream));
    KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));  // rg (host) and the staged Wo are reused below
  }
  for (int e = 0; e < E && rc == KIE_OK; ++e) {
    const size_t m = (size_t)F * d;
    rc = upload(ctx, stage, mw->gate_q[l] + (size_t)e * m, m);
    if (rc == KIE_OK) rc = upload(ctx, stage + m, mw->up_q[l] + (size_t)e * m, m);
    if (rc == KIE_OK) {
      KIE_CUDA(ctx, kie_launch_pack_fp8(stage, stage + m, lw + pl.w.egu + (size_t)e * pl.w.egu_bytes, 2 * F, d,
                                        pl.n_cta, ctx->stream));
      KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
      rc = upload(ctx, stage, mw->down_q[l] + (size_t)e * m, m);
    }
    if (rc == KIE_OK) {
      KIE_CUDA(ctx, kie_launch_pack_fp8(stage, nullptr, lw + pl.w.edn + (size_t)e * pl.w.edn_bytes, d, F, pl.n_cta,
                                        ctx->stream));
      KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
    }
  }
  if (rc != KIE_OK) return rc;
  std::vector<float> sgu((size_t)E * 2 * F), gain(d);
  for (size_t i = 0; i < (size_t)E * F; ++i) {
    sgu[2 * i] = mw->gate_s[l][i];
    sgu[2 * i + 1] = mw->up_s[l][i];
  }
  for (int i = 0; i < d; ++i) {
    __half_raw r;
    r.x = w->ffn_norm[l][i];
    gain[i] = __half2float(__half(r));
  }
  rc = upload(ctx, lw + pl.w.esgu, sgu.data(), sgu.size() * 4);
  if (rc == KIE_OK) rc = upload(ctx, lw + pl.w.esdn, mw->down_s[l], (size_t)E * d * 4);
  if (rc == KIE_OK) rc = upload(ctx, ctx->wbuf + pl.w.gffn + (size_t)l * d * 4, gain.data(), (size_t)d * 4);
  if (rc == KIE_OK) KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));  // the host vectors die here
  return rc;
}

int repack_weights(kie_ctx *ctx, const kie_weights *w, const kie_moe_weights *mw) {
  const kie_config &c = ctx->cfg;
  const Plan &pl = ctx->plan;
  const bool moe = ctx->moe.n_experts > 0;
  const int d = c.d_model, dh = c.head_dim, dq = c.n_heads * dh, F = c.ffn_dim;
  const int Mqkv = (c.n_heads + 2 * c.n_kv_heads) * dh;
  const size_t stage_elems = std::max({(size_t)Mqkv * d, (size_t)d * dq, (size_t)2 * F * d, (size_t)c.vocab * d});
  uint16_t *stage = nullptr, *gain = nullptr;
  cudaError_t e = cudaMalloc(&stage, stage_elems * 2);
  if (e != cudaSuccess) return fail(ctx, KIE_ERR_OOM, "staging buffer for the repack: out of device memory");
  e = cudaMalloc(&gain, (size_t)std::max(d, F) * 2);
  if (e != cudaSuccess) {
    cudaFree(stage);
    return fail(ctx, KIE_ERR_OOM, "staging buffer for the repack: out of device memory");
  }
  std::vector<uint16_t> host(std::max((size_t)Mqkv * d, (size_t)2 * F * d));
  int rc = KIE_OK;
  for (int l = 0; l < c.n_layers && rc == KIE_OK; ++l) {
    uint8_t *lw = ctx->wbuf + (size_t)l * pl.w.layer_stride;
    uint8_t *tw = moe ? nullptr : ctx->wbuf + pl.w.tc + (size_t)l * pl.w.tc_layer_stride;
    fuse_qkv(c, w->wq[l], w->wk[l], w->wv[l], host.data());
    rc = upload_and_pack(ctx, host.data(), Mqkv, d, lw + pl.w.qkv, w->attn_norm[l], stage, gain,
                         tw ? tw + pl.w.tc_off[0] : nullptr);
    if (rc == KIE_OK)
      rc = upload_and_pack(ctx, w->wo[l], d, dq, lw + pl.w.wo, nullptr, stage, gain, tw ? tw + pl.w.tc_off[1] : nullptr);
    if (moe) {
      if (rc == KIE_OK) rc = repack_moe_layer(ctx, w, mw, l, reinterpret_cast<uint8_t *>(stage));
      continue;
    }
    if (rc == KIE_OK) {
      fuse_gate_up(c, w->w_gate[l], w->w_up[l], host.data());
      rc = upload_and_pack(ctx, host.data(), 2 * F, d, lw + pl.w.gu, w->ffn_norm[l], stage, gain, tw + pl.w.tc_off[2]);
    }
    if (rc == KIE_OK)
      rc = upload_and_pack(ctx, w->w_down[l], d, F, lw + pl.w.down, nullptr, stage, gain, tw + pl.w.tc_off[3]);
  }
  if (rc == KIE_OK) rc = upload_and_pack(ctx, w->lm_head, c.vocab, d, ctx->wbuf + pl.w.lm, w->final_norm, stage, gain);
  if (rc == KIE_OK) {
    e = cudaMemcpyAsync(ctx->wbuf + pl.w.embed, w->embed, (size_t)c.vocab * d * 2, cudaMemcpyHostToDevice, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) rc = cuda_fail(ctx, e, "embedding upload");
  }
  cudaFree(stage);
  cudaFree(gain);
  return rc;
}

// RoPE table: row p holds (cos, sin) of p * theta^(-2i/dh) for i < dh/2, evaluated in fp64, stored fp32.
int upload_rope(kie_ctx *ctx) {
  const kie_config &c = ctx->cfg;
  const int half = c.head_dim / 2;
  std::vector<float> tab((size_t)c.max_seq * half * 2);
  for (int i = 0; i < half; ++i) {
    const double inv_freq = std::exp(-2.0 * i / c.head_dim * std::log((double)c.rope_theta));
    for (int p = 0; p < c.max_seq; ++p) {
      const double ang = (double)p * inv_freq;
      tab[((size_t)p * half + i) * 2] = (float)std::cos(ang);
      tab[((size_t)p * half + i) * 2 + 1] = (float)std::sin(ang);
    }
  }
  KIE_CUDA(ctx, cudaMemcpyAsync(ctx->wsbuf + ctx->plan.ws.rope, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice,
                                ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  return KIE_OK;
}

// Point the per-launch scratch of p at `base` laid out as `l`.
void point_scratch(kie::DecodeParams &p, uint8_t *base, const ScratchLayout &l) {
  p.x = (float *)(base + l.x);
  p.h = (float *)(base + l.h);
  p.q = (float *)(base + l.q);
  p.o = (float *)(base + l.o);
  p.a = (float *)(base + l.a);
  p.rlog = (float *)(base + l.rlog);
  p.part_o = (float *)(base + l.part_o);
  p.part_ml = (float *)(base + l.part_ml);
  p.ctl = (kie::Ctl *)(base + l.ctl);
}

void fill_base(kie_ctx *ctx) {
  const kie_config &c = ctx->cfg;
  const Plan &pl = ctx->plan;
  kie::DecodeParams &p = ctx->base;
  std::memset(&p, 0, sizeof(p));
  p.L = c.n_layers;
  p.d = c.d_model;
  p.Hq = c.n_heads;
  p.Hkv = c.n_kv_heads;
  p.dh = c.head_dim;
  p.F = c.ffn_dim;
  p.V = c.vocab;
  p.max_seq = c.max_seq;
  p.n_cta = pl.n_cta;
  p.nslot = pl.nslot;
  p.vec_floats = pl.vec_floats;
  p.out_floats = pl.out_floats;
  p.out_res = pl.out_res;
  p.out_rope = pl.out_rope;
  p.out_moe = pl.out_moe;
  p.E = ctx->moe.n_experts;
  p.top_k = ctx->moe.top_k;
  p.off_rg = (long long)pl.w.rg;
  p.off_rgwo = (long long)pl.w.rgwo;
  p.off_egu = (long long)pl.w.egu;
  p.off_edn = (long long)pl.w.edn;
  p.off_esgu = (long long)pl.w.esgu;
  p.off_esdn = (long long)pl.w.esdn;
  p.egu_bytes = (long long)pl.w.egu_bytes;
  p.edn_bytes = (long long)pl.w.edn_bytes;
  p.gffn = (const float *)(ctx->wbuf + pl.w.gffn);
  p.eps = c.rms_eps;
  p.wbase = ctx->wbuf;
  p.layer_stride = (long long)pl.w.layer_stride;
  p.off_qkv = (long long)pl.w.qkv;
  p.off_wo = (long long)pl.w.wo;
  p.off_gu = (long long)pl.w.gu;
  p.off_down = (long long)pl.w.down;
  p.w_lm = ctx->wbuf + pl.w.lm;
  p.embed = (const __half *)(ctx->wbuf + pl.w.embed);
  p.kv = (__half *)ctx->kvbuf;
  uint8_t *ws = ctx->wsbuf;
  p.rope = (const float2 *)(ws + pl.ws.rope);
  point_scratch(p, ws, pl.ws.scr);
  p.logits = (float *)(ws + pl.ws.logits);
  p.smax = pl.ws.smax;
  p.persist = (kie::Persist *)(ws + pl.ws.persist);
  p.trace = (uint32_t *)(ws + pl.ws.trace);
  p.trace_arrive = (unsigned long long *)(ws + pl.ws.trace_arrive);
  p.cta_stats = (unsigned long long *)(ws + pl.ws.stats);
  p.skip_cta = -1;
  p.skip_barrier = -1;
}

// moe / mw: null for a dense model.
int create_common(const kie_config *cfg, const kie_moe_config *moe, const kie_weights *w, const kie_moe_weights *mw,
                  void *stream, void *wdev, size_t wbytes, void *kvdev, size_t kvbytes, void *wsdev, size_t wsbytes,
                  kie_ctx **out) {
  if (!out) return fail(nullptr, KIE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (const char *m = check_config(cfg)) return fail(nullptr, KIE_ERR_INVALID, m);
  if (const char *m = check_moe(cfg, moe)) return fail(nullptr, KIE_ERR_INVALID, m);
  const bool dense = moe == nullptr;
  if (!w || !w->embed || !w->lm_head || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
      !w->ffn_norm || (dense && (!w->w_gate || !w->w_up || !w->w_down)))
    return fail(nullptr, KIE_ERR_INVALID, "a weight pointer is NULL");
  for (int l = 0; l < cfg->n_layers; ++l)
    if (!w->attn_norm[l] || !w->wq[l] || !w->wk[l] || !w->wv[l] || !w->wo[l] || !w->ffn_norm[l] ||
        (dense && (!w->w_gate[l] || !w->w_up[l] || !w->w_down[l])))
      return fail(nullptr, KIE_ERR_INVALID, "a per-layer weight pointer is NULL");
  if (!dense) {
    if (!mw || !mw->router || !mw->gate_q || !mw->up_q || !mw->down_q || !mw->gate_s || !mw->up_s || !mw->down_s)
      return fail(nullptr, KIE_ERR_INVALID, "a MoE weight pointer is NULL");
    for (int l = 0; l < cfg->n_layers; ++l)
      if (!mw->router[l] || !mw->gate_q[l] || !mw->up_q[l] || !mw->down_q[l] || !mw->gate_s[l] || !mw->up_s[l] ||
          !mw->down_s[l])
        return fail(nullptr, KIE_ERR_INVALID, "a per-layer MoE weight pointer is NULL");
  }
  DeviceInfo di;
  std::string err;
  if (!device_info(&di, &err)) return fail(nullptr, KIE_ERR_CUDA, err);
  kie_ctx *ctx = new kie_ctx();
  ctx->device = di.dev;
  ctx->cfg = *cfg;
  if (moe) ctx->moe = *moe;
  ctx->stream = (cudaStream_t)stream;
  if (const char *m = make_plan(cfg, moe, di.sms, di.smem_optin, &ctx->plan)) {
    delete ctx;
    return fail(nullptr, KIE_ERR_INVALID, m);
  }
  const int nb = kie_decode_max_blocks_per_sm(ctx->plan.smem);
  if (nb < 1) {
    delete ctx;
    return fail(nullptr, KIE_ERR_LAUNCH, "the decode kernel cannot be resident with its shared memory");
  }
  const Plan &pl = ctx->plan;
  if (wdev) {
    if (wbytes < pl.w.total || kvbytes < pl.kv_bytes || wsbytes < pl.ws.total || ((uintptr_t)wdev % ALIGN) ||
        ((uintptr_t)kvdev % ALIGN) || ((uintptr_t)wsdev % ALIGN)) {
      delete ctx;
      return fail(nullptr, KIE_ERR_INVALID, "a caller buffer is too small or not 256-byte aligned");
    }
    ctx->wbuf = (uint8_t *)wdev;
    ctx->kvbuf = (uint8_t *)kvdev;
    ctx->wsbuf = (uint8_t *)wsdev;
  } else {
    ctx->owns = true;
    if (cudaMalloc(&ctx->wbuf, pl.w.total) != cudaSuccess || cudaMalloc(&ctx->kvbuf, pl.kv_bytes) != cudaSuccess ||
        cudaMalloc(&ctx->wsbuf, pl.ws.total) != cudaSuccess) {
      cudaGetLastError();
      kie_destroy(ctx);
      return fail(nullptr, KIE_ERR_OOM, "device allocation failed");
    }
  }
  if (cudaMallocHost(&ctx->pinned, ((size_t)cfg->max_seq + 64) * 4) != cudaSuccess) {
    cudaGetLastError();
    kie_destroy(ctx);
    return fail(nullptr, KIE_ERR_OOM, "pinned host allocation failed");
  }
  int rc = KIE_OK;
  cudaError_t e = cudaMemsetAsync(ctx->kvbuf, 0, pl.kv_bytes, ctx->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->wsbuf, 0, pl.ws.total, ctx->stream);
  if (e != cudaSuccess) rc = cuda_fail(ctx, e, "clearing device buffers");
  if (rc == KIE_OK) rc = repack_weights(ctx, w, mw);
  if (rc == KIE_OK) rc = upload_rope(ctx);
  if (rc != KIE_OK) {
    g_create_error = ctx->err;
    kie_destroy(ctx);
    return rc;
  }
  fill_base(ctx);
  *out = ctx;
  return KIE_OK;
}

// One launch of the decode kernel. forced_dev / out_tokens_dev / out_logits_dev may be null. scratch: the
// per-launch scratch (laid out by scratch_layout), or null for the ctx workspace's. route_in_dev / route_out_dev:
// forced and returned expert selections ([n][L][top_k], sparse MoE), or null.
int launch(kie_ctx *ctx, int n, int mode, int lm_last_only, const int *forced_dev, int *out_tokens_dev,
           float *out_logits_dev, uint8_t *scratch = nullptr, const int *route_in_dev = nullptr,
           int *route_out_dev = nullptr) {
  kie::DecodeParams p = ctx->base;
  if (scratch) point_scratch(p, scratch, ctx->plan.ws.scr);
  p.forced_experts = route_in_dev;
  p.out_experts = route_out_dev;
  p.pos0 = ctx->pos;
  p.n = n;
  p.mode = mode;
  p.lm_last_only = lm_last_only;
  p.forced = forced_dev;
  p.out_tokens = out_tokens_dev;
  p.out_logits = out_logits_dev;
  p.timeout_ns = ctx->timeout_ns;
  p.skip_cta = ctx->skip_cta;
  p.skip_barrier = ctx->skip_barrier;
  ctx->skip_cta = ctx->skip_barrier = -1;
  const Plan &pl = ctx->plan;
  KIE_CUDA(ctx, cudaMemsetAsync(p.ctl, 0, sizeof(kie::Ctl), ctx->stream));
  KIE_CUDA(ctx, cudaMemsetAsync(ctx->wsbuf + pl.ws.stats, 0, (size_t)pl.n_cta * 32, ctx->stream));
  cudaError_t e = kie_launch_decode(p, pl.smem, ctx->stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return fail(ctx, KIE_ERR_LAUNCH, "cooperative launch refused: the grid cannot be co-resident");
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "decode kernel launch");
  ctx->pos += n;
  return KIE_OK;
}

// Wait for the stream and read the status word of the last launch (whose scratch was `scratch`, or the ctx
// workspace's when null).
int finish(kie_ctx *ctx, uint8_t *scratch = nullptr) {
  int32_t *st = ctx->pinned + ctx->cfg.max_seq;
  const uint8_t *ctl = (scratch ? scratch : ctx->wsbuf) + ctx->plan.ws.scr.ctl;
  KIE_CUDA(ctx, cudaMemcpyAsync(st, ctl + offsetof(kie::Ctl, status), 8, cudaMemcpyDeviceToHost, ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  if (st[0] != kie::ST_OK) {
    ctx->pos = 0;
    ctx->has_logits = false;
    char buf[160];
    std::snprintf(buf, sizeof buf, "device wait timed out (status %d, first timed-out barrier %d); sequence reset",
                  st[0], st[1] - 1);
    return fail(ctx, KIE_ERR_TIMEOUT, buf);
  }
  return KIE_OK;
}

}  // namespace

extern "C" {

static int query_buffers(const kie_config *cfg, const kie_moe_config *moe, int n_cta, kie_buffer_sizes *out) {
  if (!out) return KIE_ERR_INVALID;
  if (const char *m = check_config(cfg)) return fail(nullptr, KIE_ERR_INVALID, m);
  if (const char *m = check_moe(cfg, moe)) return fail(nullptr, KIE_ERR_INVALID, m);
  DeviceInfo di{0, n_cta, 232448};
  std::string err;
  if (n_cta <= 0) {
    if (!device_info(&di, &err)) return fail(nullptr, KIE_ERR_CUDA, err);
  }
  Plan pl;
  if (const char *m = make_plan(cfg, moe, di.sms, di.smem_optin, &pl)) return fail(nullptr, KIE_ERR_INVALID, m);
  out->weights_bytes = pl.w.total;
  out->kv_bytes = pl.kv_bytes;
  out->workspace_bytes = pl.ws.total;
  out->n_cta = pl.n_cta;
  return KIE_OK;
}

int kie_query_buffers(const kie_config *cfg, int n_cta, kie_buffer_sizes *out) {
  return query_buffers(cfg, nullptr, n_cta, out);
}

int kie_query_buffers_moe(const kie_config *cfg, const kie_moe_config *moe, int n_cta, kie_buffer_sizes *out) {
  if (!moe) return fail(nullptr, KIE_ERR_INVALID, "moe is NULL");
  return query_buffers(cfg, moe, n_cta, out);
}

int kie_create(const kie_config *cfg, const kie_weights *w, void *stream, kie_ctx **out) {
  return create_common(cfg, nullptr, w, nullptr, stream, nullptr, 0, nullptr, 0, nullptr, 0, out);
}

int kie_create_moe(const kie_config *cfg, const kie_moe_config *moe, const kie_weights *w, const kie_moe_weights *mw,
                   void *stream, kie_ctx **out) {
  if (!moe) return fail(nullptr, KIE_ERR_INVALID, "moe is NULL");
  return create_common(cfg, moe, w, mw, stream, nullptr, 0, nullptr, 0, nullptr, 0, out);
}

int kie_create_moe_with_buffers(const kie_config *cfg, const kie_moe_config *moe, const kie_weights *w,
                                const kie_moe_weights *mw, void *stream, void *weights_dev, size_t weights_bytes,
                                void *kv_dev, size_t kv_bytes, void *workspace_dev, size_t workspace_bytes,
                                kie_ctx **out) {
  if (!moe) return fail(nullptr, KIE_ERR_INVALID, "moe is NULL");
  if (!weights_dev || !kv_dev || !workspace_dev) return fail(nullptr, KIE_ERR_INVALID, "a device buffer is NULL");
  return create_common(cfg, moe, w, mw, stream, weights_dev, weights_bytes, kv_dev, kv_bytes, workspace_dev,
                       workspace_bytes, out);
}

int kie_create_with_buffers(const kie_config *cfg, const kie_weights *w, void *stream, void *weights_dev,
                            size_t weights_bytes, void *kv_dev, size_t kv_bytes, void *workspace_dev,
                            size_t workspace_bytes, kie_ctx **out) {
  if (!weights_dev || !kv_dev || !workspace_dev) return fail(nullptr, KIE_ERR_INVALID, "a device buffer is NULL");
  return create_common(cfg, nullptr, w, nullptr, stream, weights_dev, weights_bytes, kv_dev, kv_bytes, workspace_dev,
                       workspace_bytes, out);
}

int kie_prefill(kie_ctx *ctx, const int32_t *tokens, int n) {
  if (!ctx) return KIE_ERR_INVALID;
  if (!tokens || n < 1) return fail(ctx, KIE_ERR_INVALID, "prefill needs n >= 1 tokens");
  if ((long long)ctx->pos + n > ctx->cfg.max_seq) return fail(ctx, KIE_ERR_CAPACITY, "prompt exceeds max_seq");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= ctx->cfg.vocab) return fail(ctx, KIE_ERR_INVALID, "token id out of range");
  std::memcpy(ctx->pinned, tokens, (size_t)n * 4);
  int *tin = (int *)(ctx->wsbuf + ctx->plan.ws.tok_in);
  KIE_CUDA(ctx, cudaMemcpyAsync(tin, ctx->pinned, (size_t)n * 4, cudaMemcpyHostToDevice, ctx->stream));
  if (ctx->moe.n_experts > 0) {
    // sparse MoE: the prompt goes through the decode kernel position by position (each token routes to its own
    // experts), teacher-forced, with the LM head at the last position only
    int rc = launch(ctx, n, kie::MODE_FORCED, 1, tin, nullptr, nullptr);
    if (rc == KIE_OK) rc = finish(ctx);
    if (rc == KIE_OK) ctx->has_logits = true;
    return rc;
  }
  // batched: the prompt moves through each layer in chunks of up to PF_TOKENS tokens (kie_prefill.cu)
  const WsLayout &ws = ctx->plan.ws;
  const WeightLayout &wl = ctx->plan.w;
  uint8_t *b = ctx->wsbuf;
  kie::PrefillBufs pb{(float *)(b + ws.pf_x), (float *)(b + ws.pf_h), (float *)(b + ws.pf_q),
                      (float *)(b + ws.pf_o), (float *)(b + ws.pf_a), (float *)(b + ws.pf_scale),
                      (float *)(b + ws.pf_part), (float *)(b + ws.pf_att_o), (float *)(b + ws.pf_att_ml),
                      ctx->wbuf + wl.tc, (long long)wl.tc_layer_stride,
                      {(long long)wl.tc_off[0], (long long)wl.tc_off[1], (long long)wl.tc_off[2], (long long)wl.tc_off[3]},
                      b + ws.pf_tcb, &ctx->base.ctl->status, ctx->timeout_ns};
  KIE_CUDA(ctx, cudaMemsetAsync(ctx->wsbuf + ctx->plan.ws.scr.ctl, 0, sizeof(kie::Ctl), ctx->stream));
  const cudaError_t e = kie_run_prefill(ctx->base, pb, tin, ctx->pos, n, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "prefill launch");
  ctx->pos += n;
  const int rc = finish(ctx);  // the status word: a tensor-core GEMM wait that ran out resets the sequence
  if (rc == KIE_OK) ctx->has_logits = true;
  return rc;
}

int kie_decode_async(kie_ctx *ctx, int n, int32_t *out_tokens_dev) {
  if (!ctx) return KIE_ERR_INVALID;
  if (n < 1 || !out_tokens_dev) return fail(ctx, KIE_ERR_INVALID, "decode needs n >= 1 and an output buffer");
  if (!ctx->has_logits) return fail(ctx, KIE_ERR_INVALID, "decode before prefill: there are no current logits");
  if ((long long)ctx->pos + n > ctx->cfg.max_seq) return fail(ctx, KIE_ERR_CAPACITY, "decode exceeds max_seq");
  return launch(ctx, n, kie::MODE_DECODE, 0, nullptr, out_tokens_dev, nullptr);
}

int kie_sync(kie_ctx *ctx) {
  if (!ctx) return KIE_ERR_INVALID;
  return finish(ctx);
}

int kie_decode(kie_ctx *ctx, int n, int32_t *out_tokens) {
  if (!ctx) return KIE_ERR_INVALID;
  if (!out_tokens) return fail(ctx, KIE_ERR_INVALID, "out_tokens is NULL");
  int *tout = (int *)(ctx->wsbuf + ctx->plan.ws.tok_out);
  int rc = kie_decode_async(ctx, n, tout);
  if (rc != KIE_OK) return rc;
  KIE_CUDA(ctx, cudaMemcpyAsync(ctx->pinned, tout, (size_t)n * 4, cudaMemcpyDeviceToHost, ctx->stream));
  rc = finish(ctx);
  if (rc == KIE_OK) std::memcpy(out_tokens, ctx->pinned, (size_t)n * 4);
  return rc;
}

// Teacher-forced launches in chunks of LOGIT_CHUNK steps (the per-step logits of a chunk fit the workspace).
// Without current logits (allowed only when allow_start is set) the first emitted token is undefined: -1.
static int decode_forced_impl(kie_ctx *ctx, int n, const int32_t *forced, const int32_t *forced_experts,
                              int32_t *out_tokens, float *out_logits, int32_t *out_experts, bool allow_start) {
  if (!ctx) return KIE_ERR_INVALID;
  if (n < 1 || !forced || !out_tokens) return fail(ctx, KIE_ERR_INVALID, "forced decode needs n >= 1 and buffers");
  if (!ctx->has_logits && !allow_start)
    return fail(ctx, KIE_ERR_INVALID, "decode before prefill: there are no current logits");
  if ((long long)ctx->pos + n > ctx->cfg.max_seq) return fail(ctx, KIE_ERR_CAPACITY, "decode exceeds max_seq");
  for (int i = 0; i < n; ++i)
    if (forced[i] < 0 || forced[i] >= ctx->cfg.vocab) return fail(ctx, KIE_ERR_INVALID, "token id out of range");
  const int E = ctx->moe.n_experts, K = ctx->moe.top_k, L = ctx->cfg.n_layers;
  if ((forced_experts || out_experts) && E == 0)
    return fail(ctx, KIE_ERR_INVALID, "expert selections are given or asked for, but the model is dense");
  if (forced_experts)
    for (size_t i = 0; i < (size_t)n * L * K; ++i)
      if (forced_experts[i] < 0 || forced_experts[i] >= E) return fail(ctx, KIE_ERR_INVALID, "expert id out of range");
  const bool fresh = !ctx->has_logits;
  const int V = ctx->cfg.vocab;
  const size_t per_step = (size_t)L * K;  // expert ids per forward
  int *tin = (int *)(ctx->wsbuf + ctx->plan.ws.tok_in);
  int *tout = (int *)(ctx->wsbuf + ctx->plan.ws.tok_out);
  float *chunk = (float *)(ctx->wsbuf + ctx->plan.ws.chunk);
  int *rin = (int *)(ctx->wsbuf + ctx->plan.ws.route_in);
  int *rout = (int *)(ctx->wsbuf + ctx->plan.ws.route_out);
  for (int done = 0; done < n;) {
    const int m = std::min(LOGIT_CHUNK, n - done);
    std::memcpy(ctx->pinned, forced + done, (size_t)m * 4);
    KIE_CUDA(ctx, cudaMemcpyAsync(tin, ctx->pinned, (size_t)m * 4, cudaMemcpyHostToDevice, ctx->stream));
    if (forced_experts)
      KIE_CUDA(ctx, cudaMemcpyAsync(rin, forced_experts + (size_t)done * per_step, (size_t)m * per_step * 4,
                                    cudaMemcpyHostToDevice, ctx->stream));
    int rc = launch(ctx, m, kie::MODE_FORCED, 0, tin, tout, out_logits ? chunk : nullptr, nullptr,
                    forced_experts ? rin : nullptr, out_experts ? rout : nullptr);
    if (rc != KIE_OK) return rc;
    KIE_CUDA(ctx, cudaMemcpyAsync(out_tokens + done, tout, (size_t)m * 4, cudaMemcpyDeviceToHost, ctx->stream));
    if (out_logits)
      KIE_CUDA(ctx, cudaMemcpyAsync(out_logits + (size_t)done * V, chunk, (size_t)m * V * 4, cudaMemcpyDeviceToHost,
                                    ctx->stream));
    if (out_experts)
      KIE_CUDA(ctx, cudaMemcpyAsync(out_experts + (size_t)done * per_step, rout, (size_t)m * per_step * 4,
                                    cudaMemcpyDeviceToHost, ctx->stream));
    rc = finish(ctx);
    if (rc != KIE_OK) return rc;
    ctx->has_logits = true;
    done += m;
  }
  if (fresh) out_tokens[0] = -1;
  return KIE_OK;
}

int kie_decode_forced(kie_ctx *ctx, int n, const int32_t *forced, int32_t *out_tokens, float *out_logits) {
  return decode_forced_impl(ctx, n, forced, nullptr, out_tokens, out_logits, nullptr, false);
}

int kie_decode_forced_routed(kie_ctx *ctx, int n, const int32_t *forced, const int32_t *forced_experts,
                             int32_t *out_tokens, float *out_logits, int32_t *out_experts) {
  return decode_forced_impl(ctx, n, forced, forced_experts, out_tokens, out_logits, out_experts, true);
}

int kie_get_logits(kie_ctx *ctx, float *out) {
  if (!ctx) return KIE_ERR_INVALID;
  if (!out) return fail(ctx, KIE_ERR_INVALID, "out is NULL");
  if (!ctx->has_logits) return fail(ctx, KIE_ERR_INVALID, "no current logits");
  KIE_CUDA(ctx, cudaMemcpyAsync(out, ctx->wsbuf + ctx->plan.ws.logits, (size_t)ctx->cfg.vocab * 4,
                                cudaMemcpyDeviceToHost, ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  return KIE_OK;
}

int kie_position(const kie_ctx *ctx) { return ctx ? ctx->pos : KIE_ERR_INVALID; }

int kie_reset(kie_ctx *ctx) {
  if (!ctx) return KIE_ERR_INVALID;
  ctx->pos = 0;
  ctx->has_logits = false;
  return KIE_OK;
}

int kie_set_timeout_ns(kie_ctx *ctx, uint64_t ns) {
  if (!ctx || ns == 0) return KIE_ERR_INVALID;
  ctx->timeout_ns = ns;
  return KIE_OK;
}

int kie_get_barrier_stats(kie_ctx *ctx, kie_barrier_stats *out) {
  if (!ctx || !out) return KIE_ERR_INVALID;
  const Plan &pl = ctx->plan;
  const int n = pl.n_cta;
  std::vector<unsigned long long> st((size_t)n * 4);
  KIE_CUDA(ctx, cudaMemcpyAsync(st.data(), ctx->wsbuf + pl.ws.stats, st.size() * 8, cudaMemcpyDeviceToHost, ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  const long long bars = (long long)st[1];
  const int traced = (int)std::min<long long>(bars, kie::TRACE_CAP);
  std::vector<uint32_t> tr((size_t)std::max(traced, 1) * n);
  if (traced > 0) {
    KIE_CUDA(ctx, cudaMemcpyAsync(tr.data(), ctx->wsbuf + pl.ws.trace, (size_t)traced * n * 4, cudaMemcpyDeviceToHost,
                                  ctx->stream));
    KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  }
  double wait = 0, cnt = 0, lat = 0;
  for (int i = 0; i < n; ++i) {
    wait += (double)st[(size_t)i * 4];
    cnt += (double)st[(size_t)i * 4 + 1];
  }
  for (int b = 0; b < traced; ++b) {
    uint32_t m = 0xFFFFFFFFu;
    for (int i = 0; i < n; ++i) m = std::min(m, tr[(size_t)b * n + i]);
    lat += m;
  }
  out->barriers = bars;
  out->mean_wait_ns = cnt > 0 ? wait / cnt : 0.0;
  out->mean_latency_ns = traced > 0 ? lat / traced : 0.0;
  out->total_ns = (double)(st[3] - st[2]);
  return KIE_OK;
}

int kie_get_barrier_trace(kie_ctx *ctx, int first, int count, uint64_t *arrive_ns, uint32_t *wait_ns) {
  if (!ctx || first < 0 || count < 0 || (count > 0 && (!arrive_ns || !wait_ns)))
    return fail(ctx, KIE_ERR_INVALID, "bad trace request");
  const Plan &pl = ctx->plan;
  const size_t n = (size_t)pl.n_cta;
  unsigned long long bars = 0;
  KIE_CUDA(ctx, cudaMemcpyAsync(&bars, ctx->wsbuf + pl.ws.stats + 8, 8, cudaMemcpyDeviceToHost, ctx->stream));
  KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  const long long avail = std::min<long long>((long long)bars, kie::TRACE_CAP);
  const int m = (int)std::max<long long>(0, std::min<long long>(count, avail - first));
  if (m > 0) {
    KIE_CUDA(ctx, cudaMemcpyAsync(arrive_ns, ctx->wsbuf + pl.ws.trace_arrive + (size_t)first * n * 8, (size_t)m * n * 8,
                                  cudaMemcpyDeviceToHost, ctx->stream));
    KIE_CUDA(ctx, cudaMemcpyAsync(wait_ns, ctx->wsbuf + pl.ws.trace + (size_t)first * n * 4, (size_t)m * n * 4,
                                  cudaMemcpyDeviceToHost, ctx->stream));
    KIE_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
  }
  return m;
}

int kie_debug_skip_arrival(kie_ctx *ctx, int cta, int barrier) {
  if (!ctx) return KIE_ERR_INVALID;
  ctx->skip_cta = cta;
  ctx->skip_barrier = barrier;
  return KIE_OK;
}

int kie_profile_attention(kie_ctx *ctx, int c, int n_layers) {
  if (!ctx) return KIE_ERR_INVALID;
  if (c < 1 || c > ctx->cfg.max_seq || n_layers < 1 || n_layers > ctx->cfg.n_layers)
    return fail(ctx, KIE_ERR_INVALID, "profile_attention needs 1 <= c <= max_seq and 1 <= n_layers <= n_layers");
  kie::DecodeParams p = ctx->base;
  p.timeout_ns = ctx->timeout_ns;
  const Plan &pl = ctx->plan;
  KIE_CUDA(ctx, cudaMemsetAsync(p.ctl, 0, sizeof(kie::Ctl), ctx->stream));
  KIE_CUDA(ctx, cudaMemsetAsync(ctx->wsbuf + pl.ws.stats, 0, (size_t)pl.n_cta * 32, ctx->stream));
  const cudaError_t e = kie_launch_attention(p, pl.smem, c, n_layers, ctx->stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return fail(ctx, KIE_ERR_LAUNCH, "cooperative launch refused: the grid cannot be co-resident");
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "attention kernel launch");
  const bool had = ctx->has_logits;
  const int pos = ctx->pos;
  const int rc = finish(ctx);
  if (rc == KIE_OK) {  // the sequence is untouched (the step writes only the attention outputs and partials)
    ctx->has_logits = had;
    ctx->pos = pos;
  }
  return rc;
}

int kie_n_cta(const kie_ctx *ctx) { return ctx ? ctx->plan.n_cta : KIE_ERR_INVALID; }

const char *kie_last_error(const kie_ctx *ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

void kie_destroy(kie_ctx *ctx) {
  if (!ctx) return;
  if (ctx->stream || ctx->wbuf) cudaStreamSynchronize(ctx->stream);
  if (ctx->owns) {
    cudaFree(ctx->wbuf);
    cudaFree(ctx->kvbuf);
    cudaFree(ctx->wsbuf);
  }
  if (ctx->pinned) cudaFreeHost(ctx->pinned);
  delete ctx;
}

size_t kie_gemv_packed_bytes(int M, int K) { return (size_t)M * K * 2; }

static int gemv_ncta(int n_cta) {
  if (n_cta > 0) return n_cta;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return sms;
}

int kie_gemv_pack(const uint16_t *W_dev, int M, int K, int n_cta, uint16_t *packed_dev, void *stream) {
  if (!W_dev || !packed_dev || M < 2 || M % 2 || K < 8 || K % 8) return fail(nullptr, KIE_ERR_INVALID, "bad GEMV shape");
  if (((uintptr_t)W_dev | (uintptr_t)packed_dev) % 16) return fail(nullptr, KIE_ERR_INVALID, "unaligned buffer");
  const int n = gemv_ncta(n_cta);
  if (n < 1) return fail(nullptr, KIE_ERR_CUDA, "device query failed");
  cudaError_t e = kie_launch_pack(W_dev, packed_dev, M, K, n, nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? KIE_OK : fail(nullptr, KIE_ERR_CUDA, cudaGetErrorString(e));
}

int kie_gemv(const uint16_t *packed_dev, const uint16_t *x_dev, float *y_dev, int M, int K, int n_cta, void *stream) {
  if (!packed_dev || !x_dev || !y_dev || M < 2 || M % 2 || K < 8 || K % 8) return fail(nullptr, KIE_ERR_INVALID, "bad GEMV shape");
  if (((uintptr_t)packed_dev | (uintptr_t)x_dev | (uintptr_t)y_dev) % 16) return fail(nullptr, KIE_ERR_INVALID, "unaligned buffer");
  DeviceInfo di;
  std::string err;
  if (!device_info(&di, &err)) return fail(nullptr, KIE_ERR_CUDA, err);
  const int n = n_cta > 0 ? n_cta : di.sms;
  const int out_floats = max_rows_per_cta(M, n) + 2;
  const size_t fixed = kie::smem_bytes(0, K, out_floats);
  const long long room = (long long)di.smem_optin - (long long)fixed - 1024;
  const int nslot = std::min(16, room > 0 ? (int)(room / (kie::SLOT_BYTES + 16)) : 0);
  if (nslot < 2) return fail(nullptr, KIE_ERR_INVALID, "K too large for the shared-memory input vector");
  cudaError_t e = kie_launch_gemv((const uint8_t *)packed_dev, (const __half *)x_dev, y_dev, M, K, n, nslot,
                                  DEFAULT_TIMEOUT_NS, (cudaStream_t)stream);
  return e == cudaSuccess ? KIE_OK : fail(nullptr, KIE_ERR_CUDA, cudaGetErrorString(e));
}

int64_t kie_packed_offset_fp8(int M, int K, int n_cta, int r, int c) {
  if (M < 2 || M % 2 || K < 16 || K % 16 || n_cta < 1 || r < 0 || r >= M || c < 0 || c >= K) return -1;
  return kie::packed_offset_fp8(M, K, n_cta, r, c);
}

int64_t kie_packed_offset(int M, int K, int n_cta, int r, int c) {
  if (M < 2 || M % 2 || K < 1 || n_cta < 1 || r < 0 || r >= M || c < 0 || c >= K) return -1;
  return kie::packed_offset(M, K, n_cta, r, c);
}

int kie_rows_of_cta(int M, int n_cta, int cta, int *r0, int *r1) {
  if (M < 2 || M % 2 || n_cta < 1 || cta < 0 || cta >= n_cta || !r0 || !r1) return KIE_ERR_INVALID;
  const kie::RowRange r = kie::rows_of_cta(M, n_cta, cta);
  *r0 = r.r0;
  *r1 = r.r1;
  return KIE_OK;
}

}  // extern "C"

// ---- decode without device allocation ---------------------------------------------------------------------
//
// kie_decode_noalloc runs the same kernel through the same launch path as kie_decode, but the per-launch scratch
// (activations, split-KV partials and the control block, laid out by scratch_layout) lives in the static array
// below instead of the ctx workspace. Nothing in this path allocates device or host memory. The array is a
// file-scope __device__ object, so each GPU that loads the library holds KIE_NOALLOC_SCRATCH_BYTES of it until the
// process exits; host code never uses its name as an address, only the device address that cudaGetSymbolAddress
// returns for the ctx's device (which must be current).

static __device__ __align__(256) unsigned char g_noalloc_scratch[KIE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int NOALLOC_MAX_DEVICES = 64;
void *g_noalloc_addr[NOALLOC_MAX_DEVICES];  // device address of g_noalloc_scratch per device (null: not set up)
std::mutex g_noalloc_mutex;

// Once per device, with that device current: the device address of the static scratch array.
int noalloc_scratch(kie_ctx *ctx, uint8_t **out) {
  int dev = 0;
  KIE_CUDA(ctx, cudaGetDevice(&dev));
  if (dev != ctx->device) {
    char buf[160];
    std::snprintf(buf, sizeof buf, "kie_decode_noalloc: the ctx's device %d must be current (device %d is)",
                  ctx->device, dev);
    return fail(ctx, KIE_ERR_INVALID, buf);
  }
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return fail(ctx, KIE_ERR_INVALID, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(ctx, e, "cudaGetSymbolAddress(static decode scratch)");
    g_noalloc_addr[dev] = p;
  }
  *out = (uint8_t *)g_noalloc_addr[dev];
  return KIE_OK;
}

}  // namespace

extern "C" int kie_decode_noalloc(kie_ctx *ctx, int n, int32_t *out_tokens_dev) {
  if (!ctx) return KIE_ERR_INVALID;
  if (n < 1 || !out_tokens_dev) return fail(ctx, KIE_ERR_INVALID, "decode needs n >= 1 and an output buffer");
  if (!ctx->has_logits) return fail(ctx, KIE_ERR_INVALID, "decode before prefill: there are no current logits");
  if ((long long)ctx->pos + n > ctx->cfg.max_seq) return fail(ctx, KIE_ERR_CAPACITY, "decode exceeds max_seq");
  const size_t need = ctx->plan.ws.scr.total;
  if (need > KIE_NOALLOC_SCRATCH_BYTES) {
    char buf[200];
    std::snprintf(buf, sizeof buf,
                  "this model needs %zu bytes of decode scratch; the static scratch of kie_decode_noalloc holds %u",
                  need, (unsigned)KIE_NOALLOC_SCRATCH_BYTES);
    return fail(ctx, KIE_ERR_INVALID, buf);
  }
  uint8_t *scr = nullptr;
  int rc = noalloc_scratch(ctx, &scr);
  if (rc != KIE_OK) return rc;
  // launch() clears the control block (the array keeps whatever the previous call left in it) and takes any
  // armed kie_debug_skip_arrival, like every other launch
  rc = launch(ctx, n, kie::MODE_DECODE, 0, nullptr, out_tokens_dev, nullptr, scr);
  if (rc != KIE_OK) return rc;
  return finish(ctx, scr);
}
