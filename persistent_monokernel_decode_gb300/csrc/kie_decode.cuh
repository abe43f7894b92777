// Parameters and control block of the persistent decode kernel (shared by the kernel and the C ABI).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace kie {

constexpr int MAX_GROUP = 8;         // query heads per KV head supported by the attention step
constexpr int ATT_SUB = 32;          // positions per online-softmax sub-chunk (one lane each)
constexpr int MAX_KV_HEADS = 64;
constexpr int TRACE_CAP = 4096;      // grid barriers whose per-CTA waits are recorded per launch
constexpr int MAX_EXPERTS = 256;     // sparse-MoE experts per layer supported by the router step
constexpr int MAX_TOP_K = 8;         // experts per token
constexpr int MOE_SEL_FLOATS = 32;   // selection area of the row-result region: ids, weights, sequence word

// Zeroed by the host before every launch.
struct Ctl {
  unsigned bar_count;
  unsigned pad0[31];
  int status;
  int where;
  unsigned pad1[30];
  unsigned long long amax[2];  // packed (orderable logit, ~index) argmax of the even / odd token
  unsigned pad2[28];
  unsigned att_cnt[MAX_KV_HEADS];  // split-KV pieces per KV head published so far in this launch
};

// Survives across launches.
struct Persist {
  int next_token;  // argmax of the current logits
  int pad[31];
};

enum Mode { MODE_DECODE = 0, MODE_FORCED = 1 };

struct DecodeParams {
  int L, d, Hq, Hkv, dh, F, V, max_seq;
  int n_cta, nslot, vec_floats, out_floats;
  int out_res, out_rope;  // floats into the row-result area: this CTA's x and h slices, the token's RoPE row
  float eps;
  // packed weights: layer l's projections start at wbase + l * layer_stride (+ off_*)
  const uint8_t *wbase;
  long long layer_stride, off_qkv, off_wo, off_gu, off_down;
  const uint8_t *w_lm;
  const __half *embed;  // [V][d], plain
  // state and activations (device)
  __half *kv;           // [L][2][Hkv][max_seq][dh]; K rows hold each RoPE pair (i, i + dh/2) adjacent
  const float2 *rope;   // [max_seq][dh/2] (cos, sin)
  float *x, *h, *q, *o, *a, *logits;
  float *part_o, *part_ml;  // [Hkv][smax][group][dh], [Hkv][smax][group][2]
  int smax;                 // split-KV pieces per KV head at most
  Ctl *ctl;
  Persist *persist;
  uint32_t *trace;                 // [TRACE_CAP][n_cta] barrier wait (ns)
  unsigned long long *trace_arrive;  // [TRACE_CAP][n_cta] %globaltimer at arrival (ns)
  unsigned long long *cta_stats;   // [n_cta][4]: wait ns, barriers, start, end
  // this launch
  int pos0, n, mode, lm_last_only;
  const int *forced;   // [n] device (forced mode)
  int *out_tokens;     // [n] device or null
  float *out_logits;   // [n][V] device or null
  unsigned long long timeout_ns;
  int skip_cta, skip_barrier;
  // sparse-MoE FFN (E > 0; E == 0 is the dense FFN above). Per layer: the router folded by linearity, rg =
  // router o g_ffn [E][d] and rgwo = rg Wo [E][dq] (fp32, row-major), and E SwiGLU experts of width F with FP8
  // E4M3 weights in the packed layout with FP8_TILE_COLS-wide blocks, each row with an fp32 scale. In the layer
  // block: off_rg, off_rgwo; off_egu + e * egu_bytes = expert e's gate/up rows interleaved [2F][d]; off_edn +
  // e * edn_bytes = its down rows [d][F]; off_esgu: scales [E][2F] (interleaved like the rows); off_esdn: scales
  // [E][d].
  int E, top_k;
  int out_moe;  // floats into the row-result area: the selection (MOE_SEL_FLOATS), then the staged row scales
  long long off_rg, off_rgwo, off_egu, off_edn, off_esgu, off_esdn, egu_bytes, edn_bytes;
  const float *gffn;  // [L][d] FFN RMSNorm gains (fp32), applied to the staged vector (FP8 weights keep them out)
  float *rlog;        // [2][E] the current layer's partial router logits: rg x and rgwo o
  // testing aids (device, or null): forced_experts [n][L][top_k] replaces each layer's own top_k selection (the
  // routing weights are still the softmax of this launch's router logits over the given experts); out_experts
  // [n][L][top_k] receives the kernel's own selection, in selection order
  const int *forced_experts;
  int *out_experts;
};

}  // namespace kie
