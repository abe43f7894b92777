/*
 * CPU oracle for batch-1 greedy decode of a dense Llama-style decoder. TEST INFRASTRUCTURE ONLY:
 * it is loaded by the tests, by __graft_entry__.smoke() and by the bench's CPU-baseline leg, never by
 * the product path, and it shares no code, header, table or constant with the GPU library.
 *
 * What it computes (the Kog monokernel pages, "inside the monokernel" and the fusion list in the same
 * section: the monokernel folds RMSNorm, repacks QKV, precomputes RoPE and recomputes attention; all four
 * are exact reformulations of the plain forward, so this file computes the plain forward, unfolded):
 *   x = E[t]; per layer: u = rmsnorm(x) * g_attn; q, k, v = Wq u, Wk u, Wv u; RoPE(q, k, pos);
 *   cache[pos] = fp16(k), fp16(v); o_h = softmax(q_h K_g^T / sqrt(dh)) V_g with g = h / (Hq / Hkv);
 *   x += Wo o; u = rmsnorm(x) * g_ffn; x += Wd (silu(Wg u) * (Wu u));
 *   logits = Wlm (rmsnorm(x) * g_final); next token = argmax (lowest index on ties).
 * The pages leave the architecture details open (pre-norm, no biases, SwiGLU, rotate-half RoPE, 0-based
 * positions, contiguous GQA groups, fp16 only in weights and K/V cache); this file takes that plainest
 * Llama reading.
 *
 * Precision: fp16 weights and K/V cache, arithmetic in REAL = float (orc_*_f32) or double (orc_*_f64).
 * Build with -ffp-contract=off so that every product and sum is rounded as written.
 *
 * Sparse-MoE layers (orc_set_moe; the pages' "Extending to frontier MoE models" section of the Kog blog post
 * and the MoE projection of the creeta article's "2B demo vs frontier scale" section): the FFN of a layer is
 *   r = W_router u (fp16 router); S = the top_k experts by r (lowest index first on ties);
 *   w_e = softmax over {r_e : e in S}; x += sum_{e in S} w_e * Wd_e (silu(Wg_e u) * (Wu_e u)),
 * where an expert weight is E4M3(q) * s_row (OCP FP8 E4M3, per-output-row fp32 scale), applied as
 * y_row = s_row * sum_k E4M3(q_row,k) x_k.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_seq;
  float rope_theta, rms_eps;
} orc_config;

typedef struct {
  const uint16_t *embed, *lm_head, *final_norm;
  const uint16_t *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
  const uint16_t *const *ffn_norm, *const *w_gate, *const *w_up, *const *w_down;
} orc_weights;

/* Sparse-MoE FFN weights (borrowed), per layer: router [E][d] fp16; gate/up [E][F_e][d] and down [E][d][F_e]
 * E4M3 codes; gate_s/up_s [E][F_e] and down_s [E][d] row scales. */
typedef struct {
  int n_experts, top_k, expert_ffn;
  const uint16_t *const *router;
  const uint8_t *const *gate_q, *const *up_q, *const *down_q;
  const float *const *gate_s, *const *up_s, *const *down_s;
} orc_moe;

typedef struct {
  orc_config cfg;
  orc_weights w; /* borrowed: the caller keeps every tensor alive */
  orc_moe moe;   /* n_experts == 0: dense FFN */
  const void **moe_ptrs; /* owned copies of the MoE per-layer pointer arrays */
  const uint16_t **ptrs; /* owned copies of the per-layer pointer arrays */
  int precision;         /* 32 or 64 */
  int pos;
  uint16_t *kv; /* [L][2][Hkv][max_seq][dh] fp16 bits */
  void *x, *u, *q, *k, *v, *o, *t, *g, *up, *scores;
  void *rl, *acc; /* MoE: router logits [E], FFN output [d] */
  double route_margin; /* MoE diagnostic: smallest gap between the last selected and the best unselected logit */
  int *route_ids;      /* MoE: experts selected by each layer of the last forward [L][top_k], in selection order */
  double *route_gap;   /* MoE: that layer's gap (k-th selected logit minus the best unselected one) [L] */
} orc_model;

/* ---- binary16 <-> real, from the format's definition ---------------------------------------------- */

static float half_table[65536];
static int half_table_ready = 0;

static double half_decode(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static void half_init(void) {
  if (half_table_ready) return;
  for (int i = 0; i < 65536; ++i) half_table[i] = (float)half_decode((uint16_t)i);
  half_table_ready = 1;
}

static inline float half_value(uint16_t h) { return half_table[h]; }

/* ---- OCP FP8 E4M3 ("fn": no infinities, 0x7F / 0xFF NaN) -> real, from the format's definition ---------- */

static double e4m3_table[256];
static int e4m3_table_ready = 0;

static double e4m3_decode(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, f = b & 7;
  double v;
  if (e == 15 && f == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)f, -9); /* subnormal: f/8 * 2^-6 */
  else
    v = ldexp(1.0 + f / 8.0, e - 7);
  return sign ? -v : v;
}

static void e4m3_init(void) {
  if (e4m3_table_ready) return;
  for (int i = 0; i < 256; ++i) e4m3_table[i] = e4m3_decode((uint8_t)i);
  e4m3_table_ready = 1;
}

/* Round a real to the nearest binary16 (ties to even) by scaling to the format's quantum at that
 * magnitude and rounding to an integer there (nearbyint in the default round-to-nearest-even mode). */
static uint16_t half_bits(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7E00;
  if (a == 0.0) return sign;
  int E;
  frexp(a, &E); /* a = m * 2^E, m in [0.5, 1): leading bit weighs 2^(E-1) */
  int lead = E - 1;
  double quantum = ldexp(1.0, (lead < -14 ? -14 : lead) - 10);
  double r = nearbyint(a / quantum) * quantum; /* exact: scaling by powers of two */
  if (r >= 65520.0) return sign | 0x7C00;
  if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24)); /* subnormal (or min normal) */
  frexp(r, &E);
  lead = E - 1;
  uint16_t mant = (uint16_t)(r / ldexp(1.0, lead - 10) - 1024.0);
  return sign | (uint16_t)((lead + 15) << 10) | mant;
}

/* ---- the two instantiations ----------------------------------------------------------------------- */

#define REAL float
#define NAME(x) x##_f32
#define SQRT sqrtf
#define EXP expf
#include "oracle_impl.h"
#undef REAL
#undef NAME
#undef SQRT
#undef EXP

#define REAL double
#define NAME(x) x##_f64
#define SQRT sqrt
#define EXP exp
#include "oracle_impl.h"
#undef REAL
#undef NAME
#undef SQRT
#undef EXP

/* ---- exported API (ctypes) ------------------------------------------------------------------------ */

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

double orc_half_to_double(uint16_t h) { return half_decode(h); }
uint16_t orc_double_to_half(double v) { return half_bits(v); }

int orc_argmax_f32(const float *v, int n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

int orc_argmax_f64(const double *v, int n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

void orc_rmsnorm_f32(const float *x, const uint16_t *g, int n, float eps, float *out) { half_init(); rmsnorm_f32(x, g, n, eps, out); }
void orc_rmsnorm_f64(const double *x, const uint16_t *g, int n, double eps, double *out) { half_init(); rmsnorm_f64(x, g, n, eps, out); }
void orc_gemv_f32(const uint16_t *W, const float *x, int M, int K, float *y) { half_init(); gemv_f32(W, x, M, K, y); }
void orc_gemv_f64(const uint16_t *W, const double *x, int M, int K, double *y) { half_init(); gemv_f64(W, x, M, K, y); }
void orc_rope_f32(float *v, int dh, int pos, double theta) { rope_f32(v, dh, pos, theta); }
void orc_rope_f64(double *v, int dh, int pos, double theta) { rope_f64(v, dh, pos, theta); }
float orc_silu_f32(float z) { return silu_f32(z); }
double orc_silu_f64(double z) { return silu_f64(z); }

void orc_attention_f32(const float *q, const uint16_t *K, const uint16_t *V, int c, int dh, float *out) {
  half_init();
  float *sc = (float *)malloc(sizeof(float) * (size_t)(c > 0 ? c : 1));
  attention_f32(q, K, V, c, dh, (size_t)dh, sc, out);
  free(sc);
}

void orc_attention_f64(const double *q, const uint16_t *K, const uint16_t *V, int c, int dh, double *out) {
  half_init();
  double *sc = (double *)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
  attention_f64(q, K, V, c, dh, (size_t)dh, sc, out);
  free(sc);
}

void orc_destroy(orc_model *m);

/* NULL on a bad cfg or a failed host allocation (nothing is leaked). */
orc_model *orc_create(const orc_config *cfg, const orc_weights *w, int precision) {
  half_init();
  if (!cfg || !w || (precision != 32 && precision != 64)) return NULL;
  if (cfg->n_layers < 0 || cfg->d_model <= 0 || cfg->n_heads <= 0 || cfg->n_kv_heads <= 0 ||
      cfg->n_heads % cfg->n_kv_heads || cfg->head_dim <= 0 || cfg->head_dim % 2 || cfg->ffn_dim <= 0 ||
      cfg->vocab <= 0 || cfg->max_seq <= 0)
    return NULL;
  orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
  if (!m) return NULL;
  m->route_margin = INFINITY;
  m->cfg = *cfg;
  m->precision = precision;
  int L = cfg->n_layers;
  m->ptrs = (const uint16_t **)calloc((size_t)(9 * (L > 0 ? L : 1)), sizeof(uint16_t *));
  if (!m->ptrs) {
    orc_destroy(m);
    return NULL;
  }
  const uint16_t *const *src[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm, w->w_gate, w->w_up, w->w_down};
  const uint16_t *const **dst[9] = {&m->w.attn_norm, &m->w.wq, &m->w.wk, &m->w.wv, &m->w.wo,
                                    &m->w.ffn_norm, &m->w.w_gate, &m->w.w_up, &m->w.w_down};
  for (int j = 0; j < 9; ++j) {
    const uint16_t **slot = m->ptrs + (size_t)j * (L > 0 ? L : 1);
    for (int l = 0; l < L; ++l) slot[l] = src[j][l];
    *dst[j] = slot;
  }
  m->w.embed = w->embed;
  m->w.lm_head = w->lm_head;
  m->w.final_norm = w->final_norm;
  size_t es = precision == 32 ? sizeof(float) : sizeof(double);
  int d = cfg->d_model, qd = cfg->n_heads * cfg->head_dim, kd = cfg->n_kv_heads * cfg->head_dim;
  int wide = d > qd ? d : qd;
  m->kv = (uint16_t *)calloc((size_t)L * 2 * cfg->n_kv_heads * cfg->max_seq * cfg->head_dim + 1, 2);
  m->x = calloc((size_t)d, es);
  m->u = calloc((size_t)d, es);
  m->q = calloc((size_t)qd, es);
  m->k = calloc((size_t)kd, es);
  m->v = calloc((size_t)kd, es);
  m->o = calloc((size_t)qd, es);
  m->t = calloc((size_t)wide, es);
  m->g = calloc((size_t)cfg->ffn_dim, es);
  m->up = calloc((size_t)cfg->ffn_dim, es);
  m->scores = calloc((size_t)cfg->max_seq * cfg->n_heads, es); /* one score row per query head */
  if (!m->kv || !m->x || !m->u || !m->q || !m->k || !m->v || !m->o || !m->t || !m->g || !m->up || !m->scores) {
    orc_destroy(m);
    return NULL;
  }
  return m;
}

void orc_destroy(orc_model *m) {
  if (!m) return;
  free(m->ptrs);
  free(m->moe_ptrs);
  free(m->rl);
  free(m->acc);
  free(m->route_ids);
  free(m->route_gap);
  free(m->kv);
  free(m->x); free(m->u); free(m->q); free(m->k); free(m->v);
  free(m->o); free(m->t); free(m->g); free(m->up); free(m->scores);
  free(m);
}

int orc_pos(const orc_model *m) { return m->pos; }
void orc_reset(orc_model *m) { m->pos = 0; }

/* Forward one token; logits is float[vocab] (precision 32) or double[vocab] (precision 64), or NULL to skip the
 * final norm and LM head (a prompt position whose logits are not needed; the cache and state are the same).
 * Returns 0, or -1 when the cache is full or the token is out of range. */
int orc_forward(orc_model *m, int token, void *logits) {
  if (m->pos >= m->cfg.max_seq || token < 0 || token >= m->cfg.vocab) return -1;
  if (m->precision == 32)
    forward_f32(m, token, (float *)logits);
  else
    forward_f64(m, token, (double *)logits);
  return 0;
}

/* Read back the cached K (kv = 0) or V (kv = 1) row of (layer, kv_head, pos) as fp16 bits. */
void orc_kv_row(const orc_model *m, int layer, int kv, int head, int pos, uint16_t *out) {
  const orc_config *c = &m->cfg;
  size_t S = (size_t)c->max_seq * c->head_dim;
  const uint16_t *p = m->kv + ((size_t)layer * 2 + kv) * c->n_kv_heads * S + head * S + (size_t)pos * c->head_dim;
  memcpy(out, p, sizeof(uint16_t) * (size_t)c->head_dim);
}

/* ---- sparse-MoE layers ------------------------------------------------------------------------------------- */

/* Give the model sparse-MoE FFN layers (replacing the dense ones). Pointers are borrowed. Returns 0, or -1 for
 * an invalid description (top_k outside 1..min(n_experts, 64), n_experts > 64, expert_ffn < 1). */
int orc_set_moe(orc_model *m, const orc_moe *moe) {
  e4m3_init();
  if (!m || !moe || moe->n_experts < 1 || moe->n_experts > 1024 || moe->top_k < 1 || moe->top_k > moe->n_experts ||
      moe->expert_ffn < 1)
    return -1;
  const int L = m->cfg.n_layers > 0 ? m->cfg.n_layers : 1;
  free(m->moe_ptrs);
  m->moe_ptrs = (const void **)calloc((size_t)7 * L, sizeof(void *));
  m->moe = *moe;
  const void *const *src[7] = {(const void *const *)moe->router, (const void *const *)moe->gate_q,
                               (const void *const *)moe->up_q, (const void *const *)moe->down_q,
                               (const void *const *)moe->gate_s, (const void *const *)moe->up_s,
                               (const void *const *)moe->down_s};
  for (int j = 0; j < 7; ++j)
    for (int l = 0; l < m->cfg.n_layers; ++l) m->moe_ptrs[(size_t)j * L + l] = src[j][l];
  m->moe.router = (const uint16_t *const *)(m->moe_ptrs + 0 * (size_t)L);
  m->moe.gate_q = (const uint8_t *const *)(m->moe_ptrs + 1 * (size_t)L);
  m->moe.up_q = (const uint8_t *const *)(m->moe_ptrs + 2 * (size_t)L);
  m->moe.down_q = (const uint8_t *const *)(m->moe_ptrs + 3 * (size_t)L);
  m->moe.gate_s = (const float *const *)(m->moe_ptrs + 4 * (size_t)L);
  m->moe.up_s = (const float *const *)(m->moe_ptrs + 5 * (size_t)L);
  m->moe.down_s = (const float *const *)(m->moe_ptrs + 6 * (size_t)L);
  const size_t es = m->precision == 32 ? sizeof(float) : sizeof(double);
  const int d = m->cfg.d_model, Fe = moe->expert_ffn;
  const int gmax = Fe > m->cfg.ffn_dim ? Fe : m->cfg.ffn_dim;
  free(m->g);
  free(m->up);
  m->g = calloc((size_t)gmax, es);
  m->up = calloc((size_t)gmax, es);
  free(m->rl);
  free(m->acc);
  free(m->route_ids);
  free(m->route_gap);
  m->rl = calloc((size_t)moe->n_experts, es);
  m->acc = calloc((size_t)d, es);
  m->route_ids = (int *)calloc((size_t)L * moe->top_k, sizeof(int));
  m->route_gap = (double *)calloc((size_t)L, sizeof(double));
  if (!m->moe_ptrs || !m->g || !m->up || !m->rl || !m->acc || !m->route_ids || !m->route_gap) return -1;
  return 0;
}

/* The routing of the last forward: ids [n_layers][top_k] (each layer's experts in selection order: descending
 * router logit, the lowest id first among equal ones) and gaps [n_layers] (that layer's k-th selected logit
 * minus its best unselected one; +inf when every expert is selected). Either may be NULL. Returns -1 for a dense
 * model. */
int orc_route_ids(const orc_model *m, int *ids, double *gaps) {
  if (!m || m->moe.n_experts < 1) return -1;
  const int L = m->cfg.n_layers;
  if (ids) memcpy(ids, m->route_ids, sizeof(int) * (size_t)L * m->moe.top_k);
  if (gaps) memcpy(gaps, m->route_gap, sizeof(double) * (size_t)L);
  return 0;
}

/* The MoE FFN output of layer l for a given normalised input u (float or double by the model's precision). */
/* The smallest routing margin seen since the last call with reset != 0 (or since creation): over every MoE layer
 * evaluated, the top_k-th largest router logit minus the largest unselected one (+inf when every expert is
 * selected). A test uses it to tell routing decisions that rounding cannot change from near-ties. */
double orc_route_margin(orc_model *m, int reset) {
  const double v = m->route_margin;
  if (reset) m->route_margin = INFINITY;
  return v;
}

void orc_moe_ffn(orc_model *m, int layer, const void *u, void *out) {
  if (m->precision == 32)
    moe_ffn_f32(m, layer, (const float *)u, (float *)out);
  else
    moe_ffn_f64(m, layer, (const double *)u, (double *)out);
}

double orc_e4m3_to_double(uint8_t b) { return e4m3_decode(b); }
void orc_gemv_fp8_f64(const uint8_t *W, const float *s, const double *x, int M, int K, double *y) {
  e4m3_init();
  gemv_fp8_f64(W, s, x, M, K, y);
}
void orc_gemv_fp8_f32(const uint8_t *W, const float *s, const float *x, int M, int K, float *y) {
  e4m3_init();
  gemv_fp8_f32(W, s, x, M, K, y);
}
void orc_topk_softmax_f64(const double *r, int n, int top_k, int *idx, double *w) { topk_softmax_f64(r, n, top_k, idx, w); }
