/*
 * Body of the CPU oracle, compiled twice by oracle.c: once with REAL = float (the reference precision:
 * fp16 weights and KV cache, fp32 arithmetic) and once with REAL = double (to bound the fp32 version's
 * own rounding). Every loop is the plain definition, summed in index order.
 *
 * Expects from the includer: REAL, NAME(x), SQRT(x), EXP(x).
 */

/* u = x / sqrt(mean(x^2) + eps) * g  (RMSNorm; the gain g is fp16). */
static void NAME(rmsnorm)(const REAL *x, const uint16_t *g, int n, REAL eps, REAL *out) {
  REAL ss = 0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  REAL denom = SQRT(ss / (REAL)n + eps);
  for (int i = 0; i < n; ++i) out[i] = (x[i] / denom) * (REAL)half_value(g[i]);
}

/* y = W x with W [M, K] row-major fp16, each row summed sequentially over k. */
static void NAME(gemv)(const uint16_t *W, const REAL *x, int M, int K, REAL *y) {
#pragma omp parallel for schedule(static) if (M >= 256)
  for (int r = 0; r < M; ++r) {
    const uint16_t *w = W + (size_t)r * K;
    REAL acc = 0;
    for (int k = 0; k < K; ++k) acc += (REAL)half_value(w[k]) * x[k];
    y[r] = acc;
  }
}

/* Rotary embedding, "rotate-half" pairing: dimension i is paired with i + dh/2 (i < dh/2), rotated by
 * the angle pos * theta^(-2i/dh). The angle and its cosine and sine are evaluated in fp64. */
static void NAME(rope)(REAL *v, int dh, int pos, double theta) {
  int half = dh / 2;
  for (int i = 0; i < half; ++i) {
    double angle = (double)pos * pow(theta, -2.0 * (double)i / (double)dh);
    REAL c = (REAL)cos(angle), s = (REAL)sin(angle);
    REAL a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* One attention head over c cached positions: s_j = q . K[j] / sqrt(dh); p = softmax(s) with the maximum
 * subtracted; out = sum_j p_j V[j]. K and V are fp16 rows of length dh, `stride` elements apart. */
static void NAME(attention)(const REAL *q, const uint16_t *K, const uint16_t *V, int c, int dh, size_t stride,
                            REAL *scores, REAL *out) {
  REAL root = SQRT((REAL)dh);
  for (int j = 0; j < c; ++j) {
    const uint16_t *k = K + (size_t)j * stride;
    REAL dot = 0;
    for (int e = 0; e < dh; ++e) dot += q[e] * (REAL)half_value(k[e]);
    scores[j] = dot / root;
  }
  REAL m = scores[0];
  for (int j = 1; j < c; ++j)
    if (scores[j] > m) m = scores[j];
  REAL l = 0;
  for (int j = 0; j < c; ++j) {
    scores[j] = EXP(scores[j] - m);
    l += scores[j];
  }
  for (int e = 0; e < dh; ++e) out[e] = 0;
  for (int j = 0; j < c; ++j) {
    REAL p = scores[j] / l;
    const uint16_t *v = V + (size_t)j * stride;
    for (int e = 0; e < dh; ++e) out[e] += p * (REAL)half_value(v[e]);
  }
}

/* silu(z) = z / (1 + exp(-z)). */
static REAL NAME(silu)(REAL z) { return z / ((REAL)1 + EXP(-z)); }

/* y = dequant(W) x for E4M3 codes W [M][K] with row scales s [M]: y_r = s_r * sum_k E4M3(W_rk) x_k, in order. */
static void NAME(gemv_fp8)(const uint8_t *W, const float *s, const REAL *x, int M, int K, REAL *y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < M; ++r) {
    const uint8_t *row = W + (size_t)r * K;
    REAL acc = 0;
    for (int k = 0; k < K; ++k) acc += (REAL)e4m3_table[row[k]] * x[k];
    y[r] = (REAL)s[r] * acc;
  }
}

/* The top_k largest of r[0..n) (the lowest index first among equal values), in descending order, and the
 * softmax over the selected values (max-subtracted). */
static void NAME(topk_softmax)(const REAL *r, int n, int top_k, int *idx, REAL *w) {
  for (int j = 0; j < top_k; ++j) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
      int taken = 0;
      for (int i = 0; i < j; ++i) taken |= idx[i] == e;
      if (!taken && (best < 0 || r[e] > r[best])) best = e;
    }
    idx[j] = best;
  }
  REAL mx = r[idx[0]], sum = 0;
  for (int j = 1; j < top_k; ++j) mx = r[idx[j]] > mx ? r[idx[j]] : mx;
  for (int j = 0; j < top_k; ++j) {
    w[j] = EXP(r[idx[j]] - mx);
    sum += w[j];
  }
  for (int j = 0; j < top_k; ++j) w[j] /= sum;
}

/* The sparse-MoE FFN of layer l on the normalised input u: out = sum_{e in top_k} w_e Wd_e (silu(Wg_e u) *
 * (Wu_e u)), the experts taken in the order topk_softmax returns them. */
static void NAME(moe_ffn)(orc_model *m, int l, const REAL *u, REAL *out) {
  const orc_moe *mo = &m->moe;
  const int d = m->cfg.d_model, Fe = mo->expert_ffn, E = mo->n_experts;
  REAL *rl = (REAL *)m->rl, *g = (REAL *)m->g, *up = (REAL *)m->up, *t = (REAL *)m->t;
  int idx[1024];
  REAL w[1024];
  NAME(gemv)(mo->router[l], u, E, d, rl);
  NAME(topk_softmax)(rl, E, mo->top_k, idx, w);
  {
    double best_out = -INFINITY;
    for (int e = 0; e < E; ++e) {
      int taken = 0;
      for (int j = 0; j < mo->top_k; ++j) taken |= idx[j] == e;
      if (!taken && (double)rl[e] > best_out) best_out = (double)rl[e];
    }
    const double gap = (double)rl[idx[mo->top_k - 1]] - best_out;
    if (gap < m->route_margin) m->route_margin = gap;
    m->route_gap[l] = gap;
    for (int j = 0; j < mo->top_k; ++j) m->route_ids[(size_t)l * mo->top_k + j] = idx[j];
  }
  for (int i = 0; i < d; ++i) out[i] = 0;
  for (int j = 0; j < mo->top_k; ++j) {
    const int e = idx[j];
    NAME(gemv_fp8)(mo->gate_q[l] + (size_t)e * Fe * d, mo->gate_s[l] + (size_t)e * Fe, u, Fe, d, g);
    NAME(gemv_fp8)(mo->up_q[l] + (size_t)e * Fe * d, mo->up_s[l] + (size_t)e * Fe, u, Fe, d, up);
    for (int i = 0; i < Fe; ++i) g[i] = NAME(silu)(g[i]) * up[i];
    NAME(gemv_fp8)(mo->down_q[l] + (size_t)e * d * Fe, mo->down_s[l] + (size_t)e * d, g, d, Fe, t);
    for (int i = 0; i < d; ++i) out[i] += w[j] * t[i];
  }
}

/* One decoder forward of `token` at position m->pos: appends K and V (rounded to fp16) to the cache,
 * writes the logits of the next position (skipped when logits is NULL: a prompt position whose logits are not
 * wanted), advances pos. */
static void NAME(forward)(orc_model *m, int token, REAL *logits) {
  const orc_config *c = &m->cfg;
  const int d = c->d_model, Hq = c->n_heads, Hkv = c->n_kv_heads, dh = c->head_dim, F = c->ffn_dim;
  const int group = Hq / Hkv, pos = m->pos;
  const size_t S = (size_t)c->max_seq * dh; /* elements per [layer][k|v][kv-head] plane */
  REAL *x = (REAL *)m->x, *u = (REAL *)m->u, *q = (REAL *)m->q, *k = (REAL *)m->k, *v = (REAL *)m->v;
  REAL *o = (REAL *)m->o, *t = (REAL *)m->t, *g = (REAL *)m->g, *up = (REAL *)m->up, *sc = (REAL *)m->scores;

  for (int i = 0; i < d; ++i) x[i] = (REAL)half_value(m->w.embed[(size_t)token * d + i]);

  for (int l = 0; l < c->n_layers; ++l) {
    NAME(rmsnorm)(x, m->w.attn_norm[l], d, (REAL)c->rms_eps, u);
    NAME(gemv)(m->w.wq[l], u, Hq * dh, d, q);
    NAME(gemv)(m->w.wk[l], u, Hkv * dh, d, k);
    NAME(gemv)(m->w.wv[l], u, Hkv * dh, d, v);
    for (int h = 0; h < Hq; ++h) NAME(rope)(q + h * dh, dh, pos, c->rope_theta);
    for (int h = 0; h < Hkv; ++h) NAME(rope)(k + h * dh, dh, pos, c->rope_theta);

    uint16_t *Kl = m->kv + (size_t)l * 2 * Hkv * S, *Vl = Kl + (size_t)Hkv * S;
    for (int h = 0; h < Hkv; ++h)
      for (int e = 0; e < dh; ++e) {
        Kl[h * S + (size_t)pos * dh + e] = half_bits((double)k[h * dh + e]);
        Vl[h * S + (size_t)pos * dh + e] = half_bits((double)v[h * dh + e]);
      }
    /* heads are independent: each gets its own score row, so running them on several threads changes no sum */
#pragma omp parallel for schedule(static) if (pos >= 255)
    for (int h = 0; h < Hq; ++h) {
      int kvh = h / group;
      NAME(attention)(q + h * dh, Kl + kvh * S, Vl + kvh * S, pos + 1, dh, (size_t)dh, sc + (size_t)h * c->max_seq,
                      o + h * dh);
    }
    NAME(gemv)(m->w.wo[l], o, d, Hq * dh, t);
    for (int i = 0; i < d; ++i) x[i] += t[i];

    NAME(rmsnorm)(x, m->w.ffn_norm[l], d, (REAL)c->rms_eps, u);
    if (m->moe.n_experts > 0) {
      REAL *acc = (REAL *)m->acc;
      NAME(moe_ffn)(m, l, u, acc);
      for (int i = 0; i < d; ++i) x[i] += acc[i];
      continue;
    }
    NAME(gemv)(m->w.w_gate[l], u, F, d, g);
    NAME(gemv)(m->w.w_up[l], u, F, d, up);
    for (int i = 0; i < F; ++i) g[i] = NAME(silu)(g[i]) * up[i];
    NAME(gemv)(m->w.w_down[l], g, d, F, t);
    for (int i = 0; i < d; ++i) x[i] += t[i];
  }
  if (logits) {
    NAME(rmsnorm)(x, m->w.final_norm, d, (REAL)c->rms_eps, u);
    NAME(gemv)(m->w.lm_head, u, c->vocab, d, logits);
  }
  m->pos = pos + 1;
}
