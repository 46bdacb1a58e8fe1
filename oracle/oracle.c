/*
 * CPU oracle for one decode step of the parallel-layer MoE model.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg, never by the product path.  It shares
 * no code with the CUDA path.  Plain loops, fp64 arithmetic, OpenMP only over
 * independent output rows / heads (no blocking, fusion or reordering of any
 * sum beyond the definition).
 *
 * Definition followed ("Inside the megakernel serving engine for North Mini
 * Code"): §Where the speedup comes from, item 1 (parallel transformer layer:
 * attention and the MoE feed-forward both read one normalised input and are
 * rejoined by a fused residual add + RMSNorm); §Tasks (QKV with RoPE,
 * attention over the paged KV cache, O-proj, router scoring of the experts,
 * top-k per token, expert gate/up with SiLU-and-multiply, expert down, the
 * router-weighted sum of each token's expert outputs, LM head).
 *
 * Readings where the pages are silent:
 *   pre-norm parallel layer  h' = h + Attn(x) + MoE(x),  x = RMSNorm(h; g_l);
 *   a final RMSNorm with its own gain before the LM head;
 *   RMSNorm(h) = h / sqrt(mean(h^2) + eps) * g;
 *   RoPE rotates pairs (i, i + d/2) by pos * theta^(-2i/d);
 *   the new token sits at 0-based position seq_len and attends to itself;
 *   attention scale 1/sqrt(d), softmax over all cached keys;
 *   routing: softmax over all experts, keep the top-k, renormalise over them;
 *   the top-k order is decided on the fp32-rounded logits (the precision the
 *   device computes them in), larger first, equal values -> lower index;
 *   no shared expert, no biases, no QK-norm.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ BF16 */

double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round to BF16 through fp32: the C cast rounds fp64 -> fp32 to nearest even,
 * then the low 16 bits are rounded to nearest even (the usual bias trick). */
uint16_t orc_double_to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

double orc_round_bf16(double x) { return orc_bf16_to_double(orc_double_to_bf16(x)); }

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

/* ------------------------------------------------------------- RMSNorm
 * §Tasks / Fig 4 (residual add + RMSNorm): out_i = h_i / sqrt(mean(h^2)+eps) * g_i */
void orc_rmsnorm(int n, const double* h, const uint16_t* gain, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; i++) ss += h[i] * h[i];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; i++) out[i] = h[i] * r * orc_bf16_to_double(gain[i]);
}

/* ---------------------------------------------------------------- RoPE
 * §Tasks, QKV_PROJ applies RoPE: pair (i, i + d/2) rotated by angle
 * pos * theta^(-2i/d). */
void orc_rope(int d, double* v, long pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; i++) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    double x1 = v[i], x2 = v[i + half];
    v[i] = x1 * c - x2 * s;
    v[i + half] = x2 * c + x1 * s;
  }
}

/* ------------------------------------------------------------- mat-vec
 * y[j][r] = sum_c w[r][c] * x[j][c] for nvec vectors (one weight read). */
void orc_matvec(int rows, int cols, const uint16_t* w, int nvec, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; r++) {
    const uint16_t* wr = w + (size_t)r * cols;
    for (int j = 0; j < nvec; j++) {
      const double* xj = x + (size_t)j * cols;
      double acc = 0.0;
      for (int c = 0; c < cols; c++) acc += orc_bf16_to_double(wr[c]) * xj[c];
      y[(size_t)j * rows + r] = acc;
    }
  }
}

/* ------------------------------------------------------------- E4M3
 * The OCP 8-bit floating point specification, E4M3: sign bit 7, exponent
 * bits 6..3 with bias 7, mantissa bits 2..0.  Exponent field 0 holds the
 * subnormals (m / 8) * 2^-6; the encoding has no infinities and uses
 * S.1111.111 for NaN, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_double(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* The dequantised row w[c] = scale[r] * e4m3(q[r][c]) (exact in fp64), then
 * the same sum as orc_matvec. */
void orc_matvec_e4m3(int rows, int cols, const uint8_t* q, const float* scale, const double* x,
                     double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; r++) {
    const uint8_t* qr = q + (size_t)r * cols;
    const double s = (double)scale[r];
    double acc = 0.0;
    for (int c = 0; c < cols; c++) acc += (s * orc_e4m3_to_double(qr[c])) * x[c];
    y[r] = acc;
  }
}

/* --------------------------------------------------- paged attention
 * §Tasks, ATTN_DECODE / Fig 2 (paged attention): one query head against the
 * n_keys cached keys of its KV head, key p read at physical page
 * page_table[p / P], slot p % P.  out = sum_p softmax_p(q.k_p / sqrt(d)) v_p. */
int orc_paged_attention(const orc_dims* dm, const uint16_t* k_pool, const uint16_t* v_pool,
                        const int32_t* page_table, int n_keys, int kv_head,
                        const double* q, double* out) {
  const int d = dm->head_dim, P = dm->page_size, hkv = dm->n_kv_heads;
  if (n_keys <= 0) return ORC_ERR_ARG;
  double* s = (double*)malloc(sizeof(double) * (size_t)n_keys);
  if (!s) return ORC_ERR_NOMEM;
  const double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int p = 0; p < n_keys; p++) {
    int32_t pg = page_table[p / P];
    if (pg < 0 || pg >= dm->num_pages) { free(s); return ORC_ERR_PAGE; }
    const uint16_t* k = k_pool + (((size_t)pg * hkv + kv_head) * P + (p % P)) * d;
    double dot = 0.0;
    for (int i = 0; i < d; i++) dot += q[i] * orc_bf16_to_double(k[i]);
    s[p] = dot * scale;
    if (s[p] > mx) mx = s[p];
  }
  double den = 0.0;
  for (int p = 0; p < n_keys; p++) { s[p] = exp(s[p] - mx); den += s[p]; }
  for (int i = 0; i < d; i++) out[i] = 0.0;
  for (int p = 0; p < n_keys; p++) {
    int32_t pg = page_table[p / P];
    const uint16_t* v = v_pool + (((size_t)pg * hkv + kv_head) * P + (p % P)) * d;
    double wgt = s[p] / den;
    for (int i = 0; i < d; i++) out[i] += wgt * orc_bf16_to_double(v[i]);
  }
  free(s);
  return ORC_OK;
}

/* ------------------------------------------------------------- routing
 * §Tasks, ROUTER_GEMM / ROUTER_TOPK: score the experts, keep the top-k per
 * token; routing weights = softmax over all experts, renormalised over the
 * kept ones. */
void orc_route(int n_experts, int top_k, const double* logits, int32_t* idx, double* w,
               double* gap) {
  float r32[1024];
  int E = n_experts;
  for (int e = 0; e < E; e++) r32[e] = (float)logits[e];
  unsigned char used[1024];
  memset(used, 0, sizeof(used));
  for (int j = 0; j < top_k; j++) {
    int best = -1;
    for (int e = 0; e < E; e++) {
      if (used[e]) continue;
      if (best < 0 || r32[e] > r32[best]) best = e;   /* strict: ties keep the lower index */
    }
    used[best] = 1;
    idx[j] = best;
  }
  if (gap) {
    int nxt = -1;
    for (int e = 0; e < E; e++)
      if (!used[e] && (nxt < 0 || r32[e] > r32[nxt])) nxt = e;
    *gap = nxt < 0 ? INFINITY : (double)r32[idx[top_k - 1]] - (double)r32[nxt];
  }
  double mx = -INFINITY;
  for (int e = 0; e < E; e++) if (logits[e] > mx) mx = logits[e];
  double den = 0.0;
  for (int e = 0; e < E; e++) den += exp(logits[e] - mx);
  double sel = 0.0;
  for (int j = 0; j < top_k; j++) {
    w[j] = exp(logits[idx[j]] - mx) / den;
    sel += w[j];
  }
  for (int j = 0; j < top_k; j++) w[j] /= sel;
}

/* ----------------------------------------------------------------- MoE
 * §Tasks, MOE_UPGATE_ACT / MOE_DOWN / MOE_COMBINE: for each kept expert e,
 * a = SiLU(W_g^e x) * (W_u^e x), y = W_d^e a; out = sum_j w_j y_j. */
void orc_moe(const orc_dims* dm, const orc_model* m, int layer, const double* x, int n_sel,
             const int32_t* idx, const double* w, unsigned flags, double* out) {
  const int H = dm->hidden, I = dm->moe_inter;
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int i = 0; i < H; i++) out[i] = 0.0;
  for (int j = 0; j < n_sel; j++) {
    int e = idx[j];
    const orc_fp8_experts* f = m->fp8;
    if (f) {
      orc_matvec_e4m3(I, H, f->q_gate[layer] + (size_t)e * I * H, f->s_gate[layer] + (size_t)e * I, x, g);
      orc_matvec_e4m3(I, H, f->q_up[layer] + (size_t)e * I * H, f->s_up[layer] + (size_t)e * I, x, u);
    } else {
      orc_matvec(I, H, m->w_gate[layer] + (size_t)e * I * H, 1, x, g);
      orc_matvec(I, H, m->w_up[layer] + (size_t)e * I * H, 1, x, u);
    }
    for (int i = 0; i < I; i++) {
      double silu = g[i] / (1.0 + exp(-g[i]));
      g[i] = silu * u[i];
      if (flags & ORC_BF16_A) g[i] = orc_round_bf16(g[i]);
    }
    if (f) orc_matvec_e4m3(H, I, f->q_down[layer] + (size_t)e * H * I, f->s_down[layer] + (size_t)e * H, g, y);
    else orc_matvec(H, I, m->w_down[layer] + (size_t)e * H * I, 1, g, y);
    for (int i = 0; i < H; i++) out[i] += w[j] * y[i];
  }
  free(g); free(u); free(y);
}

/* ----------------------------------------------------- one layer, batch */
typedef struct { double *x, *qkv, *att, *ap, *rl, *mo, *wt; int32_t* idx; } layer_bufs;

/* Routing imposed from outside (for comparing with an implementation that
 * decided a near tie the other way): where force[l * B + b] is set, token b
 * of layer l uses the experts force_idx[(l * B + b) * k + j] instead of its
 * own top-k, with the routing weights renormalised over them as usual. */
typedef struct { const int32_t* idx; const uint8_t* mask; } orc_force;

static int layer_body(const orc_dims* dm, const orc_model* m, int l, int B,
                      const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                      unsigned flags, double* h, orc_trace* tr, const layer_bufs* bf,
                      const orc_force* fr) {
  const int H = dm->hidden, hq = dm->n_q_heads, hkv = dm->n_kv_heads, d = dm->head_dim;
  const int E = dm->n_experts, K = dm->top_k, P = dm->page_size, L = dm->n_layers;
  const int QD = hq * d, R = (hq + 2 * hkv) * d, grp = hq / hkv;
  double *x = bf->x, *qkv = bf->qkv, *att = bf->att, *ap = bf->ap, *rl = bf->rl, *mo = bf->mo;
  double* wt = bf->wt;
  int32_t* idx = bf->idx;

  if (tr && tr->h_in) memcpy(tr->h_in + (size_t)l * B * H, h, sizeof(double) * (size_t)B * H);
  /* x = RMSNorm(h; g_l) */
  for (int b = 0; b < B; b++) {
    orc_rmsnorm(H, h + (size_t)b * H, m->attn_norm[l], dm->rms_eps, x + (size_t)b * H);
    if (flags & ORC_BF16_X)
      for (int i = 0; i < H; i++) x[(size_t)b * H + i] = orc_round_bf16(x[(size_t)b * H + i]);
  }
  if (tr && tr->x) memcpy(tr->x + (size_t)l * B * H, x, sizeof(double) * (size_t)B * H);

  /* [q; k; v] = W_qkv x, RoPE on q and k at the token's position, append k, v */
  orc_matvec(R, H, m->w_qkv[l], B, x, qkv);
  for (int b = 0; b < B; b++) {
    double* q = qkv + (size_t)b * R;
    double* k = q + QD;
    double* v = k + hkv * d;
    long pos = seq_lens[b];
    for (int hh = 0; hh < hq; hh++) {
      orc_rope(d, q + (size_t)hh * d, pos, dm->rope_theta);
      if (flags & ORC_BF16_Q)
        for (int i = 0; i < d; i++) q[hh * d + i] = orc_round_bf16(q[hh * d + i]);
    }
    for (int g = 0; g < hkv; g++) orc_rope(d, k + (size_t)g * d, pos, dm->rope_theta);
    int pidx = (int)(pos / P);
    if (pidx >= max_pages) return ORC_ERR_PAGE;
    int32_t pg = page_tables[(size_t)b * max_pages + pidx];
    if (pg < 0 || pg >= dm->num_pages) return ORC_ERR_PAGE;
    for (int g = 0; g < hkv; g++) {
      size_t off = (((size_t)pg * hkv + g) * P + (pos % P)) * d;
      for (int i = 0; i < d; i++) {
        m->k_pool[l][off + i] = orc_double_to_bf16(k[g * d + i]);
        m->v_pool[l][off + i] = orc_double_to_bf16(v[g * d + i]);
      }
    }
    if (tr && tr->q) memcpy(tr->q + ((size_t)l * B + b) * QD, q, sizeof(double) * QD);
  }

  /* attention: every query head over its KV head's seq_len + 1 keys */
  {
    int err = ORC_OK;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; b++)
      for (int hh = 0; hh < hq; hh++) {
        const double* q = qkv + (size_t)b * R + (size_t)hh * d;
        double* o = att + (size_t)b * QD + (size_t)hh * d;
        int e2 = orc_paged_attention(dm, m->k_pool[l], m->v_pool[l],
                                     page_tables + (size_t)b * max_pages, seq_lens[b] + 1,
                                     hh / grp, q, o);
        if (e2 != ORC_OK) {
#pragma omp critical
          err = e2;
        }
        if (flags & ORC_BF16_ATTN)
          for (int i = 0; i < d; i++) o[i] = orc_round_bf16(o[i]);
      }
    if (err != ORC_OK) return err;
  }
  if (tr && tr->attn) memcpy(tr->attn + (size_t)l * B * QD, att, sizeof(double) * (size_t)B * QD);

  /* O-proj */
  orc_matvec(H, QD, m->w_o[l], B, att, ap);
  if (tr && tr->attn_proj) memcpy(tr->attn_proj + (size_t)l * B * H, ap, sizeof(double) * (size_t)B * H);

  /* router, top-k, experts */
  orc_matvec(E, H, m->w_router[l], B, x, rl);
  for (int b = 0; b < B; b++) {
    double gap;
    orc_route(E, K, rl + (size_t)b * E, idx + (size_t)b * K, wt + (size_t)b * K, &gap);
    if (tr && tr->gap) tr->gap[(size_t)l * B + b] = gap;
    if (fr && fr->mask[(size_t)l * B + b]) {
      /* the imposed experts; weights p_j / sum of p over them, p = softmax of
       * the logits (the same operations as orc_route's) */
      const double* r = rl + (size_t)b * E;
      const int32_t* fi = fr->idx + ((size_t)l * B + b) * K;
      double mx = -INFINITY, den = 0.0, sel = 0.0;
      for (int e = 0; e < E; e++) if (r[e] > mx) mx = r[e];
      for (int e = 0; e < E; e++) den += exp(r[e] - mx);
      for (int j = 0; j < K; j++) {
        if (fi[j] < 0 || fi[j] >= E) return ORC_ERR_ARG;
        idx[(size_t)b * K + j] = fi[j];
        wt[(size_t)b * K + j] = exp(r[fi[j]] - mx) / den;
        sel += wt[(size_t)b * K + j];
      }
      for (int j = 0; j < K; j++) wt[(size_t)b * K + j] /= sel;
    }
    orc_moe(dm, m, l, x + (size_t)b * H, K, idx + (size_t)b * K, wt + (size_t)b * K, flags,
            mo + (size_t)b * H);
  }
  if (tr && tr->router) memcpy(tr->router + (size_t)l * B * E, rl, sizeof(double) * (size_t)B * E);
  if (tr && tr->idx) memcpy(tr->idx + (size_t)l * B * K, idx, sizeof(int32_t) * (size_t)B * K);
  if (tr && tr->w) memcpy(tr->w + (size_t)l * B * K, wt, sizeof(double) * (size_t)B * K);
  if (tr && tr->moe) memcpy(tr->moe + (size_t)l * B * H, mo, sizeof(double) * (size_t)B * H);

  /* parallel residual: h = h + attn_proj + moe */
  for (size_t i = 0; i < (size_t)B * H; i++) h[i] = h[i] + ap[i] + mo[i];
  if (tr && tr->h_in && l == L - 1) memcpy(tr->h_in + (size_t)L * B * H, h, sizeof(double) * (size_t)B * H);

  return ORC_OK;
}

static int layer_forward(const orc_dims* dm, const orc_model* m, int l, int B,
                         const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                         unsigned flags, double* h, orc_trace* tr, const orc_force* fr) {
  const int H = dm->hidden, QD = dm->n_q_heads * dm->head_dim;
  const int R = (dm->n_q_heads + 2 * dm->n_kv_heads) * dm->head_dim;
  layer_bufs bf;
  bf.x = (double*)malloc(sizeof(double) * (size_t)B * H);
  bf.qkv = (double*)malloc(sizeof(double) * (size_t)B * R);
  bf.att = (double*)malloc(sizeof(double) * (size_t)B * QD);
  bf.ap = (double*)malloc(sizeof(double) * (size_t)B * H);
  bf.rl = (double*)malloc(sizeof(double) * (size_t)B * dm->n_experts);
  bf.mo = (double*)malloc(sizeof(double) * (size_t)B * H);
  bf.idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)B * dm->top_k);
  bf.wt = (double*)malloc(sizeof(double) * (size_t)B * dm->top_k);
  int rc = ORC_ERR_NOMEM;
  if (bf.x && bf.qkv && bf.att && bf.ap && bf.rl && bf.mo && bf.idx && bf.wt)
    rc = layer_body(dm, m, l, B, seq_lens, page_tables, max_pages, flags, h, tr, &bf, fr);
  free(bf.x); free(bf.qkv); free(bf.att); free(bf.ap); free(bf.rl); free(bf.mo);
  free(bf.idx); free(bf.wt);
  return rc;
}

static int check_dims(const orc_dims* dm) {
  if (!dm || dm->n_layers <= 0 || dm->hidden <= 0 || dm->n_q_heads <= 0 || dm->n_kv_heads <= 0 ||
      dm->n_q_heads % dm->n_kv_heads || dm->head_dim <= 0 || dm->head_dim % 2 ||
      dm->n_experts <= 0 || dm->n_experts > 1024 || dm->top_k <= 0 ||
      dm->top_k > dm->n_experts || dm->moe_inter <= 0 || dm->vocab <= 0 ||
      dm->page_size <= 0 || dm->num_pages <= 0)
    return ORC_ERR_ARG;
  return ORC_OK;
}

int orc_run_layers(const orc_dims* dm, const orc_model* m, int l0, int l1, int batch,
                   const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                   unsigned flags, double* h) {
  if (check_dims(dm) != ORC_OK || batch <= 0 || l0 < 0 || l1 > dm->n_layers) return ORC_ERR_ARG;
  for (int l = l0; l < l1; l++) {
    int rc = layer_forward(dm, m, l, batch, seq_lens, page_tables, max_pages, flags, h, NULL, NULL);
    if (rc != ORC_OK) return rc;
  }
  return ORC_OK;
}

/* -------------------------------------------------- one decode step
 * h = embed[token]; for every layer the parallel block above; then
 * logits = W_lm RMSNorm(h; g_f). */
int orc_decode_step_forced(const orc_dims* dm, const orc_model* m, int batch, const int32_t* tokens,
                           const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                           unsigned flags, const int32_t* force_idx, const uint8_t* force_mask,
                           double* logits, orc_trace* trace) {
  if (check_dims(dm) != ORC_OK || batch <= 0) return ORC_ERR_ARG;
  if ((force_idx == NULL) != (force_mask == NULL)) return ORC_ERR_ARG;
  orc_force fr = {force_idx, force_mask};
  const orc_force* frp = force_idx ? &fr : NULL;
  const int H = dm->hidden, V = dm->vocab;
  double* h = (double*)malloc(sizeof(double) * (size_t)batch * H);
  double* xf = (double*)malloc(sizeof(double) * (size_t)batch * H);
  if (!h || !xf) { free(h); free(xf); return ORC_ERR_NOMEM; }
  int rc = ORC_OK;
  for (int b = 0; b < batch; b++) {
    if (tokens[b] < 0 || tokens[b] >= V) { rc = ORC_ERR_ARG; goto out; }
    const uint16_t* er = m->embed + (size_t)tokens[b] * H;
    for (int i = 0; i < H; i++) h[(size_t)b * H + i] = orc_bf16_to_double(er[i]);
  }
  for (int l = 0; l < dm->n_layers; l++) {
    rc = layer_forward(dm, m, l, batch, seq_lens, page_tables, max_pages, flags, h, trace, frp);
    if (rc != ORC_OK) goto out;
  }
  for (int b = 0; b < batch; b++) {
    orc_rmsnorm(H, h + (size_t)b * H, m->final_norm, dm->rms_eps, xf + (size_t)b * H);
    if (flags & ORC_BF16_X)
      for (int i = 0; i < H; i++) xf[(size_t)b * H + i] = orc_round_bf16(xf[(size_t)b * H + i]);
  }
  if (trace && trace->xf) memcpy(trace->xf, xf, sizeof(double) * (size_t)batch * H);
  orc_matvec(V, H, m->lm_head, batch, xf, logits);
out:
  free(h); free(xf);
  return rc;
}

int orc_decode_step(const orc_dims* dm, const orc_model* m, int batch, const int32_t* tokens,
                    const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                    unsigned flags, double* logits, orc_trace* trace) {
  return orc_decode_step_forced(dm, m, batch, tokens, seq_lens, page_tables, max_pages, flags, NULL, NULL,
                                logits, trace);
}
