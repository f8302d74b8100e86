/*
 * oracle.c -- plain CPU reference of one low-batch transformer decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by tests/, by
 * __graft_entry__.smoke() and by the cpu_baseline / reference leg of
 * bench.py; never by the product path.  Shares nothing with the CUDA path.
 *
 * Each function names the passage it restates.  Page titles:
 *   [MK]  "Megakernels: Deleting the Kernel Boundary to Win Back Microseconds"
 *   [G4]  "Gemma 4 TPU megakernel" (withhopper.com)
 * Where the pages name an operation without defining it (RMSNorm, RoPE,
 * SiLU, softmax attention, top-k routing) the textbook definition is used;
 * the chosen readings are listed at the top of each function.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 0; /* 0: OpenMP default */

void orc_set_threads(int n) { g_threads = n; }

int orc_get_threads(void) {
#ifdef _OPENMP
  return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
  return 1;
#endif
}

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even,
 * in one rounding step.  Normal range: scale the significand to [128,256)
 * and round it to an integer; subnormal range: quantum 2^-133.          */
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  double ax = fabs(x);
  double r;
  if (ax < ldexp(1.0, -126)) {
    r = nearbyint(ldexp(ax, 133)); /* default rounding mode: ties to even */
    r = ldexp(r, -133);
  } else {
    int e;
    double m = frexp(ax, &e);   /* ax = m * 2^e, m in [0.5, 1) */
    double q = nearbyint(ldexp(m, 8)); /* in [128, 256] */
    r = ldexp(q, e - 8);
  }
  float f;
  if (r >= ldexp(1.0, 128)) {
    f = INFINITY;
  } else {
    f = (float)r; /* exact: r has at most 8 significant bits */
  }
  if (signbit(x)) f = -f;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* [MK] "Where the microseconds go": "RMS norm".  Reading: the usual
 * RMSNorm, x / sqrt(mean(x^2) + eps) times a per-channel gain.          */
void orc_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; i++) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; i++) out[i] = x[i] * inv * orc_bf16_to_f64(gain[i]);
}

/* [MK] "Where the microseconds go": "RoPE".  Reading: rotate-half pairing,
 * element i is rotated with element i + d/2 by the angle pos * theta^(-2i/d);
 * no frequency scaling.                                                 */
void orc_rope(double* v, int d, int pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; i++) {
    double freq = pow(theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = a * s + b * c;
  }
}

/* Matrix-vector product (the "matvec" of [MK] "What it buys"). */
void orc_gemv(const uint16_t* W, int rows, int cols, const double* x, double* y) {
  int nt = orc_get_threads();
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int r = 0; r < rows; r++) {
    const uint16_t* w = W + (size_t)r * (size_t)cols;
    double acc = 0.0;
    for (int k = 0; k < cols; k++) acc += orc_bf16_to_f64(w[k]) * x[k];
    y[r] = acc;
  }
}

/* Per-row int8 quantisation ([G4] "What's next": INT8 weights).  Reading:
 * one symmetric scale per output row, the largest magnitude mapped to 127,
 * round half to even. */
void orc_quantize_rows_int8(const uint16_t* W, int rows, int cols, int8_t* codes, float* scales) {
  for (int r = 0; r < rows; r++) {
    const uint16_t* w = W + (size_t)r * (size_t)cols;
    float m = 0.0f;
    for (int k = 0; k < cols; k++) {
      float a = fabsf((float)orc_bf16_to_f64(w[k]));
      if (a > m) m = a;
    }
    float s = m > 0.0f ? m / 127.0f : 0.0f;
    for (int k = 0; k < cols; k++) {
      long q = 0;
      if (s > 0.0f) {
        float t = (float)orc_bf16_to_f64(w[k]) / s;
        q = lrintf(t); /* the default rounding mode: nearest, ties to even */
        if (q > 127) q = 127;
        if (q < -127) q = -127;
      }
      codes[(size_t)r * (size_t)cols + k] = (int8_t)q;
    }
    scales[r] = s;
  }
}

void orc_gemv_q8(const int8_t* codes, const float* scales, int rows, int cols, const double* x,
                 double* y) {
  int nt = orc_get_threads();
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int r = 0; r < rows; r++) {
    const int8_t* q = codes + (size_t)r * (size_t)cols;
    const double s = (double)scales[r];
    double acc = 0.0;
    for (int k = 0; k < cols; k++) acc += ((double)q[k] * s) * x[k];
    y[r] = acc;
  }
}

/* [MK] op list "attention": softmax(q K^T / sqrt(d)) V over the cached rows. */
void orc_attention(const double* q, const uint16_t* K, const uint16_t* V, int n_pos, int d,
                   double* out) {
  double scale = 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_pos > 0 ? n_pos : 1));
  double mx = -INFINITY;
  for (int j = 0; j < n_pos; j++) {
    double acc = 0.0;
    for (int t = 0; t < d; t++) acc += q[t] * orc_bf16_to_f64(K[(size_t)j * d + t]);
    s[j] = acc * scale;
    if (s[j] > mx) mx = s[j];
  }
  double sum = 0.0;
  for (int j = 0; j < n_pos; j++) {
    s[j] = exp(s[j] - mx);
    sum += s[j];
  }
  for (int t = 0; t < d; t++) out[t] = 0.0;
  for (int j = 0; j < n_pos; j++) {
    double a = s[j] / sum;
    for (int t = 0; t < d; t++) out[t] += a * orc_bf16_to_f64(V[(size_t)j * d + t]);
  }
  free(s);
}

/* The partial-softmax state of a contiguous slice of positions, the unit of
 * work of a split-KV attention instruction ([MK] opcode OP_ATTENTION, whose
 * partials OP_ATTN_REDUCE combines).                                     */
void orc_attention_partial(const double* q, const uint16_t* K, const uint16_t* V, int p0,
                           int p1, int d, double* m, double* l, double* o) {
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int t = 0; t < d; t++) o[t] = 0.0;
  *l = 0.0;
  if (p1 <= p0) {
    *m = -INFINITY;
    return;
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)(p1 - p0));
  for (int j = p0; j < p1; j++) {
    double acc = 0.0;
    for (int t = 0; t < d; t++) acc += q[t] * orc_bf16_to_f64(K[(size_t)j * d + t]);
    s[j - p0] = acc * scale;
    if (s[j - p0] > mx) mx = s[j - p0];
  }
  for (int j = p0; j < p1; j++) {
    double e = exp(s[j - p0] - mx);
    *l += e;
    for (int t = 0; t < d; t++) o[t] += e * orc_bf16_to_f64(V[(size_t)j * d + t]);
  }
  *m = mx;
  free(s);
}

/* [MK] opcode OP_ATTN_REDUCE: rescale every partial to the common maximum
 * M = max m_s, then out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.  */
void orc_attention_merge(int n_parts, const double* m, const double* l, const double* o, int d,
                         double* out) {
  double M = -INFINITY;
  for (int s = 0; s < n_parts; s++)
    if (m[s] > M) M = m[s];
  double L = 0.0;
  for (int t = 0; t < d; t++) out[t] = 0.0;
  for (int s = 0; s < n_parts; s++) {
    if (l[s] == 0.0) continue; /* empty slice contributes nothing */
    double f = exp(m[s] - M);
    L += f * l[s];
    for (int t = 0; t < d; t++) out[t] += f * o[(size_t)s * d + t];
  }
  for (int t = 0; t < d; t++) out[t] /= L;
}

/* [MK] "SiLU": a * sigmoid(a). */
double orc_silu(double a) { return a / (1.0 + exp(-a)); }

/* [MK] "up and gate projections, SiLU, down projection"; h (may be NULL)
 * receives silu(Wg xn) * (Wu xn). */
void orc_swiglu_h(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int F, int H,
                  const double* xn, double* y, double* h) {
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);
  orc_gemv(wg, F, H, xn, g);
  orc_gemv(wu, F, H, xn, u);
  for (int c = 0; c < F; c++) g[c] = orc_silu(g[c]) * u[c];
  if (h) memcpy(h, g, sizeof(double) * (size_t)F);
  orc_gemv(wd, H, F, g, y);
  free(g);
  free(u);
}

void orc_swiglu(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int F, int H,
                const double* xn, double* y) {
  orc_swiglu_h(wg, wu, wd, F, H, xn, y, NULL);
}

/* [G4] component "Router".  Reading: softmax over all router logits, the
 * k largest probabilities (lower id wins a tie), renormalised to sum 1.   */
double orc_router_topk(const double* logits, int E, int k, int* ids, double* w) {
  double mx = -INFINITY;
  for (int e = 0; e < E; e++)
    if (logits[e] > mx) mx = logits[e];
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  char* taken = (char*)calloc((size_t)E, 1);
  double z = 0.0;
  for (int e = 0; e < E; e++) {
    p[e] = exp(logits[e] - mx);
    z += p[e];
  }
  for (int e = 0; e < E; e++) p[e] /= z;
  double sel = 0.0;
  for (int j = 0; j < k; j++) {
    int best = -1;
    for (int e = 0; e < E; e++)
      if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
    taken[best] = 1;
    ids[j] = best;
    sel += p[best];
  }
  double margin = 1.0;
  if (k < E) {
    int next = -1;
    for (int e = 0; e < E; e++)
      if (!taken[e] && (next < 0 || p[e] > p[next])) next = e;
    double pk = p[ids[k - 1]];
    margin = (pk - p[next]) / pk;
  }
  for (int j = 0; j < k; j++) w[j] = p[ids[j]] / sel;
  free(p);
  free(taken);
  return margin;
}

int orc_argmax(const double* v, int n) {
  int best = 0;
  for (int i = 1; i < n; i++)
    if (v[i] > v[best]) best = i;
  return best;
}

/* The GEMV of one streamed matrix: bf16 W, or its int8 form m when m is set. */
static void gemv_w(const uint16_t* W, const orc_qmat* m, int rows, int cols, const double* x,
                   double* y) {
  if (m)
    orc_gemv_q8(m->codes, m->scales, rows, cols, x, y);
  else
    orc_gemv(W, rows, cols, x, y);
}

static uint16_t* cache_row(uint16_t* base, const orc_config* c, int b, int g, int pos) {
  size_t idx = (((size_t)b * c->n_kv_heads + g) * (size_t)c->max_seq + (size_t)pos) *
               (size_t)c->head_dim;
  return base + idx;
}

/* One decode step: [MK] "One launch, one interpreter" opcode sequence
 * OP_RMS_QKV_ROPE, OP_ATTENTION/OP_ATTN_REDUCE, OP_O_PROJ_RES,
 * OP_RMS_UP_GATE, OP_DOWN_RES per layer, then OP_RMS_LM_HEAD; the MoE MLP
 * follows [G4] "Megakernels for Gemma 4" (routed experts + shared MLP).
 * Readings: query head h uses kv head h / (n_q_heads / n_kv_heads); the new
 * token attends to rows [0, P] including itself; K and V are appended as
 * bf16 before attention reads them; the shared expert is added unweighted. */
int orc_decode_step(const orc_config* cfg, const orc_weights* w, uint16_t* const* kc,
                    uint16_t* const* vc, int B, const int* tokens, const int* positions,
                    double* logits, int* argmax, int* route_ids, double* route_margin,
                    const int* forced_routes, const int* forced_mask) {
  return orc_decode_step_trace(cfg, w, kc, vc, B, tokens, positions, logits, argmax, route_ids,
                               route_margin, forced_routes, forced_mask, NULL, NULL, NULL);
}

int orc_decode_step_trace(const orc_config* cfg, const orc_weights* w, uint16_t* const* kc,
                          uint16_t* const* vc, int B, const int* tokens, const int* positions,
                          double* logits, int* argmax, int* route_ids, double* route_margin,
                          const int* forced_routes, const int* forced_mask, double* tq,
                          double* tx, double* th) {
  const int H = cfg->hidden, Hq = cfg->n_q_heads, Hkv = cfg->n_kv_heads, d = cfg->head_dim;
  const int L = cfg->n_layers, V = cfg->vocab;
  if (B <= 0 || H <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d % 2) || (Hq % Hkv)) return -1;
  for (int b = 0; b < B; b++) {
    if (tokens[b] < 0 || tokens[b] >= V) return -1;
    if (positions[b] < 0 || positions[b] >= cfg->max_seq) return -1;
  }
  const int group = Hq / Hkv;
  const int moe = cfg->n_experts > 0;
  const orc_q8* q8 = w->q8;
  if (q8 && moe) return -1; /* int8 weights: dense models only */
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* xn = (double*)malloc(sizeof(double) * (size_t)H);
  double* q = (double*)malloc(sizeof(double) * (size_t)Hq * d);
  double* k = (double*)malloc(sizeof(double) * (size_t)Hkv * d);
  double* v = (double*)malloc(sizeof(double) * (size_t)Hkv * d);
  double* att = (double*)malloc(sizeof(double) * (size_t)Hq * d);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  double* y2 = (double*)malloc(sizeof(double) * (size_t)H);
  double* rl = moe ? (double*)malloc(sizeof(double) * (size_t)cfg->n_experts) : NULL;
  int* ids = moe ? (int*)malloc(sizeof(int) * (size_t)cfg->top_k) : NULL;
  double* rw = moe ? (double*)malloc(sizeof(double) * (size_t)cfg->top_k) : NULL;

  for (int b = 0; b < B; b++) {
    const int P = positions[b];
    /* embedding gather */
    const uint16_t* erow = w->embed + (size_t)tokens[b] * H;
    for (int i = 0; i < H; i++) x[i] = orc_bf16_to_f64(erow[i]);

    for (int l = 0; l < L; l++) {
      /* OP_RMS_QKV_ROPE */
      orc_rmsnorm(x, w->attn_norm[l], H, cfg->rms_eps, xn);
      gemv_w(w->wq[l], q8 ? &q8->wq[l] : NULL, Hq * d, H, xn, q);
      gemv_w(w->wk[l], q8 ? &q8->wk[l] : NULL, Hkv * d, H, xn, k);
      gemv_w(w->wv[l], q8 ? &q8->wv[l] : NULL, Hkv * d, H, xn, v);
      for (int h = 0; h < Hq; h++) orc_rope(q + (size_t)h * d, d, P, cfg->rope_theta);
      for (int g = 0; g < Hkv; g++) orc_rope(k + (size_t)g * d, d, P, cfg->rope_theta);
      if (tq) memcpy(tq + ((size_t)l * B + b) * Hq * d, q, sizeof(double) * (size_t)Hq * d);
      for (int g = 0; g < Hkv; g++) {
        uint16_t* kr = cache_row(kc[l], cfg, b, g, P);
        uint16_t* vr = cache_row(vc[l], cfg, b, g, P);
        for (int t = 0; t < d; t++) {
          kr[t] = orc_f64_to_bf16(k[(size_t)g * d + t]);
          vr[t] = orc_f64_to_bf16(v[(size_t)g * d + t]);
        }
      }
      /* OP_ATTENTION + OP_ATTN_REDUCE */
      for (int h = 0; h < Hq; h++) {
        int g = h / group;
        orc_attention(q + (size_t)h * d, cache_row(kc[l], cfg, b, g, 0),
                      cache_row(vc[l], cfg, b, g, 0), P + 1, d, att + (size_t)h * d);
      }
      /* OP_O_PROJ_RES */
      gemv_w(w->wo[l], q8 ? &q8->wo[l] : NULL, H, Hq * d, att, y);
      for (int i = 0; i < H; i++) x[i] += y[i];
      if (tx) memcpy(tx + ((size_t)(2 * l) * B + b) * H, x, sizeof(double) * (size_t)H);
      /* OP_RMS_UP_GATE + OP_DOWN_RES (dense) or router + experts (MoE) */
      orc_rmsnorm(x, w->mlp_norm[l], H, cfg->rms_eps, xn);
      if (!moe && q8) {
        /* the same MLP with the int8 gate, up and down matrices */
        const int F = cfg->ffn;
        double* gq = (double*)malloc(sizeof(double) * (size_t)F);
        double* uq = (double*)malloc(sizeof(double) * (size_t)F);
        gemv_w(NULL, &q8->w_gate[l], F, H, xn, gq);
        gemv_w(NULL, &q8->w_up[l], F, H, xn, uq);
        for (int c = 0; c < F; c++) gq[c] = orc_silu(gq[c]) * uq[c];
        if (th) memcpy(th + ((size_t)l * B + b) * F, gq, sizeof(double) * (size_t)F);
        gemv_w(NULL, &q8->w_down[l], H, F, gq, y);
        free(gq);
        free(uq);
        for (int i = 0; i < H; i++) x[i] += y[i];
      } else if (!moe) {
        orc_swiglu_h(w->w_gate[l], w->w_up[l], w->w_down[l], cfg->ffn, H, xn, y,
                     th ? th + ((size_t)l * B + b) * cfg->ffn : NULL);
        for (int i = 0; i < H; i++) x[i] += y[i];
      } else {
        const int E = cfg->n_experts, K = cfg->top_k, Fe = cfg->expert_ffn;
        orc_gemv(w->router[l], E, H, xn, rl);
        double margin = orc_router_topk(rl, E, K, ids, rw);
        if (forced_routes && forced_mask && forced_mask[l * B + b]) {
          /* adopt the given ids; weights from this oracle's own softmax */
          double mx = -INFINITY, z = 0.0, sel = 0.0;
          for (int e = 0; e < E; e++)
            if (rl[e] > mx) mx = rl[e];
          for (int e = 0; e < E; e++) z += exp(rl[e] - mx);
          for (int j = 0; j < K; j++) {
            ids[j] = forced_routes[((size_t)l * B + b) * K + j];
            rw[j] = exp(rl[ids[j]] - mx) / z;
            sel += rw[j];
          }
          for (int j = 0; j < K; j++) rw[j] /= sel;
        }
        if (route_ids)
          for (int j = 0; j < K; j++) route_ids[((size_t)l * B + b) * K + j] = ids[j];
        if (route_margin) route_margin[(size_t)l * B + b] = margin;
        for (int i = 0; i < H; i++) y[i] = 0.0;
        for (int j = 0; j < K; j++) {
          size_t e = (size_t)ids[j];
          orc_swiglu(w->ex_gate[l] + e * Fe * H, w->ex_up[l] + e * Fe * H,
                     w->ex_down[l] + e * H * Fe, Fe, H, xn, y2);
          for (int i = 0; i < H; i++) y[i] += rw[j] * y2[i];
        }
        if (cfg->shared_ffn > 0) {
          orc_swiglu(w->sh_gate[l], w->sh_up[l], w->sh_down[l], cfg->shared_ffn, H, xn, y2);
          for (int i = 0; i < H; i++) y[i] += y2[i];
        }
        for (int i = 0; i < H; i++) x[i] += y[i];
      }
      if (tx) memcpy(tx + ((size_t)(2 * l + 1) * B + b) * H, x, sizeof(double) * (size_t)H);
    }
    /* OP_RMS_LM_HEAD */
    orc_rmsnorm(x, w->final_norm, H, cfg->rms_eps, xn);
    gemv_w(w->lm_head, q8 ? &q8->lm_head : NULL, V, H, xn, logits + (size_t)b * V);
    argmax[b] = orc_argmax(logits + (size_t)b * V, V);
  }
  free(x);
  free(xn);
  free(q);
  free(k);
  free(v);
  free(att);
  free(y);
  free(y2);
  free(rl);
  free(ids);
  free(rw);
  return 0;
}
