/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow, double-precision CPU restatement of the per-token greedy decode
 * step of a Qwen3-shaped decoder over Q8_0 (or bf16) weights.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the decode
 * library never does, and the two share no source, header or table.
 *
 * Sources (page title, then section):
 *  [P1] inferno.rs blog, "IV.4: One command buffer per token":
 *       "Eight kernels" (q8_matvec, decode_scale, rms_norm_row, rope_row,
 *       append_kv, attention_decode, add_inplace, silu_hadamard, argmax_row);
 *       "The decoder: kernels and helpers" (embed_row);
 *       "One command buffer" (the per-layer op order, final norm, lm_head,
 *       argmax); "The correctness ladder" (tie rule, test shapes).
 *  [P2] "Adding Metal to my Rust LLM engine", "The matmul pain story" (bf16 /
 *       F16 row matvec) and "What the kernels do" (Llama op order without
 *       QK-norm).
 *  [P3] "Metal LLM decode", "Verification" (a Float64 CPU reference).
 *
 * Everything is computed in f64: the int8 x f16 (or bf16) weight products are
 * exact there.  Readings taken where the pages leave a step open:
 *  - RoPE angle a = pos * theta^(-i/(hd/2)) and its cos/sin are evaluated in
 *    f64 (the pages evaluate them with precise f32 functions).
 *  - argmax: NaN never wins; ties go to the lowest index; all-NaN -> -1.
 *  - prefill is the decode step repeated over the prompt positions 0..P-1.
 * The OpenMP loops split independent output rows (or heads) across threads;
 * every output is still summed by one thread in source order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* scalar formats                                                          */
/* ---------------------------------------------------------------------- */

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * [P1] "Eight kernels", decode_scale: the scale is the little-endian pair of
 * bytes at the start of the block, read as a half. */
double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1024.0 + (double)f, e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* One Q8_0 block: 34 bytes = scale (f16, bytes 0-1 little-endian) followed by
 * 32 signed 8-bit quants; element j is scale * quant_j.
 * [P1] "Eight kernels" (BLOCK_QLEN / BLOCK_BYTES, decode_scale, q8_matvec). */
void orc_q8_0_dequant_block(const uint8_t* blk, double* out32) {
  double s = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
  for (int j = 0; j < 32; ++j) out32[j] = s * (double)(int8_t)blk[2 + j];
}

/* ---------------------------------------------------------------------- */
/* matvecs                                                                 */
/* ---------------------------------------------------------------------- */

/* y[r] = sum_b scale_rb * sum_j quant_rbj * x[32 b + j] for a row-major
 * [rows x cols] Q8_0 matrix whose rows are cols/32 consecutive blocks.
 * [P1] "Eight kernels", q8_matvec. */
void orc_q8_0_matvec(const uint8_t* w, int64_t rows, int64_t cols, const double* x, double* y) {
  const int64_t bpr = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t* row = w + r * bpr * 34;
    double sum = 0.0;
    for (int64_t b = 0; b < bpr; ++b) {
      const uint8_t* blk = row + b * 34;
      double acc = 0.0;
      for (int j = 0; j < 32; ++j) acc += (double)(int8_t)blk[2 + j] * x[b * 32 + j];
      sum += orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8))) * acc;
    }
    y[r] = sum;
  }
}

/* y = W x for a row-major [rows x cols] bf16 matrix.
 * [P2] "The matmul pain story" (one output per row, plain dot product). */
void orc_bf16_matvec(const uint16_t* w, int64_t rows, int64_t cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double sum = 0.0;
    for (int64_t c = 0; c < cols; ++c) sum += orc_bf16_to_f64(w[r * cols + c]) * x[c];
    y[r] = sum;
  }
}

/* ---------------------------------------------------------------------- */
/* elementwise and row ops                                                 */
/* ---------------------------------------------------------------------- */

/* out = x * (mean(x^2) + eps)^(-1/2) * g over n elements.
 * [P1] "Eight kernels", rms_norm_row (gain multiplies, no 1 + g). */
void orc_rmsnorm(const double* x, const float* g, int64_t n, double eps, double* out) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; ++i) out[i] = x[i] * inv * (double)g[i];
}

/* The same norm applied to `rows` consecutive rows of n (per-head QK-norm). */
void orc_rmsnorm_rows(const double* x, const float* g, int64_t rows, int64_t n, double eps,
                      double* out) {
  for (int64_t r = 0; r < rows; ++r) orc_rmsnorm(x + r * n, g, n, eps, out + r * n);
}

/* Half-split rotary embedding, in place, for n_heads consecutive heads:
 * for i < hd/2, pair (i, i + hd/2) rotates by a = pos * theta^(-i/(hd/2)):
 * (u, w) -> (u cos a - w sin a, u sin a + w cos a).
 * [P1] "Eight kernels", rope_row. */
void orc_rope(double* x, int n_heads, int head_dim, int64_t pos, double theta) {
  int half = head_dim / 2;
  for (int h = 0; h < n_heads; ++h) {
    double* xh = x + (int64_t)h * head_dim;
    for (int i = 0; i < half; ++i) {
      double freq = pow(theta, -(double)i / (double)half);
      double a = (double)pos * freq;
      double c = cos(a), s = sin(a);
      double u = xh[i], w = xh[i + half];
      xh[i] = u * c - w * s;
      xh[i + half] = u * s + w * c;
    }
  }
}

/* Decode attention for one query row against S cached rows.
 * q: [n_heads * hd]; K, V: [S][kv_stride] with kv head g at columns g*hd.
 * Query head h reads kv head h / (n_heads / n_kv): scores
 * s_t = q_h . K[t]_g / sqrt(hd); a = softmax(s) (max subtracted);
 * out_h = sum_t a_t V[t]_g.   [P1] "Eight kernels", attention_decode. */
void orc_attention(const double* q, const double* K, const double* V, int64_t S, int64_t kv_stride,
                   int n_heads, int n_kv, int hd, double* out) {
  int group = n_heads / n_kv;
  double scale = 1.0 / sqrt((double)hd);
#pragma omp parallel for schedule(static)
  for (int h = 0; h < n_heads; ++h) {
    const double* qh = q + (int64_t)h * hd;
    int64_t off = (int64_t)(h / group) * hd;
    double* sc = (double*)malloc((size_t)(S > 0 ? S : 1) * sizeof(double));
    double m = -INFINITY;
    for (int64_t t = 0; t < S; ++t) {
      double d = 0.0;
      for (int j = 0; j < hd; ++j) d += qh[j] * K[t * kv_stride + off + j];
      sc[t] = d * scale;
      if (sc[t] > m) m = sc[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < S; ++t) {
      sc[t] = exp(sc[t] - m);
      sum += sc[t];
    }
    for (int j = 0; j < hd; ++j) {
      double acc = 0.0;
      for (int64_t t = 0; t < S; ++t) acc += sc[t] * V[t * kv_stride + off + j];
      out[(int64_t)h * hd + j] = acc / sum;
    }
    free(sc);
  }
}

/* silu(z) = z / (1 + e^-z).  [P1] "Eight kernels", silu_hadamard. */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* out = silu(gate) * up, elementwise (SwiGLU). */
void orc_silu_mul(const double* gate, const double* up, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_silu(gate[i]) * up[i];
}

/* Index of the largest element; ties go to the lowest index; NaN never wins;
 * -1 when every element is NaN (or n == 0).  [P1] "Eight kernels",
 * argmax_row, and "The correctness ladder" (planted tie). */
int64_t orc_argmax(const double* x, int64_t n) {
  int64_t best = -1;
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(x[i])) continue;
    if (best < 0 || x[i] > x[best]) best = i;
  }
  return best;
}

/* ---------------------------------------------------------------------- */
/* the model                                                               */
/* ---------------------------------------------------------------------- */

typedef struct {
  const float *attn_norm, *q_norm, *k_norm, *ffn_norm;
  const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
} orc_layer;

typedef struct {
  int n_layers, hidden, n_heads, n_kv, head_dim, inter, vocab, qk_norm, wtype;
  double theta, eps;
  int64_t max_seq, next_pos;
  orc_layer* layers;
  const void* lm_head;  /* [vocab x hidden] */
  const void* embed;    /* [vocab x hidden]; the lm_head bytes when tied */
  const float* out_norm;
  double *K, *V;        /* [n_layers][max_seq][kv_width] */
  int kv_f16;           /* cached rows rounded to f16 (the quantized-KV reading) */
  double *x, *xn, *q, *k, *v, *att, *tmp, *gate, *up, *h;
} orc_model;

enum { ORC_Q8_0 = 0, ORC_BF16 = 1 };

static void matvec(const orc_model* m, const void* w, int64_t rows, int64_t cols, const double* x,
                   double* y) {
  if (m->wtype == ORC_Q8_0)
    orc_q8_0_matvec((const uint8_t*)w, rows, cols, x, y);
  else
    orc_bf16_matvec((const uint16_t*)w, rows, cols, x, y);
}

orc_model* orc_model_new(int n_layers, int hidden, int n_heads, int n_kv, int head_dim, int inter,
                         int vocab, int qk_norm, int wtype, double theta, double eps,
                         int64_t max_seq) {
  if (n_layers <= 0 || hidden <= 0 || n_heads <= 0 || n_kv <= 0 || n_heads % n_kv ||
      head_dim <= 0 || head_dim % 2 || inter <= 0 || vocab <= 0 || max_seq <= 0 ||
      (wtype != ORC_Q8_0 && wtype != ORC_BF16) ||
      (wtype == ORC_Q8_0 && (hidden % 32 || inter % 32 || (n_heads * head_dim) % 32)))
    return NULL;
  orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
  m->n_layers = n_layers; m->hidden = hidden; m->n_heads = n_heads; m->n_kv = n_kv;
  m->head_dim = head_dim; m->inter = inter; m->vocab = vocab; m->qk_norm = qk_norm;
  m->wtype = wtype; m->theta = theta; m->eps = eps; m->max_seq = max_seq; m->next_pos = 0;
  m->layers = (orc_layer*)calloc((size_t)n_layers, sizeof(orc_layer));
  int64_t qw = (int64_t)n_heads * head_dim, kvw = (int64_t)n_kv * head_dim;
  size_t kvn = (size_t)n_layers * (size_t)max_seq * (size_t)kvw;
  m->K = (double*)calloc(kvn, sizeof(double));
  m->V = (double*)calloc(kvn, sizeof(double));
  int64_t wmax = hidden > qw ? hidden : qw;
  m->x = (double*)calloc((size_t)hidden, sizeof(double));
  m->xn = (double*)calloc((size_t)(wmax > inter ? wmax : inter), sizeof(double));
  m->q = (double*)calloc((size_t)qw, sizeof(double));
  m->k = (double*)calloc((size_t)kvw, sizeof(double));
  m->v = (double*)calloc((size_t)kvw, sizeof(double));
  m->att = (double*)calloc((size_t)qw, sizeof(double));
  m->tmp = (double*)calloc((size_t)hidden, sizeof(double));
  m->gate = (double*)calloc((size_t)inter, sizeof(double));
  m->up = (double*)calloc((size_t)inter, sizeof(double));
  m->h = (double*)calloc((size_t)inter, sizeof(double));
  if (!m->K || !m->V) {
    free(m->K); free(m->V); free(m->layers); free(m);
    return NULL;
  }
  return m;
}

/* Cached K/V rows stored as f16: each element rounded to the nearest f16,
 * ties to even (IEEE binary16), when it enters the cache.  The pages keep an
 * f32 cache and list a packed-F16 KV representation as the next step ("Metal
 * LLM decode", the batched prefill+decode arm); this is that step's reading. */
int orc_set_kv_f16(orc_model* m, int on) {
  if (!m) return -1;
  m->kv_f16 = on ? 1 : 0;
  return 0;
}

static double kv_store(const orc_model* m, double x) { return m->kv_f16 ? (double)(_Float16)x : x; }

void orc_model_free(orc_model* m) {
  if (!m) return;
  free(m->K); free(m->V); free(m->layers);
  free(m->x); free(m->xn); free(m->q); free(m->k); free(m->v); free(m->att); free(m->tmp);
  free(m->gate); free(m->up); free(m->h);
  free(m);
}

/* The model keeps the caller's pointers; the caller keeps the arrays alive. */
int orc_model_set_layer(orc_model* m, int l, const float* attn_norm, const void* wq, const void* wk,
                        const void* wv, const void* wo, const float* q_norm, const float* k_norm,
                        const float* ffn_norm, const void* w_gate, const void* w_up,
                        const void* w_down) {
  if (!m || l < 0 || l >= m->n_layers) return -1;
  orc_layer* L = &m->layers[l];
  L->attn_norm = attn_norm; L->wq = wq; L->wk = wk; L->wv = wv; L->wo = wo;
  L->q_norm = q_norm; L->k_norm = k_norm; L->ffn_norm = ffn_norm;
  L->w_gate = w_gate; L->w_up = w_up; L->w_down = w_down;
  return 0;
}

int orc_model_set_head(orc_model* m, const void* lm_head, const float* out_norm, const void* embed) {
  if (!m) return -1;
  m->lm_head = lm_head;
  m->out_norm = out_norm;
  m->embed = embed ? embed : lm_head;
  return 0;
}

/* Row `token` of the embedding, dequantised.
 * [P1] "The decoder: kernels and helpers", embed_row. */
static void embed_row(const orc_model* m, int64_t token, double* x) {
  const int64_t H = m->hidden;
  if (m->wtype == ORC_Q8_0) {
    const uint8_t* row = (const uint8_t*)m->embed + token * (H / 32) * 34;
    for (int64_t b = 0; b < H / 32; ++b) orc_q8_0_dequant_block(row + b * 34, x + b * 32);
  } else {
    const uint16_t* row = (const uint16_t*)m->embed + token * H;
    for (int64_t i = 0; i < H; ++i) x[i] = orc_bf16_to_f64(row[i]);
  }
}

/* One decode step at position pos for input token `token`:
 * the op order of [P1] "One command buffer" (18 ops per layer, then final
 * norm, lm_head and argmax).  When want_logits is 0 the final norm, lm_head
 * and argmax are skipped (prefill positions before the last).
 * Returns 0, or -1 bad argument, -2 all logits NaN. */
int orc_step(orc_model* m, int64_t token, int64_t pos, int want_logits, double* logits,
             int64_t* next) {
  if (!m || token < 0 || token >= m->vocab || pos < 0 || pos >= m->max_seq || pos > m->next_pos)
    return -1;
  const int64_t H = m->hidden, hd = m->head_dim, nq = m->n_heads, nkv = m->n_kv;
  const int64_t qw = nq * hd, kvw = nkv * hd, I = m->inter;
  embed_row(m, token, m->x);
  for (int l = 0; l < m->n_layers; ++l) {
    const orc_layer* L = &m->layers[l];
    double* Kl = m->K + (int64_t)l * m->max_seq * kvw;
    double* Vl = m->V + (int64_t)l * m->max_seq * kvw;
    orc_rmsnorm(m->x, L->attn_norm, H, m->eps, m->xn);
    matvec(m, L->wq, qw, H, m->xn, m->q);
    matvec(m, L->wk, kvw, H, m->xn, m->k);
    matvec(m, L->wv, kvw, H, m->xn, m->v);
    if (m->qk_norm) {
      orc_rmsnorm_rows(m->q, L->q_norm, nq, hd, m->eps, m->q);
      orc_rmsnorm_rows(m->k, L->k_norm, nkv, hd, m->eps, m->k);
    }
    orc_rope(m->q, (int)nq, (int)hd, pos, m->theta);
    orc_rope(m->k, (int)nkv, (int)hd, pos, m->theta);
    for (int64_t i = 0; i < kvw; ++i) {  /* append_kv */
      Kl[pos * kvw + i] = kv_store(m, m->k[i]);
      Vl[pos * kvw + i] = kv_store(m, m->v[i]);
    }
    orc_attention(m->q, Kl, Vl, pos + 1, kvw, (int)nq, (int)nkv, (int)hd, m->att);
    matvec(m, L->wo, H, qw, m->att, m->tmp);
    for (int64_t i = 0; i < H; ++i) m->x[i] += m->tmp[i];  /* add_inplace */
    orc_rmsnorm(m->x, L->ffn_norm, H, m->eps, m->xn);
    matvec(m, L->w_gate, I, H, m->xn, m->gate);
    matvec(m, L->w_up, I, H, m->xn, m->up);
    orc_silu_mul(m->gate, m->up, I, m->h);
    matvec(m, L->w_down, H, I, m->h, m->tmp);
    for (int64_t i = 0; i < H; ++i) m->x[i] += m->tmp[i];
  }
  m->next_pos = pos + 1;
  if (!want_logits) {
    if (next) *next = -1;
    return 0;
  }
  orc_rmsnorm(m->x, m->out_norm, H, m->eps, m->xn);
  matvec(m, m->lm_head, m->vocab, H, m->xn, logits);
  int64_t a = orc_argmax(logits, m->vocab);
  if (next) *next = a;
  return a < 0 ? -2 : 0;
}

/* The residual stream after the last step (for closed-form checks). */
void orc_get_hidden(const orc_model* m, double* out) {
  memcpy(out, m->x, (size_t)m->hidden * sizeof(double));
}

/* Read or overwrite one cached row (layer l, position pos). */
int orc_kv_get(const orc_model* m, int l, int64_t pos, double* k, double* v) {
  if (!m || l < 0 || l >= m->n_layers || pos < 0 || pos >= m->max_seq) return -1;
  int64_t kvw = (int64_t)m->n_kv * m->head_dim;
  const double* Kl = m->K + ((int64_t)l * m->max_seq + pos) * kvw;
  const double* Vl = m->V + ((int64_t)l * m->max_seq + pos) * kvw;
  memcpy(k, Kl, (size_t)kvw * sizeof(double));
  memcpy(v, Vl, (size_t)kvw * sizeof(double));
  return 0;
}

/* Load n_pos cached rows for every layer from f32 arrays [n_layers][n_pos][kvw]
 * and set the next position to n_pos. */
int orc_kv_load(orc_model* m, int64_t n_pos, const float* k, const float* v) {
  if (!m || n_pos < 0 || n_pos > m->max_seq) return -1;
  int64_t kvw = (int64_t)m->n_kv * m->head_dim;
  for (int l = 0; l < m->n_layers; ++l)
    for (int64_t p = 0; p < n_pos; ++p)
      for (int64_t i = 0; i < kvw; ++i) {
        int64_t src = ((int64_t)l * n_pos + p) * kvw + i;
        int64_t dst = ((int64_t)l * m->max_seq + p) * kvw + i;
        m->K[dst] = kv_store(m, (double)k[src]);
        m->V[dst] = kv_store(m, (double)v[src]);
      }
  m->next_pos = n_pos;
  return 0;
}

int64_t orc_next_pos(const orc_model* m) { return m ? m->next_pos : -1; }

void orc_reset(orc_model* m) {
  if (m) m->next_pos = 0;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
