/*
 * flint_oracle.c -- plain, slow, obviously-correct CPU oracle (TEST INFRASTRUCTURE).
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * load this file's library.  It shares no code with the CUDA library.  See
 * flint_oracle.h for the page citations and the readings taken where the pages
 * are silent.  Build: gcc -O3 -fPIC -shared -ffp-contract=off -pthread.
 */
#include "flint_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* threads: a plain fork/join parallel-for over [0, n)                        */
/* ------------------------------------------------------------------------- */
static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n < 1 ? 1 : (n > 256 ? 256 : n); }
int orc_get_threads(void) { return g_threads; }

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void* ctx; int64_t lo, hi; } range_job;

static void* range_thread(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, range_fn fn, void* ctx) {
  int nt = g_threads;
  if (nt > n) nt = (int)n;
  if (nt <= 1) { if (n > 0) fn(ctx, 0, n); return; }
  pthread_t th[256];
  range_job jobs[256];
  int64_t chunk = (n + nt - 1) / nt;
  int started = 0;
  for (int t = 0; t < nt; ++t) {
    jobs[t].fn = fn; jobs[t].ctx = ctx;
    jobs[t].lo = t * chunk;
    jobs[t].hi = (t + 1) * chunk < n ? (t + 1) * chunk : n;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (t == 0) continue;  /* the caller runs chunk 0 */
    if (pthread_create(&th[t], NULL, range_thread, &jobs[t]) != 0) {
      fn(ctx, jobs[t].lo, jobs[t].hi);  /* could not start: run it here */
      jobs[t].hi = jobs[t].lo;
    }
    started = t;
  }
  fn(ctx, jobs[0].lo, jobs[0].hi);
  for (int t = 1; t <= started; ++t)
    if (jobs[t].hi > jobs[t].lo) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------- */
/* number formats                                                             */
/* ------------------------------------------------------------------------- */
/* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.  The 8 magnitudes,
 * code 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Codes 8..15 are their negatives. */
static const double E2M1_TABLE[16] = {
    0.0,  0.5,  1.0,  1.5,  2.0,  3.0,  4.0,  6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0};

double orc_e2m1_value(int code) { return E2M1_TABLE[code & 15]; }

double orc_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);          /* subnormal: m/8 * 2^(1-7) */
  else v = ldexp((double)(8 + m), e - 10);       /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Nearest of an ascending list of non-negative values, ties to the even index
 * (the index is the code, whose lowest bit is the mantissa's lowest bit). */
static int nearest_even(double a, const double* vals, int n) {
  if (a >= vals[n - 1]) return n - 1;              /* satfinite */
  int lo = 0, hi = n - 1;                           /* vals[lo] <= a < vals[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (vals[mid] <= a) lo = mid; else hi = mid;
  }
  if (vals[lo] == a) return lo;
  double dlo = a - vals[lo], dhi = vals[lo + 1] - a;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return lo + 1;
  return (lo & 1) ? lo + 1 : lo;
}

static double E4M3_ALL[256];  /* value of every byte; 0x00..0x7E ascend */
__attribute__((constructor)) static void e4m3_init(void) {
  for (int c = 0; c < 256; ++c) E4M3_ALL[c] = orc_e4m3_value(c);
}

uint8_t orc_e4m3_encode(float v) {
  int s = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (isnan(v)) return 0x7F;
  return (uint8_t)(s | nearest_even(a, E4M3_ALL, 127));
}

uint8_t orc_e2m1_encode(float v) {
  int s = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  return (uint8_t)(s | nearest_even(a, E2M1_TABLE, 8));
}

double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  /* bf16: 8 significant bits, exponent range of fp32 (normal >= 2^-126,
   * subnormal quantum 2^-133), largest finite (2 - 2^-7) * 2^127. */
  int e;
  frexp(a, &e);                  /* a = m * 2^e, 0.5 <= m < 1 */
  int q_exp = e - 8;             /* quantum of an 8-significant-bit value */
  if (q_exp < -133) q_exp = -133;
  double q = nearbyint(ldexp(a, -q_exp));   /* round half to even */
  double r = ldexp(q, q_exp);
  if (r > ldexp(255.0, 120)) return sign | 0x7F80;  /* overflow -> inf */
  float f = (float)r;                               /* exact */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* ------------------------------------------------------------------------- */
/* quantiser (fp32 arithmetic: the bytes are defined there)                    */
/* ------------------------------------------------------------------------- */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* One 16-element block with a given tensor scale. */
static void quantize_block(const float* v, float tsc, uint8_t* codes8, uint8_t* scale) {
  float amax_b = 0.0f;
  for (int j = 0; j < 16; ++j) {
    float a = fabsf(v[j]);
    if (a > amax_b) amax_b = a;
  }
  float t = amax_b / 6.0f;
  t = t / tsc;
  uint8_t s = orc_e4m3_encode(t);
  float eff = (float)E4M3_ALL[s] * tsc;   /* the e4m3 value is exact in fp32 */
  uint8_t q[16];
  for (int j = 0; j < 16; ++j) {
    if (eff == 0.0f) q[j] = 0;
    else q[j] = orc_e2m1_encode(v[j] / eff);
  }
  for (int j = 0; j < 8; ++j) codes8[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
  *scale = s;
}

typedef struct {
  const uint16_t* w; int64_t rows, cols; uint8_t* codes; uint8_t* scales; float tsc;
} qctx;

static void quantize_rows_fn(void* p, int64_t lo, int64_t hi) {
  qctx* c = (qctx*)p;
  float v[16];
  for (int64_t r = lo; r < hi; ++r)
    for (int64_t b = 0; b < c->cols / 16; ++b) {
      const uint16_t* src = c->w + r * c->cols + b * 16;
      for (int j = 0; j < 16; ++j) v[j] = bf16_to_f32(src[j]);
      quantize_block(v, c->tsc, c->codes + r * (c->cols / 2) + b * 8,
                     c->scales + r * (c->cols / 16) + b);
    }
}

int orc_quantize_nvfp4(const uint16_t* w, int64_t n_mat, int64_t rows, int64_t cols,
                       uint8_t* codes, uint8_t* scales, float* tsc) {
  if (n_mat < 0 || rows < 0 || cols < 0 || cols % 16) return ORC_ERR_ARG;
  int status = ORC_OK;
  for (int64_t m = 0; m < n_mat; ++m) {
    const uint16_t* wm = w + m * rows * cols;
    float amax = 0.0f;
    int finite = 1;
    for (int64_t i = 0; i < rows * cols; ++i) {
      float f = bf16_to_f32(wm[i]);
      if (!isfinite(f)) { finite = 0; break; }
      if (fabsf(f) > amax) amax = fabsf(f);
    }
    if (!finite) { status = ORC_ERR_NONFINITE; continue; }
    float t = (amax == 0.0f) ? 1.0f : amax / 2688.0f;   /* 2688 = 6 * 448 */
    tsc[m] = t;
    qctx c = {wm, rows, cols, codes + m * rows * (cols / 2), scales + m * rows * (cols / 16), t};
    parallel_for(rows, quantize_rows_fn, &c);
  }
  return status;
}

int orc_quantize_rows_unit(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                           uint8_t* scales) {
  if (cols % 16) return ORC_ERR_ARG;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < cols / 16; ++b)
      quantize_block(v + r * cols + b * 16, 1.0f, codes + r * (cols / 2) + b * 8,
                     scales + r * (cols / 16) + b);
  return ORC_OK;
}

static float deq_value(const uint8_t* codes_row, const uint8_t* scales_row, float tsc,
                       int64_t k) {
  int c = (codes_row[k >> 1] >> ((k & 1) * 4)) & 15;
  float p = (float)(E2M1_TABLE[c] * E4M3_ALL[scales_row[k >> 4]]);  /* exact in fp32 */
  return p * tsc;
}

void orc_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, const float* tsc,
                          int64_t n_mat, int64_t rows, int64_t cols, float* out) {
  for (int64_t m = 0; m < n_mat; ++m)
    for (int64_t r = 0; r < rows; ++r) {
      const uint8_t* cr = codes + (m * rows + r) * (cols / 2);
      const uint8_t* sr = scales + (m * rows + r) * (cols / 16);
      for (int64_t k = 0; k < cols; ++k)
        out[(m * rows + r) * cols + k] = deq_value(cr, sr, tsc[m], k);
    }
}

/* fp64 dot product of one dequantised NVFP4 row with an fp64 vector. */
static double dot_row(const orc_nvfp4* M, int64_t mat, int64_t rows, int64_t cols, int64_t r,
                      const double* x) {
  const uint8_t* cr = M->codes + (mat * rows + r) * (cols / 2);
  const uint8_t* sr = M->scales + (mat * rows + r) * (cols / 16);
  float t = M->tsc[mat];
  double acc = 0.0;
  for (int64_t k = 0; k < cols; ++k) acc += (double)deq_value(cr, sr, t, k) * x[k];
  return acc;
}

/* ------------------------------------------------------------------------- */
/* router                                                                     */
/* ------------------------------------------------------------------------- */
void orc_router(const orc_layer* L, const uint16_t* x, double* logits, int32_t* idx,
                double* w) {
  int E = L->n_experts, H = L->hidden, k = L->top_k;
  double* l = (double*)malloc(sizeof(double) * E);
  double* p = (double*)malloc(sizeof(double) * E);
  char* taken = (char*)calloc(E, 1);
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h)
      acc += orc_bf16_value(L->router_w[(int64_t)e * H + h]) * orc_bf16_value(x[h]);
    l[e] = acc + (L->router_bias ? (double)L->router_bias[e] : 0.0);
  }
  if (L->router_score == ORC_ROUTER_SIGMOID) {
    /* an independent score per expert */
    for (int e = 0; e < E; ++e) p[e] = 1.0 / (1.0 + exp(-l[e]));
  } else {
    /* softmax over all experts */
    double mx = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
  }
  /* top-k by logit, ties to the lower index */
  double psel = 0.0;
  for (int i = 0; i < k; ++i) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
    taken[best] = 1;
    idx[i] = best;
    psel += p[best];
  }
  for (int i = 0; i < k; ++i) w[i] = p[idx[i]] / psel;
  if (logits) memcpy(logits, l, sizeof(double) * E);
  free(l); free(p); free(taken);
}

/* ------------------------------------------------------------------------- */
/* MoE layer                                                                  */
/* ------------------------------------------------------------------------- */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Round a fp64 vector to fp32, NVFP4-quantise it with unit tensor scale, and
 * return the dequantised values (prompt-processing activation path). */
static void requantize_unit(double* v, int64_t n) {
  float* f = (float*)calloc(n, sizeof(float));
  uint8_t* c = (uint8_t*)calloc(n / 2, 1);
  uint8_t* s = (uint8_t*)calloc(n / 16, 1);
  float one = 1.0f;
  for (int64_t i = 0; i < n; ++i) f[i] = (float)v[i];
  orc_quantize_rows_unit(f, 1, n, c, s);
  for (int64_t i = 0; i < n; ++i) v[i] = (double)deq_value(c, s, one, i);
  free(f); free(c); free(s);
}

/* One expert's SwiGLU for input xin: y[H] = down(silu(gate xin) * up xin). */
static void expert_forward(const orc_nvfp4* G, const orc_nvfp4* U, const orc_nvfp4* D,
                           int64_t mat, int64_t F, int64_t H, const double* xin,
                           int quantize_acts, double* y) {
  double* hbuf = (double*)malloc(sizeof(double) * F);
  for (int64_t j = 0; j < F; ++j) {
    double g = dot_row(G, mat, F, H, j, xin);
    double u = dot_row(U, mat, F, H, j, xin);
    hbuf[j] = silu(g) * u;
  }
  if (quantize_acts) requantize_unit(hbuf, F);
  for (int64_t n = 0; n < H; ++n) y[n] = dot_row(D, mat, H, F, n, hbuf);
  free(hbuf);
}

typedef struct {
  const orc_layer* L; const uint16_t* x; const double* residual; int quantize_acts;
  double* out; int32_t* idx; double* w;
} fwdctx;

static void forward_tokens_fn(void* p, int64_t lo, int64_t hi) {
  fwdctx* c = (fwdctx*)p;
  const orc_layer* L = c->L;
  int64_t H = L->hidden, F = L->expert_width, Fs = L->shared_width;
  int k = L->top_k;
  double* xin = (double*)malloc(sizeof(double) * H);
  double* y = (double*)malloc(sizeof(double) * H);
  int32_t* ti = (int32_t*)malloc(sizeof(int32_t) * k);
  double* tw = (double*)malloc(sizeof(double) * k);
  for (int64_t t = lo; t < hi; ++t) {
    const uint16_t* xt = c->x + t * H;
    double* ot = c->out + t * H;
    if (k > 0) orc_router(L, xt, NULL, ti, tw);    /* k = 0: a dense layer, no router */
    for (int64_t h = 0; h < H; ++h) xin[h] = orc_bf16_value(xt[h]);
    if (c->quantize_acts) requantize_unit(xin, H);
    for (int64_t h = 0; h < H; ++h)
      ot[h] = c->residual ? c->residual[t * H + h] : orc_bf16_value(xt[h]);
    for (int i = 0; i < k; ++i) {
      expert_forward(&L->gate, &L->up, &L->down, ti[i], F, H, xin, c->quantize_acts, y);
      for (int64_t h = 0; h < H; ++h) ot[h] += tw[i] * y[h];
    }
    expert_forward(&L->sh_gate, &L->sh_up, &L->sh_down, 0, Fs, H, xin, c->quantize_acts, y);
    for (int64_t h = 0; h < H; ++h) ot[h] += y[h];
    if (c->idx) memcpy(c->idx + t * k, ti, sizeof(int32_t) * k);
    if (c->w) memcpy(c->w + t * k, tw, sizeof(double) * k);
  }
  free(xin); free(y); free(ti); free(tw);
}

int orc_moe_forward(const orc_layer* L, const uint16_t* x, const double* residual,
                    int64_t n_tok, int quantize_acts, double* out, int32_t* idx, double* w) {
  const int dense = L && L->top_k == 0 && L->n_experts == 0 && L->expert_width == 0;
  if (!L || (!dense && (L->top_k < 1 || L->top_k > L->n_experts)) || L->hidden % 16 ||
      L->expert_width % 16 || L->shared_width % 16 ||
      (L->router_score != ORC_ROUTER_SOFTMAX && L->router_score != ORC_ROUTER_SIGMOID))
    return ORC_ERR_ARG;
  fwdctx c = {L, x, residual, quantize_acts, out, idx, w};
  parallel_for(n_tok, forward_tokens_fn, &c);
  return ORC_OK;
}

void orc_rmsnorm_bf16(const double* h, int64_t n, double eps, uint16_t* out) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += h[i] * h[i];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_double(h[i] * r);
}

/* ------------------------------------------------------------------------- */
/* output head                                                                */
/* ------------------------------------------------------------------------- */
typedef struct {
  const orc_nvfp4* W; int64_t V, H, B; const double* xd; double* logits;
} headctx;

static void head_rows_fn(void* p, int64_t lo, int64_t hi) {
  headctx* c = (headctx*)p;
  for (int64_t v = lo; v < hi; ++v)
    for (int64_t b = 0; b < c->B; ++b)
      c->logits[b * c->V + v] = dot_row(c->W, 0, c->V, c->H, v, c->xd + b * c->H);
}

void orc_lm_head(const orc_nvfp4* W, int64_t V, int64_t H, const uint16_t* x, int64_t B,
                 double* logits, int32_t* argmax) {
  double* xd = (double*)malloc(sizeof(double) * B * H);
  for (int64_t i = 0; i < B * H; ++i) xd[i] = orc_bf16_value(x[i]);
  headctx c = {W, V, H, B, xd, logits};
  parallel_for(V, head_rows_fn, &c);
  for (int64_t b = 0; b < B; ++b) {
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (logits[b * V + v] > logits[b * V + best]) best = v;
    if (argmax) argmax[b] = (int32_t)best;
  }
  free(xd);
}

/* ------------------------------------------------------------------------- */
/* expert-major order of routed pairs (counting sort, stable in token order)   */
/* ------------------------------------------------------------------------- */
void orc_expert_order(const int32_t* idx, int64_t n_tok, int k, int n_experts,
                      int32_t* counts, int32_t* offsets, int32_t* perm) {
  for (int e = 0; e < n_experts; ++e) counts[e] = 0;
  for (int64_t i = 0; i < n_tok * k; ++i) counts[idx[i]]++;
  int32_t run = 0;
  for (int e = 0; e < n_experts; ++e) { offsets[e] = run; run += counts[e]; }
  int32_t* fill = (int32_t*)calloc(n_experts, sizeof(int32_t));
  for (int64_t t = 0; t < n_tok; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      perm[offsets[e] + fill[e]++] = (int32_t)(t * k + j);
    }
  free(fill);
}

/* ------------------------------------------------------------------------- */
/* Sampling after the output head                                            */
/* ------------------------------------------------------------------------- */
static double logit_or_ninf(float v) { return v == v ? (double)v : -INFINITY; }

int32_t orc_sample(const float* logits, int64_t V, double temperature, int top_k, double top_p,
                   double u, int* m_out) {
  if (top_k > V) top_k = (int)V;
  if (top_k < 1) top_k = 1;
  int64_t* cand = (int64_t*)malloc(sizeof(int64_t) * top_k);
  char* taken = (char*)calloc(V, 1);
  /* 1. top_k by repeated scans: the largest not yet taken, lowest index on ties */
  for (int i = 0; i < top_k; ++i) {
    int64_t best = -1;
    for (int64_t v = 0; v < V; ++v) {
      if (taken[v]) continue;
      if (best < 0 || logit_or_ninf(logits[v]) > logit_or_ninf(logits[best])) best = v;
    }
    taken[best] = 1;
    cand[i] = best;
  }
  const double l0 = logit_or_ninf(logits[cand[0]]);
  int32_t pick = (int32_t)cand[0];
  int m = 1;
  /* A +inf logit takes all the probability (the softmax's limit); with several, the
     lowest index (rank 0) is drawn, matching the top-k's tie order. */
  if (l0 != -INFINITY && l0 != INFINITY) {
    double* p = (double*)malloc(sizeof(double) * top_k);
    /* 2. softmax with temperature over the candidates */
    double z = 0.0;
    for (int i = 0; i < top_k; ++i) { p[i] = exp((logit_or_ninf(logits[cand[i]]) - l0) / temperature); z += p[i]; }
    for (int i = 0; i < top_k; ++i) p[i] /= z;
    /* 3. the shortest prefix reaching top_p */
    double cum = 0.0;
    m = top_k;
    for (int i = 0; i < top_k; ++i) {
      cum += p[i];
      if (cum >= top_p) { m = i + 1; break; }
    }
    double zm = 0.0;
    for (int i = 0; i < m; ++i) zm += p[i];
    /* 4.-5. renormalise and draw */
    double c = 0.0;
    pick = (int32_t)cand[m - 1];
    for (int i = 0; i < m; ++i) {
      c += p[i] / zm;
      if (u < c) { pick = (int32_t)cand[i]; break; }
    }
    free(p);
  }
  if (m_out) *m_out = m;
  free(cand); free(taken);
  return pick;
}
