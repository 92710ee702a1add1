/*
 * flint_oracle.h -- plain CPU oracle for the Flint-40B-A2B NVFP4 MoE feed-forward
 * and output-head step.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by
 * the package's smoke check and by the CPU-baseline leg of the benchmark, never by
 * the library's product path.  It shares no source with the CUDA library.
 *
 * What it follows:
 *  - "Flint: 125 tokens a second is what 2.5B active parameters buy at 273 GB/s",
 *    section "The shape, read from the headers": hidden 2,048; 256 routed experts of
 *    width 512, 6 selected per token; one shared expert of width 1,024; vocabulary
 *    150,144 with an untied output matrix.
 *  - same page, section "Why active parameters set the speed": the output head is
 *    quantised to 4 bits too; NVFP4 keeps 4-bit values with an 8-bit scale per 16
 *    values (section "Checking 125 tokens a second").
 *  - "Recursive Releases Flint, a 40B MoE Coding Model That Runs Locally at 125
 *    Tokens per Second", section "How does Flint's architecture work?": a router
 *    picks 6 experts per token, plus 1 always-active shared expert.
 * The pages leave the number formats, the quantisation recipe, the router
 * normalisation and the expert nonlinearity open; the readings taken are stated
 * beside each function below.
 *
 * All floating-point arithmetic is fp64, except the quantiser, whose bytes are
 * defined by fp32 operations (compile with -ffp-contract=off, no fast-math).
 */
#ifndef FLINT_ORACLE_H
#define FLINT_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_NONFINITE = 5 };

/* ---- number formats -------------------------------------------------------- */
/* E2M1 value of a 4-bit code (bit 3 = sign), read from the 16-entry table. */
double orc_e2m1_value(int code);
/* OCP FP8 E4M3 ("e4m3fn") value of a byte: bias 7, subnormals m*2^-9, max 448,
 * 0x7F/0xFF are NaN, no infinities. */
double orc_e4m3_value(int byte);
/* Round-to-nearest-even, saturating (|v| above the largest finite -> largest
 * finite) encoders from fp32.  Ties go to the even code. */
uint8_t orc_e4m3_encode(float v);
uint8_t orc_e2m1_encode(float v);
/* bf16 <-> wider.  bf16 -> fp64 is exact; fp64 -> bf16 rounds to nearest even. */
double orc_bf16_value(uint16_t bits);
uint16_t orc_bf16_from_double(double v);

/* ---- NVFP4 quantiser -------------------------------------------------------- */
/* w: bf16 bits [n_mat, rows, cols] -> codes [n_mat, rows, cols/2] (element 2j in the
 * low nibble of byte j), scales [n_mat, rows, cols/16] (E4M3), tsc [n_mat] (fp32).
 * Per matrix: tsc = amax/2688 (1.0 if amax == 0); per 16-block:
 * s = E4M3(amax_b/6/tsc), eff = decode(s)*tsc, q = E2M1(w/eff) (q = 0 if eff == 0).
 * Returns ORC_ERR_NONFINITE (and writes nothing for that matrix) if a weight is
 * NaN or infinite. */
int orc_quantize_nvfp4(const uint16_t* w, int64_t n_mat, int64_t rows, int64_t cols,
                       uint8_t* codes, uint8_t* scales, float* tsc);
/* Quantise fp32 rows with the tensor scale fixed at 1.0 (prefill activations). */
int orc_quantize_rows_unit(const float* v, int64_t rows, int64_t cols,
                           uint8_t* codes, uint8_t* scales);
/* fp32 dequantised values: fp32(fp32(e2m1*e4m3) * tsc). */
void orc_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, const float* tsc,
                          int64_t n_mat, int64_t rows, int64_t cols, float* out);

/* ---- MoE layer ---------------------------------------------------------------- */
typedef struct {
  const uint8_t* codes;   /* [n_mat, rows, cols/2] */
  const uint8_t* scales;  /* [n_mat, rows, cols/16] */
  const float* tsc;       /* [n_mat] */
} orc_nvfp4;

typedef struct {
  int hidden, n_experts, top_k, expert_width, shared_width;
  const uint16_t* router_w;   /* bf16 [E, H] */
  const float* router_bias;   /* fp32 [E] or NULL */
  orc_nvfp4 gate, up;         /* [E, F, H] */
  orc_nvfp4 down;             /* [E, H, F] */
  orc_nvfp4 sh_gate, sh_up;   /* [1, Fs, H] */
  orc_nvfp4 sh_down;          /* [1, H, Fs] */
  int router_score;           /* ORC_ROUTER_SOFTMAX or ORC_ROUTER_SIGMOID */
} orc_layer;

enum { ORC_ROUTER_SOFTMAX = 0, ORC_ROUTER_SIGMOID = 1 };

/* Router: logits = Wr x + b (fp64); the top_k experts by logit (ties to the lower
 * index) in that order; weights = p_i / sum of the selected p, where p is
 *  - ORC_ROUTER_SOFTMAX: the softmax over all experts (the default reading);
 *  - ORC_ROUTER_SIGMOID: the sigmoid of each logit, the scoring named in "Flint: 125
 *    tokens a second is what 2.5B active parameters buy at 273 GB/s", section "The
 *    shape, read from the headers".  Sigmoid is increasing, so the top_k by score
 *    are the top_k by logit; ranking by logit keeps that exact where fp64 sigmoids
 *    of large logits round to equal values.
 * logits may be NULL. */
void orc_router(const orc_layer* L, const uint16_t* x, double* logits, int32_t* idx,
                double* w);

/* One layer for n_tok independent tokens:
 * out = residual + sum_i w_i * down_i(silu(gate_i x) * up_i x) + shared(x).
 * residual: fp64 [n_tok, H] or NULL (then the bf16 input itself).
 * quantize_acts = 1 mirrors the prompt-processing path: x rows and the SwiGLU
 * outputs are NVFP4-quantised with unit tensor scale before each product.
 * idx/w: [n_tok, k] outputs (may be NULL).  Threads over tokens/rows.
 * A dense SwiGLU layer -- the model's two dense MLP layers, width 6,144 ("Flint: 125
 * tokens a second is what 2.5B active parameters buy at 273 GB/s", section "Built from
 * scratch?") -- is a layer with n_experts = top_k = expert_width = 0: no router, no
 * routed experts, out = residual + shared(x) with its matrices in sh_gate / sh_up /
 * sh_down.  (Reading: the pages give the dense layers' width only; they are taken as
 * the same SwiGLU block as an expert, without a router, added with weight 1.) */
int orc_moe_forward(const orc_layer* L, const uint16_t* x, const double* residual,
                    int64_t n_tok, int quantize_acts, double* out, int32_t* idx, double* w);

/* Sampling from one row of output-head logits.  "Recursive Releases Flint, a 40B MoE
 * Coding Model That Runs Locally at 125 Tokens per Second", section "How does Flint
 * perform on coding benchmarks?", samples at temperature 1.0, top-p 0.95 and top-k
 * 20 and says no more; the order taken is the usual one:
 *   1. the top_k logits (NaN read as -inf; ties to the lower index), descending;
 *   2. p_i = exp((l_i - l_0) / temperature) / sum of the same over the top_k;
 *   3. keep the shortest prefix i < m whose p sum reaches top_p (m >= 1);
 *   4. q_i = p_i / (p_0 + ... + p_{m-1});
 *   5. the draw is the first i < m with u < q_0 + ... + q_i (i = m - 1 if rounding
 *      leaves none), for an input u in [0, 1).
 * If every candidate is -inf, or the first is +inf (which then holds all the
 * probability; ties among +inf go to the lower index), the first candidate is drawn.  Returns its vocabulary
 * index; *m_out (may be NULL) receives m.  top_k is clipped to V. */
int32_t orc_sample(const float* logits, int64_t V, double temperature, int top_k, double top_p,
                   double u, int* m_out);

/* x_next = bf16(h / sqrt(mean(h^2) + eps)), gain 1. */
void orc_rmsnorm_bf16(const double* h, int64_t n, double eps, uint16_t* out);

/* Output head: logits[b, v] = sum_k deq(W[v, k]) x[b, k]; argmax with ties to the
 * lower index.  W is one NVFP4 matrix [V, H]. */
void orc_lm_head(const orc_nvfp4* W, int64_t V, int64_t H, const uint16_t* x, int64_t B,
                 double* logits, int32_t* argmax);

/* Expert-major order of the (token, slot) pairs: counts[e], offsets[e] (exclusive
 * scan), perm[offsets[e] + r] = t*k + j for the r-th pair routed to e, ascending t. */
void orc_expert_order(const int32_t* idx, int64_t n_tok, int k, int n_experts,
                      int32_t* counts, int32_t* offsets, int32_t* perm);

void orc_set_threads(int n);
int orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
