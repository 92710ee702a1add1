/*
 * flint.h -- C ABI of the Flint NVFP4 MoE feed-forward / output-head library for
 * one NVIDIA B300 (sm_103a).
 *
 * What it computes.  The token-generation step of the Flint-40B-A2B MoE body and
 * head, as described in "Flint: 125 tokens a second is what 2.5B active parameters
 * buy at 273 GB/s" (section "The shape, read from the headers": hidden 2,048; 256
 * routed SwiGLU experts of width 512 with 6 selected per token; one shared expert
 * of width 1,024; an untied 150,144-entry output head) and "Recursive Releases
 * Flint, a 40B MoE Coding Model That Runs Locally at 125 Tokens per Second"
 * (section "How does Flint's architecture work?": a router selects 6 experts per
 * token, plus 1 always-active shared expert).  Weights are NVFP4 ("Flint: 125
 * tokens a second ...", sections "Why active parameters set the speed" -- the output
 * head is 4-bit too -- and "Checking 125 tokens a second" -- 4-bit values with an
 * 8-bit scale per 16, 4.5 bits per weight).  Prompt processing ("Flint-40B-A2B:
 * AI-Built MoE Coding Model Hits 125 tok/s on MacBook Pro", section "Custom
 * Inference Kernels") is the same layer over many tokens at once.
 *
 * NVFP4 matrix [rows, cols] (blocks of 16 along cols):
 *   codes  uint8 [rows, cols/2]  E2M1 codes; element 2j in bits 0-3 of byte j,
 *                                element 2j+1 in bits 4-7 (bit 3 of a code = sign)
 *   scales uint8 [rows, cols/16] E4M3 (OCP "e4m3fn") block scales, row-major
 *   tensor_scale fp32            one per matrix
 *   value(r, c) = fp32(fp32(e2m1(code) * e4m3(scale)) * tensor_scale)
 * A stack of n_mat matrices is stored matrix after matrix.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated.  Structs passed by
 *    pointer (flint_nvfp4, flint_moe_layer) live in HOST memory and are read
 *    during the call only.
 *  - Nothing allocates, frees or synchronises, except flint_last_device_status
 *    (which synchronises the stream).  All work is enqueued on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream).  Scratch memory is the
 *    caller's workspace `ws` of `ws_bytes` bytes (see flint_workspace_bytes),
 *    256-byte aligned; two calls in flight at once need distinct workspaces.
 *  - Weight pointers (codes, scales, router_w) and activation inputs (x_bf16)
 *    must be 16-byte aligned (128-bit loads) with rows of a multiple of 32
 *    elements; outputs and per-token vectors (out, residual, logits, topk_*)
 *    need only their element's natural alignment.  Argument checks run on the
 *    host before any launch and return an error code without enqueuing
 *    anything.
 *  - Conditions found on the device (non-finite weights, a bounded wait that
 *    expired) set a device status word that flint_last_device_status reads and
 *    clears.  Kernels never trap.
 */
#ifndef FLINT_H
#define FLINT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLINT_OK = 0,
  FLINT_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, k > E, ... */
  FLINT_ERR_ALIGNMENT = 2,     /* a pointer is not 16-byte aligned */
  FLINT_ERR_SHAPE = 3,         /* cols not a multiple of 32, mismatched shapes */
  FLINT_ERR_WORKSPACE = 4,     /* ws too small or not 256-byte aligned */
  FLINT_ERR_NONFINITE = 5,     /* (device) a NaN/Inf weight was quantised */
  FLINT_ERR_TIMEOUT = 6,       /* (device) a bounded wait gave up */
  FLINT_ERR_CUDA = 7,          /* a CUDA runtime call or launch failed */
  FLINT_ERR_UNSUPPORTED = 8    /* a size beyond what this build supports */
} flint_status;

typedef void* flint_stream; /* a cudaStream_t */

/* One NVFP4 matrix or stack of matrices (device pointers; struct in host memory). */
typedef struct {
  const uint8_t* codes;       /* [n_mat, rows, cols/2] */
  const uint8_t* scales;      /* [n_mat, rows, cols/16] */
  const float* tensor_scale;  /* [n_mat] */
  int n_mat, rows, cols;
} flint_nvfp4;

/* One MoE layer.  Routed experts are stacks of n_experts matrices:
 *   gate, up : [E, F, H]      down : [E, H, F]
 *   sh_gate, sh_up : [1, Fs, H]   sh_down : [1, H, Fs]
 * router_w is bf16 [E, H]; router_bias fp32 [E] or NULL (added to the logits).
 * The decode entry points read these row-major stacks directly (one copy of every
 * weight serves decode).
 * A dense SwiGLU layer (the model's two dense MLP layers, width 6,144: "Flint: 125
 * tokens a second ...", section "Built from scratch?") is a layer with n_experts =
 * top_k = expert_width = 0: router_w, router_bias and the routed stacks are ignored
 * (may be NULL), its block is sh_gate / sh_up / sh_down (shared_width a multiple of
 * 64) and it is added with weight 1:  out = res + Wd (silu(Wg x) * (Wu x)).  The decode
 * entry points take dense layers, alone or between MoE layers; flint_moe_prefill
 * returns FLINT_ERR_UNSUPPORTED for them.
 * mma_scales: MMA scale copies (flint_nvfp4_mma_scales) of gate, up, down, sh_gate,
 * sh_up, sh_down in that order, required by flint_moe_prefill only, which reads the
 * row-major codes and these scales. */
typedef struct {
  int hidden, n_experts, top_k, expert_width, shared_width;
  const void* router_w;
  const float* router_bias;
  flint_nvfp4 gate, up, down;
  flint_nvfp4 sh_gate, sh_up, sh_down;
  const uint8_t* mma_scales[6];
  int router_score;            /* FLINT_ROUTER_SOFTMAX (0) or FLINT_ROUTER_SIGMOID (1) */
} flint_moe_layer;

/* Router scoring of a layer (flint_moe_layer.router_score).  Both select the top_k
 * experts by logit, ties to the lower index, and renormalise over the selected:
 *  - FLINT_ROUTER_SOFTMAX: w_i = exp(l_i - l_max) / sum over the selected (the
 *    softmax over all E, renormalised);
 *  - FLINT_ROUTER_SIGMOID: w_i = sigmoid(l_i) / sum of the selected sigmoids.  This is
 *    the scoring "Flint: 125 tokens a second is what 2.5B active parameters buy at 273
 *    GB/s", section "The shape, read from the headers", names.  Sigmoid is
 *    increasing, so the same experts are selected.
 * Any other value is FLINT_ERR_INVALID_ARG. */
#define FLINT_ROUTER_SOFTMAX 0
#define FLINT_ROUTER_SIGMOID 1

/* Limits of this build. */
#define FLINT_MAX_DECODE_TOKENS 8     /* B of flint_moe_decode / flint_lm_head */
#define FLINT_MAX_HIDDEN 4096
#define FLINT_MAX_EXPERTS 512
#define FLINT_MAX_TOP_K 16
#define FLINT_MAX_LAYERS 64           /* n_layers of flint_decode_tokens */

/* ----------------------------------------------------------------------------
 * flint_quantize_nvfp4 -- bf16 weights -> NVFP4.
 * Follows the 4.5-bit format of "Flint: 125 tokens a second ...", section
 * "Checking 125 tokens a second".  The pages do not give the recipe; this one is
 * the two-level NVFP4 scheme, all in fp32 with IEEE division:
 *   tsc   = amax(|W_m|) / 2688        (2688 = 6 * 448; 1.0 if amax == 0)
 *   s_b   = E4M3_rne_satfinite((amax_b / 6) / tsc)   per 16-element block
 *   eff_b = e4m3(s_b) * tsc
 *   q     = E2M1_rne_satfinite(w / eff_b)            (0 when eff_b == 0)
 * w_bf16: [n_mat, rows, cols] bf16, device.  codes/scales/tensor_scale: outputs
 * (device, caller-owned).  ws: flint_workspace_bytes(FLINT_OP_QUANTIZE, ...).
 * A NaN/Inf weight sets FLINT_ERR_NONFINITE in the device status word (the
 * matrix's outputs are then unspecified).  cols % 32 == 0.
 * -------------------------------------------------------------------------- */
flint_status flint_quantize_nvfp4(const void* w_bf16, int n_mat, int rows, int cols,
                                  uint8_t* codes, uint8_t* scales, float* tensor_scale,
                                  void* ws, size_t ws_bytes, flint_stream stream);

/* MMA scale copy of an NVFP4 stack: its block scales rearranged into the layout the
 * block-scaled tensor-core products of the prompt path read, so that the scales of a
 * 128-row tile and 64 columns are one contiguous 512-byte piece.  For matrix m,
 * row r = 128 rt + i, 16-column block b = 4 k + j (i < 128, j < 4):
 *   scales_mma[m][rt][k][16 (i % 32) + 4 (i / 32) + j] = scales[m][r][b]
 * Requires rows % 128 == 0 and cols % 64 == 0; scales_mma (device, 16-byte aligned)
 * has the size of the row-major scales.  Errors: FLINT_ERR_SHAPE for other sizes. */
flint_status flint_nvfp4_mma_scales(const flint_nvfp4* m, uint8_t* scales_mma,
                                    flint_stream stream);

/* Block-scaled FP4 tensor-core microbenchmark (tcgen05.mma kind::mxf4nvf4, operands
 * in shared memory and TMEM only), one CTA per launch slot, `ctas` CTAs:
 *   mode 0: per iteration 8 MMAs of M = 128, N = 128, K = 64 (2 * 128 * 128 * 64 FLOP
 *           each) issued back to back -- the peak of the block-scaled FP4 products
 *           that the prompt path's grouped GEMM uses;
 *   mode 1: per iteration one chain of 16 K-steps of M = 128, N = 32 with their scale
 *           copies, a commit, its wait and the accumulator read -- the latency of the
 *           decode kernel's per-tile products;
 *   modes 2-4: mode 1's chain with the scales copied once before the loop (2), the
 *           scale copies alone (3), two independent chains of 8 K-steps (4), and
 *           modes 1 and 2 with the K-steps unrolled (5, 6).
 * cycles (device, 16-byte aligned, `ctas` entries) receives each CTA's clock cycles
 * over its loop.  Errors: FLINT_ERR_INVALID_ARG for another mode or a non-positive
 * count. */
flint_status flint_bench_fp4_mma(int mode, int iters, int ctas, unsigned long long* cycles,
                                 flint_stream stream);

/* Dequantise an NVFP4 stack to fp32 [n_mat, rows, cols] (the value formula above).
 * A check and debugging aid; no workspace. */
flint_status flint_dequantize_nvfp4(const flint_nvfp4* m, float* out, flint_stream stream);

/* ----------------------------------------------------------------------------
 * flint_moe_decode -- one MoE layer for B <= FLINT_MAX_DECODE_TOKENS tokens
 * (flint_decode_tokens with one layer and no head; the tokens run one after
 * another).
 * Router: logits = Wr x + b (bf16 x bf16, fp32 accumulate); the top_k experts by
 * logit (ties to the lower index) in descending order; weights = the selected
 * scores renormalised, with softmax or sigmoid scores as layer->router_score says
 * ("Recursive Releases Flint ...", "How does Flint's architecture work?").  Experts
 * are SwiGLU:
 *   h_e = silu(Wg_e x) * (Wu_e x),  y_e = Wd_e h_e
 * and the shared expert is always added with weight 1:
 *   out = residual + sum_i w_i y_{e_i} + y_shared
 * x_bf16: [B, H] bf16.  residual: fp32 [B, H], or NULL to use x itself.
 * out: fp32 [B, H].  x_next_bf16: NULL, or bf16 [B, H] receiving
 *   RMSNorm(out) = bf16(out / sqrt(mean(out^2) + rms_eps)) (gain 1) for chaining
 *   layers.  topk_idx int32 [B, k] / topk_w fp32 [B, k]: optional outputs.
 * out may alias residual.  ws: flint_workspace_bytes(FLINT_OP_MOE_DECODE, ...).
 * -------------------------------------------------------------------------- */
flint_status flint_moe_decode(const flint_moe_layer* layer, const void* x_bf16,
                              const float* residual, float* out, void* x_next_bf16,
                              float rms_eps, int32_t* topk_idx, float* topk_w, int B,
                              void* ws, size_t ws_bytes, flint_stream stream);

/* ----------------------------------------------------------------------------
 * flint_decode_tokens -- T tokens, one after another, each through n_layers chained
 * MoE layers and (optionally) the output head, in ONE persistent kernel launch.
 * For token t:   h_0 = residual[t] (or x[t] if residual is NULL), x_0 = x[t]
 *                h_{l+1} = h_l + MoE_l(x_l)      (MoE_l as in flint_moe_decode)
 *                x_{l+1} = bf16(RMSNorm(h_{l+1}))  (eps rms_eps, gain 1)
 * and the head, when given, reads x_{n_layers}:  logits[t] = W x, argmax[t].
 * This is the per-token FFN weight stream of "Flint: 125 tokens a second ...",
 * section "Why active parameters set the speed" (every active weight read once
 * per token), and the CUDA counterpart of the single fused decode kernel of
 * "Flint-40B-A2B: AI-Built MoE Coding Model Hits 125 tok/s on MacBook Pro",
 * section "Custom Inference Kernels".
 * layers: host array of n_layers (<= FLINT_MAX_LAYERS) layers of the same hidden size.
 * head: one NVFP4 matrix [1, V, H], or NULL.  x_bf16: [T, H].  residual: fp32
 * [T, H] or NULL.  Outputs, each optional: out fp32 [T, H] = h_{n_layers};
 * x_out_bf16 [T, H] = x_{n_layers}; logits fp32 [T, V]; argmax int32 [T];
 * topk_idx int32 / topk_w fp32 [T, n_layers, kmax] (kmax = the largest top_k; layer
 * l fills its first top_k entries).
 * How it runs: clusters of 16 CTAs, one CTA per SM, as many clusters as the device
 * holds at once (at most 8; 7 on a 148-SM B300).  Each routed cluster computes all
 * router logits itself and takes one selected expert; the remaining clusters take the
 * shared expert; the only exchange between clusters is one tagged partial-sum board
 * per layer.  Every sum has a fixed order, so runs repeat bit for bit.  Every wait
 * is bounded (FLINT_ERR_TIMEOUT in the device status word if one expires; see
 * flint_set_wait_limit_ns).
 * Supported shapes: hidden a power of two in [256, 2048]; expert and shared widths
 * powers of two >= 64 with the shared width a multiple of the expert width and the
 * expert width at most 512 at hidden 2048 (1024 below); router rows per CTA
 * (n_experts / 16, rounded up) times hidden times 2 at most 64 KiB; top_k at most
 * FLINT_MAX_TOP_K.  Other shapes return FLINT_ERR_UNSUPPORTED.
 * ws: flint_workspace_bytes(FLINT_OP_MOE_DECODE, ...).
 * -------------------------------------------------------------------------- */
flint_status flint_decode_tokens(const flint_moe_layer* layers, int n_layers,
                                 const flint_nvfp4* head, const void* x_bf16,
                                 const float* residual, int T, float rms_eps, float* out,
                                 void* x_out_bf16, float* logits, int32_t* argmax,
                                 int32_t* topk_idx, float* topk_w, void* ws,
                                 size_t ws_bytes, flint_stream stream);

/* flint_decode_tokens with the head's token drawn instead of taken greedily ("Recursive
 * Releases Flint, a 40B MoE Coding Model That Runs Locally at 125 Tokens per Second",
 * section "How does Flint perform on coding benchmarks?": temperature 1.0, top-p 0.95,
 * top-k 20), fused into the same launch: the logits never need to leave the GPU.
 * tokens[t] (int32 [T]) is the draw of flint_sample_logits from token t's logits with
 * uniforms[t] (fp32 [T], the caller's numbers in [0, 1)): the top_k logits (ties to the
 * lower index), p_i = exp((l_i - l_0) / temperature) over them, the shortest prefix
 * whose p sum reaches top_p, the first i of it with uniforms[t] < (p_0 + ... + p_i) /
 * (prefix sum); a +inf or all -inf leading logit gives the first candidate.  argmax
 * (optional) is the first candidate.  top_k is clipped to the vocabulary.  Errors:
 * those of flint_decode_tokens; FLINT_ERR_INVALID_ARG for a null head, uniforms or
 * tokens, temperature not > 0 and finite, top_p outside (0, 1], top_k < 1;
 * FLINT_ERR_UNSUPPORTED for top_k > FLINT_MAX_SAMPLE_TOP_K or more than 2048
 * vocabulary rows per CTA (a vocabulary above ~229k at 112 CTAs). */
flint_status flint_decode_tokens_sample(const flint_moe_layer* layers, int n_layers,
                                        const flint_nvfp4* head, const void* x_bf16,
                                        const float* residual, int T, float rms_eps,
                                        float temperature, int top_k, float top_p,
                                        const float* uniforms, int32_t* tokens, float* out,
                                        void* x_out_bf16, float* logits, int32_t* argmax,
                                        int32_t* topk_idx, float* topk_w, void* ws,
                                        size_t ws_bytes, flint_stream stream);

/* flint_decode_tokens with a per-layer record of the chain, for checking it layer by
 * layer against a reference:  x_trace_bf16 [T, n_layers, H] receives x_l (the bf16
 * input of layer l as the kernel staged it) and h_trace fp32 [T, n_layers, H]
 * receives h_l (the residual stream entering layer l).  Either may be NULL; both
 * 16-byte aligned.  Everything else is flint_decode_tokens. */
flint_status flint_decode_tokens_trace(const flint_moe_layer* layers, int n_layers,
                                       const flint_nvfp4* head, const void* x_bf16,
                                       const float* residual, int T, float rms_eps, float* out,
                                       void* x_out_bf16, float* logits, int32_t* argmax,
                                       int32_t* topk_idx, float* topk_w, void* x_trace_bf16,
                                       float* h_trace, void* ws, size_t ws_bytes,
                                       flint_stream stream);

/* Bound, in nanoseconds of the GPU's global timer, of every wait the kernels make on
 * another CTA or on a copy (default 2 s; 0 restores it).  A wait that runs out sets
 * FLINT_ERR_TIMEOUT in the device status word and releases every other wait, and the
 * kernel runs to its end without hanging (its outputs are then unspecified).  Applies
 * to launches made after the call, from any host thread. */
flint_status flint_set_wait_limit_ns(uint64_t ns);

/* Fault-handling test aid: arms the next launch made by this host thread to withhold
 * one hand-over, so that the waits on it run out:  what = 1, the next decode launch
 * (flint_decode_tokens / flint_moe_decode / ...): CTA 0 never posts its first partial
 * sums;  what = 2, the next prompt launch (flint_moe_prefill): the gate/up GEMM's copy
 * issuer withholds its first pipeline stage;  what = 0 disarms.  Used with a short
 * flint_set_wait_limit_ns to test that an expired wait is reported
 * (FLINT_ERR_TIMEOUT) and that the next normal call succeeds.  FLINT_ERR_INVALID_ARG
 * for other values. */
flint_status flint_debug_hold_next_launch(int what);

/* ----------------------------------------------------------------------------
 * flint_decode_tokens_noalloc -- flint_decode_tokens without a workspace argument.
 * No counterpart on the Flint pages: this is a service to callers that cannot
 * allocate device memory for scratch -- a host that reserves the whole GPU up front
 * and gives its extensions no allocator, or a serving loop that must not call
 * cudaMalloc (which can block and synchronise the device).  The scratch lives in a
 * fixed device array of FLINT_NOALLOC_SCRATCH_BYTES inside the library, held on
 * every GPU that loads the library until the process exits; this entry point calls
 * no cudaMalloc/cudaFree or other allocating routine.
 *  - The first call on a device looks up that array's device address
 *    (cudaGetSymbolAddress) for the current device and caches it; make that first
 *    call before any stream capture.
 *  - All calls share the one array.  Calls whose kernels overlap on the GPU (other
 *    streams, other host threads) race on it and must be serialised by the caller.
 *    Each call clears what must start at zero; the rest is rewritten before use.
 *  - A hidden size whose scratch exceeds FLINT_NOALLOC_SCRATCH_BYTES is rejected with
 *    FLINT_ERR_UNSUPPORTED; every hidden size flint_decode_tokens supports fits.
 *  - The cached address belongs to the device's current context: after
 *    cudaDeviceReset (or any teardown of the primary context) the library must be
 *    reloaded before this entry point is called again on that device.
 * Arguments and results are those of flint_decode_tokens.
 * -------------------------------------------------------------------------- */
#define FLINT_NOALLOC_SCRATCH_BYTES (512 * 1024)
flint_status flint_decode_tokens_noalloc(const flint_moe_layer* layers, int n_layers,
                                         const flint_nvfp4* head, const void* x_bf16,
                                         const float* residual, int T, float rms_eps,
                                         float* out, void* x_out_bf16, float* logits,
                                         int32_t* argmax, int32_t* topk_idx, float* topk_w,
                                         flint_stream stream);

/* ----------------------------------------------------------------------------
 * flint_moe_prefill -- the same layer over T prompt tokens, as a token-permuted
 * grouped GEMM on block-scaled FP4 tensor cores.  Both operands of the FP4
 * products are NVFP4: x rows and the SwiGLU outputs h are quantised with the
 * recipe above and a unit tensor scale before their products.
 *   out[t] = x[t] + sum_j w_tj * y_{e_tj}(t) + y_shared(t)      (fp32 [T, H])
 * The terms are added into out with fp32 reductions in no fixed order, so out may
 * differ from run to run in its last bits (the decode entry points are bit-exact run
 * to run).  topk_idx / topk_w: optional [T, k] outputs.  expert_counts: optional int32 [E]
 * output (tokens routed to each expert); pair_order: optional int32 [T*k] output,
 * the (t*k + j) pair ids in expert-major order, ascending t within an expert.
 * ws: flint_workspace_bytes(FLINT_OP_MOE_PREFILL, ...).
 * -------------------------------------------------------------------------- */
flint_status flint_moe_prefill(const flint_moe_layer* layer, const void* x_bf16, float* out,
                               int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                               int32_t* pair_order, int T, void* ws, size_t ws_bytes,
                               flint_stream stream);

/* ----------------------------------------------------------------------------
 * flint_lm_head -- NVFP4 output head ("Flint: 125 tokens a second ...", sections
 * "The shape, read from the headers" and "Why active parameters set the speed").
 * logits[b, v] = sum_k value(W[v, k]) x[b, k]  (fp32 [B, V]); argmax[b] = the
 * largest logit's index, ties to the lower index (int32 [B]).  Either output may
 * be NULL.  W: one matrix [1, V, H], H a multiple of 128 (else FLINT_ERR_SHAPE).
 * B <= FLINT_MAX_DECODE_TOKENS; the B tokens share one pass over W (products on
 * mma.sync tensor cores with fp32 accumulation), so B = 8 reads the weights once.
 * ws: flint_workspace_bytes(FLINT_OP_LM_HEAD, ...).
 * -------------------------------------------------------------------------- */
flint_status flint_lm_head(const flint_nvfp4* W, const void* x_bf16, float* logits,
                           int32_t* argmax, int B, void* ws, size_t ws_bytes,
                           flint_stream stream);

/* ----------------------------------------------------------------------------
 * flint_sample_logits -- draw one token per row of output-head logits.  "Recursive
 * Releases Flint, a 40B MoE Coding Model That Runs Locally at 125 Tokens per Second",
 * section "How does Flint perform on coding benchmarks?", samples at temperature
 * 1.0, top-p 0.95 and top-k 20; the pages give no more, and the order taken is the
 * usual one.  Per row b:
 *   1. the top_k logits (NaN read as -inf; ties to the lower index), descending;
 *   2. p_i = exp((l_i - l_0) / temperature) / sum of the same over them;
 *   3. the shortest prefix i < m whose p sum reaches top_p (m >= 1);
 *   4. out[b] = the vocabulary index of the first i < m with
 *      uniforms[b] < (p_0 + ... + p_i) / (p_0 + ... + p_{m-1})
 *      (i = m - 1 if rounding leaves none); all candidates -inf, or a +inf logit
 *      (all the probability; several: the lowest index): the first candidate.
 * The random numbers are the caller's: uniforms fp32 [B] in [0, 1).  Computed in
 * fp32, so a draw may differ from an exact one only where uniforms[b] or top_p lies
 * within float rounding of a cumulative sum.
 * logits fp32 [B, V], out int32 [B] (device, 4-byte aligned).  top_k is clipped to V.
 * Errors: FLINT_ERR_INVALID_ARG for null pointers, B or V <= 0, top_k < 1,
 * temperature not > 0 and finite, top_p outside (0, 1]; FLINT_ERR_UNSUPPORTED for
 * top_k > FLINT_MAX_SAMPLE_TOP_K.  No workspace.
 * -------------------------------------------------------------------------- */
#define FLINT_MAX_SAMPLE_TOP_K 32
flint_status flint_sample_logits(const float* logits, int B, int V, float temperature, int top_k,
                                 float top_p, const float* uniforms, int32_t* out,
                                 flint_stream stream);

enum {
  FLINT_OP_QUANTIZE = 0,
  FLINT_OP_MOE_DECODE = 1,
  FLINT_OP_MOE_PREFILL = 2,
  FLINT_OP_LM_HEAD = 3
};

/* Workspace bytes for an op.  Arguments that an op does not use are ignored:
 *   QUANTIZE:    n_tokens = n_mat
 *   MOE_DECODE:  hidden, n_experts, top_k, width, shared_width (also for
 *                flint_decode_tokens; any number of tokens and layers)
 *   MOE_PREFILL: hidden, n_experts, top_k, width, shared_width, n_tokens = T
 *   LM_HEAD:     hidden, vocab, n_tokens = B                                  */
size_t flint_workspace_bytes(int op, int hidden, int n_experts, int top_k, int width,
                             int shared_width, int vocab, int n_tokens);

/* Synchronises `stream`, returns the device status word (FLINT_OK if no device
 * condition was raised since the last read) and clears it. */
flint_status flint_last_device_status(flint_stream stream);

/* A static description of a status code. */
const char* flint_status_string(flint_status status);

/* Library version string. */
const char* flint_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FLINT_H */
