// api.cu -- the extern "C" entry points declared in include/flint.h: argument checks on
// the host (nothing is enqueued when a check fails), workspace carving, launches.
#include <atomic>
#include <cmath>
#include <cstring>

#include "../../include/flint.h"
#include "launch.h"

namespace {

using flint::NVPtr;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
// Natural alignment of a scalar element (outputs written one element at a time).
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

// Sizes the GEMV lane layout supports: a power of two from 32 to FLINT_MAX_HIDDEN.
inline bool gemv_width_ok(int k) {
  return k >= 32 && k <= FLINT_MAX_HIDDEN && (k & (k - 1)) == 0;
}

flint_status check_nvfp4(const flint_nvfp4& m, int n_mat, int rows, int cols) {
  if (!m.codes || !m.scales || !m.tensor_scale) return FLINT_ERR_INVALID_ARG;
  if (!aligned16(m.codes) || !aligned16(m.scales) || (reinterpret_cast<uintptr_t>(m.tensor_scale) & 3u))
    return FLINT_ERR_ALIGNMENT;
  if (m.n_mat != n_mat || m.rows != rows || m.cols != cols) return FLINT_ERR_SHAPE;
  return FLINT_OK;
}

// A dense SwiGLU layer: no router and no routed experts, the block in sh_* (flint.h).
inline bool is_dense(const flint_moe_layer* L) {
  return L->n_experts == 0 && L->top_k == 0 && L->expert_width == 0;
}

flint_status check_layer(const flint_moe_layer* L) {
  if (!L) return FLINT_ERR_INVALID_ARG;
  if (L->router_score != FLINT_ROUTER_SOFTMAX && L->router_score != FLINT_ROUTER_SIGMOID)
    return FLINT_ERR_INVALID_ARG;
  if (is_dense(L)) {
    if (L->hidden <= 0 || L->shared_width <= 0) return FLINT_ERR_INVALID_ARG;
    if (L->hidden % 32 || L->shared_width % 64) return FLINT_ERR_SHAPE;
    if (!gemv_width_ok(L->hidden) || L->shared_width > 8 * FLINT_MAX_HIDDEN) return FLINT_ERR_UNSUPPORTED;
    const int H = L->hidden, Fs = L->shared_width;
    flint_status s;
    if ((s = check_nvfp4(L->sh_gate, 1, Fs, H)) != FLINT_OK) return s;
    if ((s = check_nvfp4(L->sh_up, 1, Fs, H)) != FLINT_OK) return s;
    if ((s = check_nvfp4(L->sh_down, 1, H, Fs)) != FLINT_OK) return s;
    return FLINT_OK;
  }
  if (L->hidden <= 0 || L->n_experts <= 0 || L->top_k <= 0 || L->expert_width <= 0 ||
      L->shared_width <= 0)
    return FLINT_ERR_INVALID_ARG;
  if (L->top_k > L->n_experts) return FLINT_ERR_INVALID_ARG;
  if (L->router_score != FLINT_ROUTER_SOFTMAX && L->router_score != FLINT_ROUTER_SIGMOID)
    return FLINT_ERR_INVALID_ARG;
  if (L->top_k > FLINT_MAX_TOP_K || L->n_experts > FLINT_MAX_EXPERTS) return FLINT_ERR_UNSUPPORTED;
  if (L->hidden % 32 || L->expert_width % 32 || L->shared_width % 32) return FLINT_ERR_SHAPE;
  if (!gemv_width_ok(L->hidden) || !gemv_width_ok(L->expert_width) ||
      !gemv_width_ok(L->shared_width))
    return FLINT_ERR_UNSUPPORTED;
  if (!L->router_w) return FLINT_ERR_INVALID_ARG;
  if (!aligned16(L->router_w) || (L->router_bias && !aligned16(L->router_bias)))
    return FLINT_ERR_ALIGNMENT;
  const int H = L->hidden, E = L->n_experts, F = L->expert_width, Fs = L->shared_width;
  flint_status s;
  if ((s = check_nvfp4(L->gate, E, F, H)) != FLINT_OK) return s;
  if ((s = check_nvfp4(L->up, E, F, H)) != FLINT_OK) return s;
  if ((s = check_nvfp4(L->down, E, H, F)) != FLINT_OK) return s;
  if ((s = check_nvfp4(L->sh_gate, 1, Fs, H)) != FLINT_OK) return s;
  if ((s = check_nvfp4(L->sh_up, 1, Fs, H)) != FLINT_OK) return s;
  if ((s = check_nvfp4(L->sh_down, 1, H, Fs)) != FLINT_OK) return s;
  return FLINT_OK;
}

NVPtr nv(const flint_nvfp4& m) { return NVPtr{m.codes, m.scales, m.tensor_scale}; }

// The decode kernel's view of a layer (its pass plan is filled by decode_plan_layer).
flint::DecLayer dec_layer(const flint_moe_layer& L) {
  flint::DecLayer d;
  std::memset(&d, 0, sizeof(d));
  d.router_w = static_cast<const uint16_t*>(L.router_w);
  d.router_bias = L.router_bias;
  d.gate = nv(L.gate); d.up = nv(L.up); d.down = nv(L.down);
  d.sh_gate = nv(L.sh_gate); d.sh_up = nv(L.sh_up); d.sh_down = nv(L.sh_down);
  d.E = L.n_experts; d.K = L.top_k; d.F = L.expert_width; d.Fs = L.shared_width;
  d.score = L.router_score;
  return d;
}

// Bound of every device-side wait (flint_set_wait_limit_ns) and the armed test aid of
// flint_debug_hold_next_launch (per host thread, consumed by the next launch).
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
thread_local int t_hold = 0;

flint_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FLINT_OK : FLINT_ERR_CUDA; }

}  // namespace

extern "C" {

const char* flint_version(void) { return "flint-b300 0.1 (sm_103a)"; }

const char* flint_status_string(flint_status s) {
  switch (s) {
    case FLINT_OK: return "ok";
    case FLINT_ERR_INVALID_ARG: return "invalid argument";
    case FLINT_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FLINT_ERR_SHAPE: return "shape mismatch or size not a multiple of 32";
    case FLINT_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case FLINT_ERR_NONFINITE: return "non-finite value in quantised weights";
    case FLINT_ERR_TIMEOUT: return "a bounded device wait expired";
    case FLINT_ERR_CUDA: return "CUDA runtime error";
    case FLINT_ERR_UNSUPPORTED: return "size not supported by this build";
  }
  return "unknown status";
}

size_t flint_workspace_bytes(int op, int hidden, int n_experts, int top_k, int width,
                             int shared_width, int vocab, int n_tokens) {
  switch (op) {
    case FLINT_OP_QUANTIZE:
      return ((size_t)(n_tokens > 0 ? n_tokens : 1) * sizeof(unsigned int) + 255) & ~(size_t)255;
    case FLINT_OP_MOE_DECODE:
      (void)n_experts; (void)top_k; (void)width; (void)shared_width;
      return flint::decode_workspace_bytes(hidden);
    case FLINT_OP_LM_HEAD:
      return flint::lm_head_workspace_bytes(hidden, vocab, n_tokens);
    case FLINT_OP_MOE_PREFILL:
      return flint::prefill_workspace_bytes(hidden, n_experts, top_k, width, shared_width,
                                            n_tokens);
  }
  return 0;
}

flint_status flint_quantize_nvfp4(const void* w_bf16, int n_mat, int rows, int cols,
                                  uint8_t* codes, uint8_t* scales, float* tensor_scale,
                                  void* ws, size_t ws_bytes, flint_stream stream) {
  if (!w_bf16 || !codes || !scales || !tensor_scale || !ws) return FLINT_ERR_INVALID_ARG;
  if (n_mat <= 0 || rows <= 0 || cols <= 0) return FLINT_ERR_INVALID_ARG;
  if (cols % 32) return FLINT_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(codes) || !aligned16(scales) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u))
    return FLINT_ERR_ALIGNMENT;
  if (!aligned256(ws) || ws_bytes < flint_workspace_bytes(FLINT_OP_QUANTIZE, 0, 0, 0, 0, 0, 0, n_mat))
    return FLINT_ERR_WORKSPACE;
  return from_cuda(flint::launch_quantize(static_cast<const uint16_t*>(w_bf16), n_mat, rows, cols,
                                          codes, scales, tensor_scale, ws,
                                          static_cast<cudaStream_t>(stream)));
}

flint_status flint_dequantize_nvfp4(const flint_nvfp4* m, float* out, flint_stream stream) {
  if (!m || !out) return FLINT_ERR_INVALID_ARG;
  if (m->n_mat <= 0 || m->rows <= 0 || m->cols <= 0) return FLINT_ERR_INVALID_ARG;
  if (m->cols % 32) return FLINT_ERR_SHAPE;
  flint_status s = check_nvfp4(*m, m->n_mat, m->rows, m->cols);
  if (s != FLINT_OK) return s;
  if (!aligned16(out)) return FLINT_ERR_ALIGNMENT;
  return from_cuda(flint::launch_dequantize(m->codes, m->scales, m->tensor_scale, m->n_mat,
                                            m->rows, m->cols, out,
                                            static_cast<cudaStream_t>(stream)));
}

// Sampling options of flint_decode_tokens_sample (checked by the caller).
struct SampleOpts {
  float temp, top_p;
  int top_k;
  const float* uniforms;
  int32_t* tokens;
};

static flint_status decode_tokens_impl(const flint_moe_layer* layers, int n_layers,
                                       const flint_nvfp4* head, const void* x_bf16,
                                       const float* residual, int T, float rms_eps, float* out,
                                       void* x_out_bf16, float* logits, int32_t* argmax,
                                       int32_t* topk_idx, float* topk_w, void* x_trace_bf16,
                                       float* h_trace, void* ws, size_t ws_bytes,
                                       flint_stream stream, const SampleOpts* smp = nullptr) {
  if (!layers || !x_bf16 || !ws) return FLINT_ERR_INVALID_ARG;
  if (n_layers <= 0 || T <= 0) return FLINT_ERR_INVALID_ARG;
  if (n_layers > FLINT_MAX_LAYERS) return FLINT_ERR_UNSUPPORTED;
  if (!(rms_eps >= 0.f)) return FLINT_ERR_INVALID_ARG;
  const int H = layers[0].hidden;
  for (int l = 0; l < n_layers; ++l) {
    flint_status s = check_layer(&layers[l]);
    if (s != FLINT_OK) return s;
    if (layers[l].hidden != H) return FLINT_ERR_SHAPE;
  }
  if (head) {
    if (head->n_mat != 1 || head->cols != H || head->rows <= 0) return FLINT_ERR_SHAPE;
    flint_status s = check_nvfp4(*head, 1, head->rows, head->cols);
    if (s != FLINT_OK) return s;
  } else if (logits || argmax || smp) {
    return FLINT_ERR_INVALID_ARG;
  }
  if (!aligned16(x_bf16) || (residual && !aligned4(residual)) || (out && !aligned4(out)) ||
      (x_out_bf16 && !aligned16(x_out_bf16)) || (logits && !aligned4(logits)) ||
      (argmax && !aligned4(argmax)) || (topk_idx && !aligned4(topk_idx)) ||
      (topk_w && !aligned4(topk_w)) || (x_trace_bf16 && !aligned16(x_trace_bf16)) ||
      (h_trace && !aligned16(h_trace)))
    return FLINT_ERR_ALIGNMENT;
  if (!aligned256(ws) || ws_bytes < flint::decode_workspace_bytes(H)) return FLINT_ERR_WORKSPACE;
  const int NC = flint::decode_clusters();
  if (NC < 1) return FLINT_ERR_CUDA;
  // Large (layer table), so not on the stack; one per host thread, so concurrent calls
  // from several threads never share it.  The launch copies it into the kernel's
  // parameters, so it is free again as soon as launch_decode returns.
  thread_local flint::DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  int Emax = 0, Kmax = 0;
  for (int l = 0; l < n_layers; ++l) {
    a.layer[l] = dec_layer(layers[l]);
    if (!flint::decode_plan_layer(a.layer[l], H, NC)) return FLINT_ERR_UNSUPPORTED;
    Emax = layers[l].n_experts > Emax ? layers[l].n_experts : Emax;
    Kmax = layers[l].top_k > Kmax ? layers[l].top_k : Kmax;
  }
  a.H = H; a.L = n_layers; a.T = T; a.NC = NC;
  a.RR = flint::decode_router_rows(Emax);
  a.Emax = flint::kDecCluster * a.RR;
  a.Kmax = Kmax;
  a.eps = rms_eps;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  a.hold = t_hold == 1 ? 1 : 0;
  if (t_hold == 1) t_hold = 0;
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.residual = residual;
  a.out = out;
  a.x_out = static_cast<uint16_t*>(x_out_bf16);
  if (head) {
    a.head = nv(*head);
    a.V = head->rows;
  }
  a.logits = logits;
  a.argmax = argmax;
  a.idx_out = topk_idx;
  a.w_out = topk_w;
  a.x_trace = static_cast<uint16_t*>(x_trace_bf16);
  a.h_trace = h_trace;
  if (smp) {
    // each CTA keeps its rows' logits in shared memory: at most 2048 rows per CTA
    if ((head->rows + NC * flint::kDecCluster - 1) / (NC * flint::kDecCluster) > 2048)
      return FLINT_ERR_UNSUPPORTED;
    a.temp = smp->temp;
    a.top_p = smp->top_p;
    a.top_k = smp->top_k < head->rows ? smp->top_k : head->rows;
    a.uniforms = smp->uniforms;
    a.tokens = smp->tokens;
  }
  flint::decode_carve(a, ws);
  return from_cuda(flint::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

flint_status flint_decode_tokens(const flint_moe_layer* layers, int n_layers,
                                 const flint_nvfp4* head, const void* x_bf16,
                                 const float* residual, int T, float rms_eps, float* out,
                                 void* x_out_bf16, float* logits, int32_t* argmax,
                                 int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                                 flint_stream stream) {
  return decode_tokens_impl(layers, n_layers, head, x_bf16, residual, T, rms_eps, out,
                            x_out_bf16, logits, argmax, topk_idx, topk_w, nullptr, nullptr, ws,
                            ws_bytes, stream);
}

flint_status flint_decode_tokens_sample(const flint_moe_layer* layers, int n_layers,
                                        const flint_nvfp4* head, const void* x_bf16,
                                        const float* residual, int T, float rms_eps,
                                        float temperature, int top_k, float top_p,
                                        const float* uniforms, int32_t* tokens, float* out,
                                        void* x_out_bf16, float* logits, int32_t* argmax,
                                        int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                                        flint_stream stream) {
  if (!head || !uniforms || !tokens) return FLINT_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return FLINT_ERR_INVALID_ARG;
  if (!(top_p > 0.f && top_p <= 1.f) || top_k < 1) return FLINT_ERR_INVALID_ARG;
  if (top_k > FLINT_MAX_SAMPLE_TOP_K) return FLINT_ERR_UNSUPPORTED;
  if (!aligned4(uniforms) || !aligned4(tokens)) return FLINT_ERR_ALIGNMENT;
  const SampleOpts smp{temperature, top_p, top_k, uniforms, tokens};
  return decode_tokens_impl(layers, n_layers, head, x_bf16, residual, T, rms_eps, out,
                            x_out_bf16, logits, argmax, topk_idx, topk_w, nullptr, nullptr, ws,
                            ws_bytes, stream, &smp);
}

flint_status flint_decode_tokens_trace(const flint_moe_layer* layers, int n_layers,
                                       const flint_nvfp4* head, const void* x_bf16,
                                       const float* residual, int T, float rms_eps, float* out,
                                       void* x_out_bf16, float* logits, int32_t* argmax,
                                       int32_t* topk_idx, float* topk_w, void* x_trace_bf16,
                                       float* h_trace, void* ws, size_t ws_bytes,
                                       flint_stream stream) {
  return decode_tokens_impl(layers, n_layers, head, x_bf16, residual, T, rms_eps, out,
                            x_out_bf16, logits, argmax, topk_idx, topk_w, x_trace_bf16, h_trace,
                            ws, ws_bytes, stream);
}

flint_status flint_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns ? (unsigned long long)ns : 2000000000ull, std::memory_order_relaxed);
  return FLINT_OK;
}

flint_status flint_debug_hold_next_launch(int what) {
  if (what < 0 || what > 2) return FLINT_ERR_INVALID_ARG;
  t_hold = what;
  return FLINT_OK;
}

flint_status flint_moe_decode(const flint_moe_layer* L, const void* x_bf16, const float* residual,
                              float* out, void* x_next_bf16, float rms_eps, int32_t* topk_idx,
                              float* topk_w, int B, void* ws, size_t ws_bytes,
                              flint_stream stream) {
  if (!L || !out) return FLINT_ERR_INVALID_ARG;
  if (B <= 0) return FLINT_ERR_INVALID_ARG;
  if (B > FLINT_MAX_DECODE_TOKENS) return FLINT_ERR_UNSUPPORTED;
  return decode_tokens_impl(L, 1, nullptr, x_bf16, residual, B, rms_eps, out, x_next_bf16,
                            nullptr, nullptr, topk_idx, topk_w, nullptr, nullptr, ws, ws_bytes,
                            stream);
}

flint_status flint_nvfp4_mma_scales(const flint_nvfp4* m, uint8_t* scales_mma,
                                    flint_stream stream) {
  if (!m || !scales_mma) return FLINT_ERR_INVALID_ARG;
  if (m->n_mat <= 0 || m->rows <= 0 || m->cols <= 0) return FLINT_ERR_INVALID_ARG;
  if (m->rows % 128 || m->cols % 64) return FLINT_ERR_SHAPE;
  if (!m->scales) return FLINT_ERR_INVALID_ARG;
  if (!aligned16(m->scales) || !aligned16(scales_mma)) return FLINT_ERR_ALIGNMENT;
  return from_cuda(flint::launch_mma_scales(m->scales, m->n_mat, m->rows, m->cols, scales_mma,
                                            static_cast<cudaStream_t>(stream)));
}

flint_status flint_bench_fp4_mma(int mode, int iters, int ctas, unsigned long long* cycles,
                                 flint_stream stream) {
  if (mode < 0 || mode > 6 || iters <= 0 || ctas <= 0 || !cycles) return FLINT_ERR_INVALID_ARG;
  if (!aligned16(cycles)) return FLINT_ERR_ALIGNMENT;
  return from_cuda(flint::launch_fp4_mma_bench(mode, iters, ctas, cycles, static_cast<cudaStream_t>(stream)));
}

flint_status flint_lm_head(const flint_nvfp4* W, const void* x_bf16, float* logits,
                           int32_t* argmax, int B, void* ws, size_t ws_bytes,
                           flint_stream stream) {
  if (!W || !x_bf16 || !ws) return FLINT_ERR_INVALID_ARG;
  if (!logits && !argmax) return FLINT_ERR_INVALID_ARG;
  if (B <= 0) return FLINT_ERR_INVALID_ARG;
  if (B > FLINT_MAX_DECODE_TOKENS) return FLINT_ERR_UNSUPPORTED;
  if (W->n_mat != 1 || W->rows <= 0 || W->cols <= 0) return FLINT_ERR_SHAPE;
  flint_status s = check_nvfp4(*W, 1, W->rows, W->cols);
  if (s != FLINT_OK) return s;
  if (W->cols % 128) return FLINT_ERR_SHAPE;
  if (!gemv_width_ok(W->cols)) return FLINT_ERR_UNSUPPORTED;
  if (!aligned16(x_bf16) || (logits && !aligned4(logits)) || (argmax && !aligned4(argmax)))
    return FLINT_ERR_ALIGNMENT;
  if (!aligned256(ws) ||
      ws_bytes < flint_workspace_bytes(FLINT_OP_LM_HEAD, W->cols, 0, 0, 0, 0, W->rows, B))
    return FLINT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return FLINT_ERR_CUDA;
  return from_cuda(flint::launch_lm_head(W->codes, W->scales, W->tensor_scale, W->rows, W->cols,
                                         static_cast<const uint16_t*>(x_bf16), B, logits, argmax,
                                         ws, st));
}

flint_status flint_sample_logits(const float* logits, int B, int V, float temperature, int top_k,
                                 float top_p, const float* uniforms, int32_t* out,
                                 flint_stream stream) {
  if (!logits || !uniforms || !out) return FLINT_ERR_INVALID_ARG;
  if (B <= 0 || V <= 0 || top_k < 1) return FLINT_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return FLINT_ERR_INVALID_ARG;
  if (!(top_p > 0.f) || top_p > 1.f) return FLINT_ERR_INVALID_ARG;
  if (top_k > FLINT_MAX_SAMPLE_TOP_K) return FLINT_ERR_UNSUPPORTED;
  if (!aligned4(logits) || !aligned4(uniforms) || !aligned4(out)) return FLINT_ERR_ALIGNMENT;
  return from_cuda(flint::launch_sample(logits, B, V, temperature, top_k, top_p, uniforms, out,
                                        static_cast<cudaStream_t>(stream)));
}

flint_status flint_moe_prefill(const flint_moe_layer* L, const void* x_bf16, float* out,
                               int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                               int32_t* pair_order, int T, void* ws, size_t ws_bytes,
                               flint_stream stream) {
  if (L && is_dense(L)) return FLINT_ERR_UNSUPPORTED;     // prompt path: MoE layers only
  flint_status s = check_layer(L);
  if (s != FLINT_OK) return s;
  if (!x_bf16 || !out || !ws) return FLINT_ERR_INVALID_ARG;
  if (T <= 0) return FLINT_ERR_INVALID_ARG;
  if (!flint::prefill_shape_ok(L->hidden, L->n_experts, L->top_k, L->expert_width, L->shared_width))
    return FLINT_ERR_UNSUPPORTED;
  for (int i = 0; i < 6; ++i) {
    if (!L->mma_scales[i]) return FLINT_ERR_INVALID_ARG;
    if (!aligned16(L->mma_scales[i])) return FLINT_ERR_ALIGNMENT;
  }
  if (!aligned16(x_bf16) || !aligned16(out) || (topk_idx && !aligned4(topk_idx)) ||
      (topk_w && !aligned4(topk_w)) || (expert_counts && !aligned4(expert_counts)) ||
      (pair_order && !aligned4(pair_order)))
    return FLINT_ERR_ALIGNMENT;
  if (!aligned256(ws) ||
      ws_bytes < flint_workspace_bytes(FLINT_OP_MOE_PREFILL, L->hidden, L->n_experts, L->top_k,
                                       L->expert_width, L->shared_width, 0, T))
    return FLINT_ERR_WORKSPACE;
  flint::PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.H = L->hidden; a.E = L->n_experts; a.K = L->top_k; a.F = L->expert_width;
  a.Fs = L->shared_width; a.T = T;
  a.router_w = static_cast<const uint16_t*>(L->router_w);
  a.router_bias = L->router_bias;
  a.router_score = L->router_score;
  a.gate = nv(L->gate); a.up = nv(L->up); a.down = nv(L->down);
  a.sh_gate = nv(L->sh_gate); a.sh_up = nv(L->sh_up); a.sh_down = nv(L->sh_down);
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.out = out;
  a.idx_out = topk_idx; a.w_out = topk_w;
  a.counts_out = expert_counts; a.order_out = pair_order;
  for (int i = 0; i < 6; ++i) a.sf[i] = L->mma_scales[i];
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  a.hold = t_hold == 2 ? 1 : 0;
  if (t_hold == 2) t_hold = 0;
  return from_cuda(flint::launch_prefill(a, ws, static_cast<cudaStream_t>(stream)));
}

flint_status flint_last_device_status(flint_stream stream) {
  unsigned int v = 0;
  cudaError_t e = flint::read_and_clear_status(&v, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FLINT_ERR_CUDA;
  return static_cast<flint_status>(v);
}

}  // extern "C"
