// launch.h -- host-side launchers of the Flint kernels (internal to the library).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace flint {

struct NVPtr {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tsc;
};

struct LayerPtrs {
  const uint16_t* router_w;
  const float* router_bias;
  NVPtr gate, up, sh_gate, sh_up;  // the tensor scales are read from these stacks
  const uint8_t* units;           // decode units of (gate, up, down) [E][F/8][14 H]
  const uint8_t* sh_units;        // of (sh_gate, sh_up, sh_down) [1][Fs/8][14 H]
  const float* down_tsc;          // [E]
  const float* sh_down_tsc;       // [1]
  int router_score;               // FLINT_ROUTER_SOFTMAX / FLINT_ROUTER_SIGMOID
  int pad_;
};

constexpr int kMaxLayers = 64;

struct PersistArgs {
  int H, E, K, F, Fs, L, T, V;
  float eps;
  const uint16_t* x;       // [T, H] bf16
  const float* residual;   // [T, H] or null
  float* out;              // [T, H] or null
  uint16_t* x_out;         // [T, H] or null
  NVPtr head;              // codes null: no head
  float* logits;           // [T, V] or null
  int32_t* argmax;         // [T] or null
  int32_t* idx_out;        // [T, L, K] or null
  float* w_out;            // [T, L, K] or null
  // workspace
  unsigned* bar;           // grid barrier {arrivals, generation, abort}
  unsigned long long* logits_tag;   // [tag_copies][tag_stride] {logit bits, step + 1}
  int tag_copies, tag_stride;
  float* acc;              // [2][copies][H] residual ping-pong
  float* best_v;           // [grid]
  int* best_i;             // [grid]
  int max_router_rows;     // per-CTA buffer sizes (decode_plan)
  int max_shared_units;
  int max_routed_units;
  LayerPtrs layer[kMaxLayers];
};

// Per-CTA work bounds and shared memory of the persistent decode on G CTAs.
struct DecodePlan {
  int router_rows, shared_units, routed_units;
  size_t smem;
  bool ok;
};
DecodePlan decode_plan(int H, int E, int K, int F, int Fs, int G);

// Workspace of the persistent decode with `copies` copies of the logit board;
// decode_tag_copies(E) is the number a full workspace holds.
size_t decode_workspace_bytes(int H, int E, int copies);
int decode_tag_copies(int E);
int decode_grid();                                   // CTAs of the persistent kernel
void decode_carve(PersistArgs& a, void* ws);          // a.H, a.E, a.tag_copies set
cudaError_t launch_persistent(const PersistArgs& a, cudaStream_t st);
cudaError_t launch_unit_pack(const NVPtr& gate, const NVPtr& up, const NVPtr& down, int n_mat, int H,
                             int F, uint8_t* units, cudaStream_t st);

struct PrefillArgs {
  int H, E, K, F, Fs, T;
  const uint16_t* router_w;
  const float* router_bias;
  NVPtr gate, up, down, sh_gate, sh_up, sh_down;
  const uint16_t* x;
  float* out;
  int32_t* idx_out;
  float* w_out;
  int32_t* counts_out;
  int32_t* order_out;
  const uint8_t* sf[6];    // MMA scale copies: gate, up, down, sh_gate, sh_up, sh_down
  int router_score;        // FLINT_ROUTER_SOFTMAX / FLINT_ROUTER_SIGMOID
};

size_t prefill_workspace_bytes(int H, int E, int K, int F, int Fs, int T);
bool prefill_shape_ok(int H, int E, int K, int F, int Fs);
cudaError_t launch_prefill(const PrefillArgs& a, void* ws, cudaStream_t st);
cudaError_t launch_mma_scales(const uint8_t* scales, int n_mat, int rows, int cols, uint8_t* out,
                              cudaStream_t st);

size_t lm_head_workspace_bytes(int H, int V, int B);
cudaError_t launch_lm_head(const uint8_t* codes, const uint8_t* scales, const float* tsc, int V,
                           int H, const uint16_t* x, int B, float* logits, int32_t* argmax,
                           void* ws, cudaStream_t st);

cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                          const float* uniforms, int32_t* out, cudaStream_t st);

cudaError_t launch_quantize(const uint16_t* w, int n_mat, int rows, int cols, uint8_t* codes,
                            uint8_t* scales, float* tsc, void* ws, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* tsc,
                              int n_mat, int rows, int cols, float* out, cudaStream_t st);
cudaError_t read_and_clear_status(unsigned int* out, cudaStream_t st);

}  // namespace flint
