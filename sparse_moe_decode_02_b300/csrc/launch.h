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

struct DecodeArgs {
  int H, E, K, F, Fs, B;
  const uint16_t* router_w;
  const float* router_bias;
  NVPtr gate, up, down, sh_gate, sh_up, sh_down;
  const uint16_t* x;
  const float* residual;
  float* out;
  uint16_t* x_next;
  float eps;
  int32_t* idx_out;
  float* w_out;
  // workspace
  float* logits;       // [B][E]
  int32_t* sel_idx;    // [B][K]
  float* sel_w;        // [B][K]
  float* h_routed;     // [B][K][F]
  float* h_shared;     // [B][Fs]
  unsigned int* counters;  // [4], zero between launches
};

size_t decode_workspace_bytes(int H, int E, int K, int F, int Fs, int B);
void decode_carve(DecodeArgs& a, void* ws);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

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
};

size_t prefill_workspace_bytes(int H, int E, int K, int F, int Fs, int T);
cudaError_t launch_prefill(const PrefillArgs& a, void* ws, cudaStream_t st);

size_t lm_head_workspace_bytes(int H, int V, int B);
cudaError_t launch_lm_head(const uint8_t* codes, const uint8_t* scales, const float* tsc, int V,
                           int H, const uint16_t* x, int B, float* logits, int32_t* argmax,
                           void* ws, cudaStream_t st);

cudaError_t launch_quantize(const uint16_t* w, int n_mat, int rows, int cols, uint8_t* codes,
                            uint8_t* scales, float* tsc, void* ws, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* tsc,
                              int n_mat, int rows, int cols, float* out, cudaStream_t st);
cudaError_t read_and_clear_status(unsigned int* out, cudaStream_t st);

}  // namespace flint
