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

constexpr int kMaxLayers = 64;

// ------------------------------------------------------------------ persistent decode
// Clusters of kDecCluster CTAs.  In each layer a cluster runs up to kDecMaxGroups
// groups: a group is one routed expert (one part of F outputs), or a contiguous run of
// parts of the shared (or dense) expert.  The cluster's CTAs split each part's gate/up
// rows, swap the SwiGLU values, and each CTA applies the group's down columns to its own
// H/16 output rows.
constexpr int kDecCluster = 16;
constexpr int kDecMaxClusters = 8;
constexpr int kDecMaxGroups = 2;
constexpr int kDecThreads = 512;

struct DecLayer {
  const uint16_t* router_w;          // bf16 [E][H]; null for a dense layer
  const float* router_bias;          // fp32 [E] or null
  NVPtr gate, up, down;              // routed stacks [E][F][H], [E][F][H], [E][H][F]
  NVPtr sh_gate, sh_up, sh_down;     // shared (or dense) expert [1][Fs][H], [1][Fs][H], [1][H][Fs]
  int E, K, F, Fs;
  int Wsh;                           // outputs of one shared part (a divisor of Fs)
  int score;                         // FLINT_ROUTER_SOFTMAX / FLINT_ROUTER_SIGMOID
  // group g of cluster c: rank[c][g] >= 0 is the routed expert of that rank (one part);
  // -1 is parts [p0, p0 + np) of the shared expert
  signed char rank[kDecMaxClusters][kDecMaxGroups];
  unsigned char np[kDecMaxClusters][kDecMaxGroups];
  unsigned char p0[kDecMaxClusters][kDecMaxGroups];
  unsigned char n_grp[kDecMaxClusters];
  unsigned char routed[kDecMaxClusters];   // cluster computes the router and top-k
  unsigned sh_off;                   // shared groups' buffer offset in a routed cluster
  int pad_;
};

struct DecodeArgs {
  int H, L, T, V, NC, Kmax, Emax, RR;  // RR: router rows per CTA; Emax = 16 RR (logits per step)
  float eps;
  int hold;                          // test aid: CTA 0 withholds its first partial
  unsigned long long wait_ns;        // bound of every wait
  const uint16_t* x;                 // [T][H] bf16
  const float* residual;             // [T][H] or null
  float* out;                        // [T][H] or null
  uint16_t* x_out;                   // [T][H] or null
  NVPtr head;                        // codes null: no head
  float* logits;                     // [T][V] or null
  int32_t* argmax;                   // [T] or null
  int32_t* idx_out;                  // [T][L][Kmax] or null
  float* w_out;                      // [T][L][Kmax] or null
  uint16_t* x_trace;                 // [T][L][H] or null: x_l as staged
  float* h_trace;                    // [T][L][H] or null: h_l
  unsigned* sync;                    // [64]: [0] abort flag
  unsigned long long* board;         // [2][kDecMaxClusters][H] tagged partial sums
  unsigned long long* best;          // [2][kDecMaxClusters * kDecCluster][2] tagged head maxima
  // fused sampling of the head (tokens non-null): temperature, top-k (<= 32), top-p, one
  // uniform per token; board of the CTAs' candidates [2][kDecMaxClusters * kDecCluster][32][2]
  float temp, top_p;
  int top_k;
  const float* uniforms;
  int32_t* tokens;
  unsigned long long* cand;
  DecLayer layer[kMaxLayers];
};

// Host-side plan of a decode launch.
struct DecodeShape {
  int H, E, K, F, Fs;                // E = K = 0: a dense layer (its width in Fs)
};
int decode_clusters();                               // clusters the device co-schedules (0: none)
int decode_router_rows(int E);
size_t decode_workspace_bytes(int H);
size_t decode_smem_bytes(int H, int Emax);
// Checks a layer's shape and fills its pass plan; false when this build cannot run it.
bool decode_plan_layer(DecLayer& d, int H, int NC);
void decode_carve(DecodeArgs& a, void* ws);          // a.H set
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
  const uint8_t* sf[6];    // MMA scale copies: gate, up, down, sh_gate, sh_up, sh_down
  int router_score;        // FLINT_ROUTER_SOFTMAX / FLINT_ROUTER_SIGMOID
  unsigned long long wait_ns;   // bound of every device-side wait
  int hold;                     // test aid: withhold the gate/up GEMM's first stage in CTA 0
};

size_t prefill_workspace_bytes(int H, int E, int K, int F, int Fs, int T);
bool prefill_shape_ok(int H, int E, int K, int F, int Fs);
cudaError_t launch_prefill(const PrefillArgs& a, void* ws, cudaStream_t st);
cudaError_t launch_fp4_mma_bench(int mode, int iters, int ctas, unsigned long long* cycles, cudaStream_t st);
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
