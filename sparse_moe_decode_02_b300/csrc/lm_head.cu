// lm_head.cu -- NVFP4 output head: logits = W x, argmax (ties to the lower index).
//
// The head is 2,048 -> 150,144, untied and quantised to 4 bits ("Flint: 125 tokens a
// second is what 2.5B active parameters buy at 273 GB/s", sections "The shape, read
// from the headers" and "Why active parameters set the speed").  The vocabulary is
// split over a grid of 2 CTAs per SM; each warp streams rows with 128-bit loads and
// NR rows in flight, keeps a running (max, index) per token, and the CTA's best goes to
// the workspace; the last CTA to finish reduces those to the argmax.  Up to two tokens
// are held in registers per pass; larger batches take ceil(B/2) passes.
#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kHeadWarps = 8;
constexpr int kHeadThreads = 32 * kHeadWarps;
constexpr int kHeadNR = 4;   // rows in flight per slice

struct HeadArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tsc;
  int V, H, B, b0;        // tokens [b0, b0 + NT) in this pass
  const uint16_t* x;
  float* logits;          // [B][V] or null
  int32_t* argmax;        // [B] or null
  float* best_v;          // ws [grid][FLINT_MAX_DECODE_TOKENS]
  int* best_i;            // ws [grid][FLINT_MAX_DECODE_TOKENS]
  unsigned int* counter;  // ws, zero between launches
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <int CPL, int NT>
__global__ void __launch_bounds__(kHeadThreads, 2) k_lm_head(HeadArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = a.H / (32 * CPL);
  const int RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int gwarp = blockIdx.x * kHeadWarps + warp, nwarps = gridDim.x * kHeadWarps;
  const size_t cb = a.H / 2, sb = a.H / 16;
  const float tsc = a.tsc[0];
  XStage<CPL, 1> xs[NT];
  const int nt = min(NT, a.B - a.b0);
#pragma unroll
  for (int t = 0; t < NT; ++t)
    stage_bf16<CPL>(xs[t], nullptr, a.x + (size_t)(a.b0 + (t < nt ? t : 0)) * a.H, sl, LPR);
  float bv[NT];
  int bi[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) { bv[t] = -INFINITY; bi[t] = 0x7FFFFFFF; }
  const int rows_per_task = RPP * kHeadNR;
  const int n_tasks = (a.V + rows_per_task - 1) / rows_per_task;
  for (int task = gwarp; task < n_tasks; task += nwarps) {
    RowRegs<CPL> r[kHeadNR];
#pragma unroll
    for (int p = 0; p < kHeadNR; ++p) {
      int row = task * rows_per_task + p * RPP + slice;
      row = row < a.V ? row : a.V - 1;
      load_row<CPL>(r[p], a.codes + row * cb, a.scales + row * sb, sl, LPR);
    }
#pragma unroll
    for (int p = 0; p < kHeadNR; ++p) {
      const int row = task * rows_per_task + p * RPP + slice;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = sum_lanes_rt(dot_row<CPL, 1>(r[p], xs[t]), LPR) * (tsc * xs[t].unscale);
        if (t < nt && row < a.V) {
          if (sl == 0 && a.logits) a.logits[(size_t)(a.b0 + t) * a.V + row] = v;
          const float vv = (v == v) ? v : -INFINITY;
          if (better(vv, row, bv[t], bi[t])) { bv[t] = vv; bi[t] = row; }
        }
      }
    }
  }
  // block reduction of the running best, per token
  __shared__ float sv[kHeadWarps][NT];
  __shared__ int si[kHeadWarps][NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float v = bv[t];
    int i = bi[t];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    if (lane == 0) { sv[warp][t] = v; si[warp][t] = i; }
  }
  __syncthreads();
  if (threadIdx.x < NT) {
    const int t = threadIdx.x;
    float v = sv[0][t];
    int i = si[0][t];
    for (int w = 1; w < kHeadWarps; ++w)
      if (better(sv[w][t], si[w][t], v, i)) { v = sv[w][t]; i = si[w][t]; }
    a.best_v[blockIdx.x * FLINT_MAX_DECODE_TOKENS + t] = v;
    a.best_i[blockIdx.x * FLINT_MAX_DECODE_TOKENS + t] = i;
  }
  // last CTA: argmax over the CTAs' bests
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < nt) {
    const int t = warp;
    float v = -INFINITY;
    int i = 0x7FFFFFFF;
    for (int c = lane; c < (int)gridDim.x; c += 32) {
      const float cv = __ldcg(a.best_v + c * FLINT_MAX_DECODE_TOKENS + t);
      const int ci = __ldcg(a.best_i + c * FLINT_MAX_DECODE_TOKENS + t);
      if (better(cv, ci, v, i)) { v = cv; i = ci; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    if (lane == 0 && a.argmax) a.argmax[a.b0 + t] = (i < a.V) ? i : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.counter = 0;
}

static int head_grid() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms * 2;
}

size_t lm_head_workspace_bytes(int H, int V, int B) {
  (void)H; (void)V; (void)B;
  const size_t grid = 2 * 1024;  // upper bound on CTAs (2 per SM)
  return grid * FLINT_MAX_DECODE_TOKENS * (sizeof(float) + sizeof(int)) + 256;
}

template <int CPL>
static cudaError_t launch_head_cpl(HeadArgs a, cudaStream_t st) {
  const int grid = head_grid();
  for (int b0 = 0; b0 < a.B; b0 += 2) {
    a.b0 = b0;
    if (a.B - b0 >= 2) k_lm_head<CPL, 2><<<grid, kHeadThreads, 0, st>>>(a);
    else k_lm_head<CPL, 1><<<grid, kHeadThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_lm_head(const uint8_t* codes, const uint8_t* scales, const float* tsc, int V,
                           int H, const uint16_t* x, int B, float* logits, int32_t* argmax,
                           void* ws, cudaStream_t st) {
  HeadArgs a;
  a.codes = codes; a.scales = scales; a.tsc = tsc; a.V = V; a.H = H; a.B = B; a.b0 = 0;
  a.x = x; a.logits = logits; a.argmax = argmax;
  char* p = static_cast<char*>(ws);
  a.counter = reinterpret_cast<unsigned int*>(p);
  p += 256;
  a.best_v = reinterpret_cast<float*>(p);
  p += (size_t)2 * 1024 * FLINT_MAX_DECODE_TOKENS * sizeof(float);
  a.best_i = reinterpret_cast<int*>(p);
  if (H <= 1024) return launch_head_cpl<1>(a, st);
  if (H <= 2048) return launch_head_cpl<2>(a, st);
  return launch_head_cpl<4>(a, st);
}

}  // namespace flint
