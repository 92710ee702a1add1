// sample.cu -- sampling from output-head logits ("Recursive Releases Flint, a 40B MoE
// Coding Model That Runs Locally at 125 Tokens per Second", section "How does Flint
// perform on coding benchmarks?": temperature 1.0, top-p 0.95, top-k 20).
//
// One CTA per row of logits:
//   1. the top_k-th largest order key, exactly, by a 4-pass radix select (8 bits per
//      pass, shared-memory histograms); NaN reads as -inf;
//   2. the candidates: every logit above that key, then the lowest-index logits equal
//      to it (index order from a block-wide scan of per-thread counts over contiguous
//      chunks), top_k in all;
//   3. one warp sorts them (bitonic, by logit descending, lower index first) and
//      computes p_i = exp((l_i - l_0) / T) over them, the shortest prefix whose p sum
//      reaches top_p, and the draw from the renormalised prefix for the caller's u.
#include "common.cuh"

namespace flint {
namespace smp {

constexpr int kThreads = 1024;

__device__ __forceinline__ float nan_to_ninf(float v) { return v == v ? v : -INFINITY; }
__device__ __forceinline__ unsigned skey(float v) {
  const unsigned u = __float_as_uint(nan_to_ninf(v));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);     // increasing in v; >= 1
}
__device__ __forceinline__ bool before(unsigned ka, int ia, unsigned kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kThreads) k_sample(const float* __restrict__ logits, int V, float temp,
                                                    int K, float top_p, const float* __restrict__ uniforms,
                                                    int32_t* __restrict__ out) {
  __shared__ unsigned s_hist[256];
  __shared__ unsigned s_sel, s_need;
  __shared__ unsigned s_wsum[kThreads / 32];
  __shared__ int s_nc;
  __shared__ unsigned s_ck[32];
  __shared__ int s_ci[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = logits + (size_t)blockIdx.x * V;

  // ---- 1. the K-th largest key: prefix/mask grow by 8 bits a pass; need = its rank
  // among the keys that match the prefix so far
  unsigned prefix = 0u, mask = 0u, need = (unsigned)K;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s_hist[tid] = 0u;
    __syncthreads();
#pragma unroll 1
    for (int v = tid; v < V; v += kThreads) {
      const unsigned key = skey(row[v]);
      if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins [8 l, 8 l + 8); counts above a bin come from higher bins
      unsigned c[8], sum = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = s_hist[8 * lane + j]; sum += c[j]; }
      unsigned suf = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      unsigned acc = suf - sum;
      if (acc < need && suf >= need) {
#pragma unroll 1
        for (int j = 7; j >= 0; --j) {
          if (acc + c[j] >= need) { s_sel = 8u * lane + j; s_need = need - acc; break; }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= s_sel << shift;
    mask |= 255u << shift;
    need = s_need;
    __syncthreads();
  }
  const unsigned thr = prefix;          // K - need logits lie above it

  // ---- 2. candidates: those above thr, then the `need` lowest-index ones equal to it
  if (tid == 0) s_nc = 0;
  __syncthreads();
  const int chunk = (V + kThreads - 1) / kThreads;
  const int v0 = min(V, tid * chunk), v1 = min(V, v0 + chunk);
  unsigned eq = 0u;
#pragma unroll 1
  for (int v = v0; v < v1; ++v) {
    const unsigned key = skey(row[v]);
    if (key > thr) {
      const int slot = atomicAdd(&s_nc, 1);
      s_ck[slot] = key;
      s_ci[slot] = v;
    } else if (key == thr) {
      ++eq;
    }
  }
  unsigned incl = eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned w = s_wsum[lane];
    unsigned wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_wsum[lane] = wi - w;               // equal keys in lower warps
  }
  __syncthreads();
  unsigned rank = s_wsum[warp] + incl - eq;
#pragma unroll 1
  for (int v = v0; v < v1 && rank < need; ++v) {
    if (skey(row[v]) == thr) {
      const int slot = atomicAdd(&s_nc, 1);
      s_ck[slot] = thr;
      s_ci[slot] = v;
      ++rank;
    }
  }
  __syncthreads();

  // ---- 3. sort, probabilities, top-p prefix, draw (warp 0)
  if (warp != 0) return;
  unsigned key = lane < K ? s_ck[lane] : 0u;
  int idx = lane < K ? s_ci[lane] : 0x7FFFFFFF;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned ok = __shfl_xor_sync(0xffffffffu, key, stride);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, stride);
      const bool lower = (lane & stride) == 0;
      const bool first_block = (lane & size) == 0 || size == 32;
      const bool other_first = before(ok, oi, key, idx);
      const bool take = (lower == first_block) ? other_first : (!other_first && !(ok == key && oi == idx));
      if (take) { key = ok; idx = oi; }
    }
  }
  const float l = lane < K ? nan_to_ninf(row[idx]) : -INFINITY;
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  int pick_lane = 0;
  if (l0 != -INFINITY) {
    float p = lane < K ? expf((l - l0) / temp) : 0.f;
    float z = p;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    p /= z;
    float c = p;                         // inclusive prefix sums of p in rank order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) c += t;
    }
    const unsigned reach = __ballot_sync(0xffffffffu, lane < K && c >= top_p);
    const int m = reach ? __ffs(reach) : K;
    const float zm = __shfl_sync(0xffffffffu, c, m - 1);
    const float u = uniforms[blockIdx.x];
    const unsigned hit = __ballot_sync(0xffffffffu, lane < m && u < c / zm);
    pick_lane = hit ? __ffs(hit) - 1 : m - 1;
  }
  const int pick = __shfl_sync(0xffffffffu, idx, pick_lane);
  if (lane == 0) out[blockIdx.x] = pick;
}

}  // namespace smp

cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                          const float* uniforms, int32_t* out, cudaStream_t st) {
  const int K = top_k < V ? top_k : V;
  smp::k_sample<<<B, smp::kThreads, 0, st>>>(logits, V, temperature, K, top_p, uniforms, out);
  return cudaGetLastError();
}

}  // namespace flint
