// sample.cu -- sampling from output-head logits ("Recursive Releases Flint, a 40B MoE
// Coding Model That Runs Locally at 125 Tokens per Second", section "How does Flint
// perform on coding benchmarks?": temperature 1.0, top-p 0.95, top-k 20).
//
// One CTA per row of logits:
//   1. every warp takes the largest order key of its strided share (NaN reads as
//      -inf); the top_k-th largest of these 32 maxima is at or below the top_k-th
//      largest logit (at least top_k warps hold a logit at or above it);
//   2. the logits at or above it (typically a few more than top_k) are ranked exactly
//      by (logit descending, lower index first).  When ties leave more than kMaxCand of
//      them, a radix select (four 8-bit histogram passes) finds the top_k-th largest
//      key instead, and the lowest-index logits equal to it complete the set;
//   3. one warp computes p_i = exp((l_i - l_0) / T) over the top_k, the shortest
//      prefix whose p sum reaches top_p, and the draw from the renormalised prefix for
//      the caller's u.
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

// Candidates by radix select (any input): the K-th largest key exactly by four 8-bit
// histogram passes, then every key above it and the lowest-index keys equal to it.
// Leaves the K candidates, unordered, in s_ck / s_ci.
__device__ void radix_candidates(const float* row, int V, int K, unsigned* s_hist, unsigned* s_wsum,
                                 int* s_nc, unsigned* s_ck, int* s_ci, unsigned* s_sel, unsigned* s_need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned prefix = 0u, mask = 0u, need = (unsigned)K;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s_hist[tid] = 0u;
    __syncthreads();
#pragma unroll 4
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
          if (acc + c[j] >= need) { *s_sel = 8u * lane + j; *s_need = need - acc; break; }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= *s_sel << shift;
    mask |= 255u << shift;
    need = *s_need;
    __syncthreads();
  }
  const unsigned thr = prefix;          // K - need keys lie above it
  if (tid == 0) *s_nc = 0;
  __syncthreads();
  const int chunk = (V + kThreads - 1) / kThreads;
  const int v0 = min(V, tid * chunk), v1 = min(V, v0 + chunk);
  unsigned eq = 0u;
#pragma unroll 1
  for (int v = v0; v < v1; ++v) {
    const unsigned key = skey(row[v]);
    if (key > thr) {
      const int slot = atomicAdd(s_nc, 1);
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
      const int slot = atomicAdd(s_nc, 1);
      s_ck[slot] = thr;
      s_ci[slot] = v;
      ++rank;
    }
  }
  __syncthreads();
}

constexpr int kMaxCand = 2048;   // candidates the fast path ranks directly

__global__ void __launch_bounds__(kThreads) k_sample(const float* __restrict__ logits, int V, float temp,
                                                    int K, float top_p, const float* __restrict__ uniforms,
                                                    int32_t* __restrict__ out) {
  __shared__ unsigned s_hist[256];
  __shared__ unsigned s_sel, s_need;
  __shared__ unsigned s_wsum[kThreads / 32];
  __shared__ int s_nc;
  __shared__ unsigned s_ck[32];
  __shared__ int s_ci[32];
  __shared__ unsigned s_wm[kThreads / 32];
  __shared__ unsigned s_fk[kMaxCand];
  __shared__ int s_fi[kMaxCand];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = logits + (size_t)blockIdx.x * V;

  // ---- 1. fast path: the K-th largest of the warps' maxima bounds the K-th largest
  // logit from below (at least K warps hold a logit at or above it).  Rows whose
  // start and length are multiples of 4 floats are read as float4.
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  unsigned tmax = 0u;                    // 0: no logit (every key is >= 1)
  if (vec) {
#pragma unroll 4
    for (int q = tid; q < V / 4; q += kThreads) {
      const float4 f = row4[q];
      tmax = max(tmax, max(max(skey(f.x), skey(f.y)), max(skey(f.z), skey(f.w))));
    }
  } else {
#pragma unroll 8
    for (int v = tid; v < V; v += kThreads) tmax = max(tmax, skey(row[v]));
  }
  const unsigned wmax = __reduce_max_sync(0xffffffffu, tmax);
  if (lane == 0) s_wm[warp] = wmax;
  if (tid == 0) s_nc = 0;
  __syncthreads();
  if (warp == 0) {
    // rank of warp `lane`'s maximum among the 32 (ties to the lower warp); K <= 32
    const unsigned m = s_wm[lane];
    int rk = 0;
#pragma unroll
    for (int j = 0; j < kThreads / 32; ++j) rk += before(s_wm[j], j, m, lane) ? 1 : 0;
    if (rk == K - 1) s_sel = m;
  }
  __syncthreads();
  const unsigned thr = s_sel;
  if (vec) {
#pragma unroll 4
    for (int q = tid; q < V / 4; q += kThreads) {
      const float4 f = row4[q];
      const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned key = skey(e[j]);
        if (key >= thr) {
          const int slot = atomicAdd(&s_nc, 1);
          if (slot < kMaxCand) { s_fk[slot] = key; s_fi[slot] = 4 * q + j; }
        }
      }
    }
  } else {
#pragma unroll 8
    for (int v = tid; v < V; v += kThreads) {
      const unsigned key = skey(row[v]);
      if (key >= thr) {
        const int slot = atomicAdd(&s_nc, 1);
        if (slot < kMaxCand) { s_fk[slot] = key; s_fi[slot] = v; }
      }
    }
  }
  __syncthreads();
  const int n = s_nc;
  if (n <= kMaxCand) {
    // exact ranks among the candidates; the K best go to s_ck / s_ci in rank order
#pragma unroll 1
    for (int j = tid; j < n; j += kThreads) {
      const unsigned kj = s_fk[j];
      const int ij = s_fi[j];
      int r = 0;
#pragma unroll 4
      for (int i = 0; i < n; ++i) r += before(s_fk[i], s_fi[i], kj, ij) ? 1 : 0;
      if (r < K) { s_ck[r] = kj; s_ci[r] = ij; }
    }
    __syncthreads();
  } else {
    __syncthreads();
    radix_candidates(row, V, K, s_hist, s_wsum, &s_nc, s_ck, s_ci, &s_sel, &s_need);
  }

  // ---- 2. sort (a no-op after the fast path), probabilities, top-p prefix, draw (warp 0)
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
  // A +inf logit holds all the probability (the limit of the softmax); among several the
  // lowest index, i.e. rank 0, is taken, as the top-k orders ties.  All -inf: rank 0 too.
  int pick_lane = 0;
  if (l0 != -INFINITY && l0 != INFINITY) {
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
