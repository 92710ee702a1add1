// decode.cu -- one Flint MoE layer for a few tokens (token generation).
//
// The layer ("Flint: 125 tokens a second is what 2.5B active parameters buy at 273
// GB/s", section "The shape, read from the headers"; "Recursive Releases Flint, a 40B
// MoE Coding Model That Runs Locally at 125 Tokens per Second", section "How does
// Flint's architecture work?") is three weight streams with two data dependencies:
//
//   k_router_shared  router GEMV (bf16) + the shared expert's gate/up rows (they need
//                    only x), then, in the last CTA to finish, softmax/top-k per token
//   k_routed_gateup  the selected experts' gate/up rows -> h = silu(g) * u
//   k_down_combine   down rows of the selected experts and the shared expert, combined
//                    per output row in a fixed order (deterministic, no atomics), plus
//                    the residual; the last CTA optionally writes RMSNorm(out) in bf16
//
// Every weight byte is read once per call, with coalesced 128-bit loads, by warps
// that hold the activation vector in registers (see gemv.cuh).
#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kDownRows = 8;   // output rows per CTA of k_down_combine

// All threads fence their global writes, then one atomic tells whether this CTA is the
// last of the grid to finish.  The last CTA sees every other CTA's writes.
__device__ __forceinline__ bool last_cta_done(unsigned int* counter) {
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(counter, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last;
}

// Softmax top-k of one token's logits by one warp: largest logit first, ties to the
// lower expert index; weight_i = exp(l_i - l_max) / sum_selected exp(l_j - l_max),
// which equals p_i / sum_selected p_j for the full softmax p.
__device__ void topk_warp(const DecodeArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  constexpr int kMaxPerLane = FLINT_MAX_EXPERTS / 32;
  float v[kMaxPerLane];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    float l = (e < a.E) ? __ldcg(a.logits + (size_t)b * a.E + e) : -INFINITY;
    v[i] = (l == l) ? l : -INFINITY;   // NaN never wins, but an index is always found
  }
  int sel_e[FLINT_MAX_TOP_K];
  float sel_l[FLINT_MAX_TOP_K];
  for (int s = 0; s < a.K; ++s) {
    float bv = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sel_e[s] = be;
    sel_l[s] = bv;
  }
  float p[FLINT_MAX_TOP_K];
  float z = 0.f;
  for (int s = 0; s < a.K; ++s) { p[s] = expf(sel_l[s] - sel_l[0]); z += p[s]; }
  for (int s = 0; s < a.K; ++s) {
    if (lane == s) {
      const float w = p[s] / z;
      a.sel_idx[b * a.K + s] = sel_e[s];
      a.sel_w[b * a.K + s] = w;
      if (a.idx_out) a.idx_out[b * a.K + s] = sel_e[s];
      if (a.w_out) a.w_out[b * a.K + s] = w;
    }
  }
}

// ---------------------------------------------------------------- router + shared
template <int CPL>
__global__ void __launch_bounds__(kThreads, 2) k_router_shared(DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = a.H / (32 * CPL);
  const int RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int gwarp = blockIdx.x * kWarps + warp, nwarps = gridDim.x * kWarps;
  const int n_router = (a.E + RPP - 1) / RPP;
  const int n_shared = (a.Fs + 2 * RPP - 1) / (2 * RPP);
  const size_t cb = a.H / 2, sb = a.H / 16;
  for (int b = 0; b < a.B; ++b) {
    XStage<CPL, 1> xs;
    XRawBF16<CPL> xr;
    stage_bf16<CPL>(xs, &xr, a.x + (size_t)b * a.H, sl, LPR);
    for (int t = gwarp; t < n_router + n_shared; t += nwarps) {
      if (t < n_router) {
        const int row = t * RPP + slice;
        const bool ok = row < a.E;
        RowBF16<CPL> r;
        load_row_bf16<CPL>(r, a.router_w + (size_t)(ok ? row : 0) * a.H, sl, LPR);
        float v = sum_lanes_rt(dot_row_bf16<CPL>(r, xr), LPR);
        if (ok && sl == 0)
          a.logits[(size_t)b * a.E + row] = v + (a.router_bias ? a.router_bias[row] : 0.f);
      } else {
        const int j0 = (t - n_router) * 2 * RPP + slice;
        const int j1 = j0 + RPP;
        const int r0 = j0 < a.Fs ? j0 : 0, r1 = j1 < a.Fs ? j1 : 0;
        RowRegs<CPL> g0, u0, g1, u1;
        load_row<CPL>(g0, a.sh_gate.codes + r0 * cb, a.sh_gate.scales + r0 * sb, sl, LPR);
        load_row<CPL>(u0, a.sh_up.codes + r0 * cb, a.sh_up.scales + r0 * sb, sl, LPR);
        load_row<CPL>(g1, a.sh_gate.codes + r1 * cb, a.sh_gate.scales + r1 * sb, sl, LPR);
        load_row<CPL>(u1, a.sh_up.codes + r1 * cb, a.sh_up.scales + r1 * sb, sl, LPR);
        const float gs = a.sh_gate.tsc[0] * xs.unscale, us = a.sh_up.tsc[0] * xs.unscale;
        const float vg0 = sum_lanes_rt(dot_row<CPL, 1>(g0, xs), LPR);
        const float vu0 = sum_lanes_rt(dot_row<CPL, 1>(u0, xs), LPR);
        const float vg1 = sum_lanes_rt(dot_row<CPL, 1>(g1, xs), LPR);
        const float vu1 = sum_lanes_rt(dot_row<CPL, 1>(u1, xs), LPR);
        if (sl == 0) {
          if (j0 < a.Fs) a.h_shared[(size_t)b * a.Fs + j0] = silu(vg0 * gs) * (vu0 * us);
          if (j1 < a.Fs) a.h_shared[(size_t)b * a.Fs + j1] = silu(vg1 * gs) * (vu1 * us);
        }
      }
    }
  }
  if (last_cta_done(&a.counters[0])) {
    if (warp < a.B) topk_warp(a, warp);
    __syncthreads();
    if (threadIdx.x == 0) a.counters[0] = 0;
  }
}

// ---------------------------------------------------------------- routed gate/up
template <int CPL>
__global__ void __launch_bounds__(kThreads, 2) k_routed_gateup(DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = a.H / (32 * CPL);
  const int RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int gwarp = blockIdx.x * kWarps + warp, nwarps = gridDim.x * kWarps;
  const int per_slot = (a.F + 2 * RPP - 1) / (2 * RPP);
  const size_t cb = a.H / 2, sb = a.H / 16;
  for (int b = 0; b < a.B; ++b) {
    XStage<CPL, 1> xs;
    stage_bf16<CPL>(xs, nullptr, a.x + (size_t)b * a.H, sl, LPR);
    for (int t = gwarp; t < a.K * per_slot; t += nwarps) {
      const int i = t / per_slot;
      int e = __ldcg(a.sel_idx + b * a.K + i);
      if (e < 0 || e >= a.E) { raise_status(FLINT_ERR_INVALID_ARG); e = 0; }
      const int j0 = (t % per_slot) * 2 * RPP + slice;
      const int j1 = j0 + RPP;
      const size_t r0 = (size_t)e * a.F + (j0 < a.F ? j0 : 0);
      const size_t r1 = (size_t)e * a.F + (j1 < a.F ? j1 : 0);
      RowRegs<CPL> g0, u0, g1, u1;
      load_row<CPL>(g0, a.gate.codes + r0 * cb, a.gate.scales + r0 * sb, sl, LPR);
      load_row<CPL>(u0, a.up.codes + r0 * cb, a.up.scales + r0 * sb, sl, LPR);
      load_row<CPL>(g1, a.gate.codes + r1 * cb, a.gate.scales + r1 * sb, sl, LPR);
      load_row<CPL>(u1, a.up.codes + r1 * cb, a.up.scales + r1 * sb, sl, LPR);
      const float gs = a.gate.tsc[e] * xs.unscale, us = a.up.tsc[e] * xs.unscale;
      const float vg0 = sum_lanes_rt(dot_row<CPL, 1>(g0, xs), LPR);
      const float vu0 = sum_lanes_rt(dot_row<CPL, 1>(u0, xs), LPR);
      const float vg1 = sum_lanes_rt(dot_row<CPL, 1>(g1, xs), LPR);
      const float vu1 = sum_lanes_rt(dot_row<CPL, 1>(u1, xs), LPR);
      if (sl == 0) {
        float* h = a.h_routed + ((size_t)b * a.K + i) * a.F;
        if (j0 < a.F) h[j0] = silu(vg0 * gs) * (vu0 * us);
        if (j1 < a.F) h[j1] = silu(vg1 * gs) * (vu1 * us);
      }
    }
  }
}

// ---------------------------------------------------------------- down + combine
// One pass over `nrows` output rows [n0, n0 + nrows) of one down matrix [H, Kin] with
// the staged input; writes scaled partial sums to part[0..nrows).
template <int CPL>
__device__ __forceinline__ void down_rows(const NVPtr& m, size_t mat, int H, int Kin, int n0,
                                          int nrows, const float* __restrict__ hin,
                                          float* part) {
  const int lane = threadIdx.x & 31;
  const int LPR = Kin / (32 * CPL);
  const int RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  XStage<CPL, 2> xs;
  stage_f32<CPL>(xs, hin, sl, LPR);
  const float scale = m.tsc[mat] * xs.unscale;
  const size_t cb = Kin / 2, sb = Kin / 16;
  constexpr int NP = 4;  // passes with loads in flight together
  for (int p0 = 0; p0 < nrows; p0 += NP * RPP) {
    RowRegs<CPL> r[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      int n = n0 + p0 + p * RPP + slice;
      n = (p0 + p * RPP + slice < nrows && n < H) ? n : n0;
      const size_t row = mat * H + n;
      load_row<CPL>(r[p], m.codes + row * cb, m.scales + row * sb, sl, LPR);
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const float v = sum_lanes_rt(dot_row<CPL, 2>(r[p], xs), LPR);
      const int rr = p0 + p * RPP + slice;
      if (sl == 0 && rr < nrows && n0 + rr < H) part[rr] = v * scale;
    }
  }
}

template <int CPLF, int CPLS>
__global__ void __launch_bounds__(kThreads, 2) k_down_combine(DecodeArgs a) {
  __shared__ float part[FLINT_MAX_TOP_K + 1][kDownRows];
  __shared__ float red[kWarps];
  const int warp = threadIdx.x >> 5;
  const int n0 = blockIdx.x * kDownRows;
  const int V = a.K + 2;  // routed slots, then the shared expert in two halves
  for (int b = 0; b < a.B; ++b) {
    for (int v = warp; v < V; v += kWarps) {
      if (v < a.K) {
        int e = __ldcg(a.sel_idx + b * a.K + v);
        if (e < 0 || e >= a.E) { raise_status(FLINT_ERR_INVALID_ARG); e = 0; }
        down_rows<CPLF>(a.down, e, a.H, a.F, n0, kDownRows,
                        a.h_routed + ((size_t)b * a.K + v) * a.F, part[v]);
      } else {
        const int half = v - a.K;
        down_rows<CPLS>(a.sh_down, 0, a.H, a.Fs, n0 + half * (kDownRows / 2), kDownRows / 2,
                        a.h_shared + (size_t)b * a.Fs, &part[a.K][half * (kDownRows / 2)]);
      }
    }
    __syncthreads();
    if (threadIdx.x < kDownRows && n0 + threadIdx.x < a.H) {
      const int n = n0 + threadIdx.x;
      const size_t o = (size_t)b * a.H + n;
      float acc = a.residual ? a.residual[o] : bf16_bits_to_f32(a.x[o]);
      float moe = 0.f;
      for (int s = 0; s < a.K; ++s) moe = fmaf(__ldcg(a.sel_w + b * a.K + s), part[s][threadIdx.x], moe);
      moe += part[a.K][threadIdx.x];
      a.out[o] = acc + moe;
    }
    __syncthreads();
  }
  if (a.x_next && last_cta_done(&a.counters[1])) {
    for (int b = 0; b < a.B; ++b) {
      float ss = 0.f;
      for (int n = threadIdx.x; n < a.H; n += kThreads) {
        const float v = __ldcg(a.out + (size_t)b * a.H + n);
        ss = fmaf(v, v, ss);
      }
      ss = sum_lanes<32>(ss);
      if ((threadIdx.x & 31) == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
      for (int w = 0; w < kWarps; ++w) tot += red[w];
      const float r = 1.0f / sqrtf(tot / (float)a.H + a.eps);
      for (int n = threadIdx.x; n < a.H; n += kThreads)
        a.x_next[(size_t)b * a.H + n] = f32_to_bf16_rn(__ldcg(a.out + (size_t)b * a.H + n) * r);
      __syncthreads();
    }
    if (threadIdx.x == 0) a.counters[1] = 0;
  }
}

// ---------------------------------------------------------------- host side
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t decode_workspace_bytes(int H, int E, int K, int F, int Fs, int B) {
  (void)H;
  size_t s = 0;
  s += align256(sizeof(float) * B * E);
  s += align256(sizeof(int32_t) * B * K);
  s += align256(sizeof(float) * B * K);
  s += align256(sizeof(float) * (size_t)B * K * F);
  s += align256(sizeof(float) * (size_t)B * Fs);
  s += align256(sizeof(unsigned int) * 4);
  return s;
}

void decode_carve(DecodeArgs& a, void* ws) {
  char* p = static_cast<char*>(ws);
  a.logits = reinterpret_cast<float*>(p); p += align256(sizeof(float) * a.B * a.E);
  a.sel_idx = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * a.B * a.K);
  a.sel_w = reinterpret_cast<float*>(p); p += align256(sizeof(float) * a.B * a.K);
  a.h_routed = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (size_t)a.B * a.K * a.F);
  a.h_shared = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (size_t)a.B * a.Fs);
  a.counters = reinterpret_cast<unsigned int*>(p);
}

static int g_num_sms = 0;
static int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

template <int CPLH>
static cudaError_t launch_decode_h(const DecodeArgs& a, cudaStream_t st) {
  const int sms = num_sms();
  k_router_shared<CPLH><<<sms * 2, kThreads, 0, st>>>(a);
  k_routed_gateup<CPLH><<<sms * 2, kThreads, 0, st>>>(a);
  const int grid_down = (a.H + kDownRows - 1) / kDownRows;
  const int cf = a.F > 1024 ? 2 : 1, cs = a.Fs > 1024 ? 2 : 1;
  if (cf == 1 && cs == 1) k_down_combine<1, 1><<<grid_down, kThreads, 0, st>>>(a);
  else if (cf == 1) k_down_combine<1, 2><<<grid_down, kThreads, 0, st>>>(a);
  else if (cs == 1) k_down_combine<2, 1><<<grid_down, kThreads, 0, st>>>(a);
  else k_down_combine<2, 2><<<grid_down, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.H <= 1024) return launch_decode_h<1>(a, st);
  if (a.H <= 2048) return launch_decode_h<2>(a, st);
  return launch_decode_h<4>(a, st);
}

}  // namespace flint
