// decode.cu -- persistent decode kernel: T tokens x L chained Flint MoE layers (+ head)
// in one cooperative launch (one CTA per SM).
//
// The layer ("Flint: 125 tokens a second is what 2.5B active parameters buy at 273
// GB/s", section "The shape, read from the headers"; "Recursive Releases Flint, a 40B
// MoE Coding Model That Runs Locally at 125 Tokens per Second", section "How does
// Flint's architecture work?") needs its weights once per token and has one data
// dependency that no schedule can hide: which experts are read depends on the router.
// Per layer the kernel runs two phases separated by grid-wide barriers:
//
//  A  every warp stages x_l (RMSNorm of the running residual h_l, computed redundantly
//     per warp) in registers.  Router CTAs compute the bf16 router logits.  Shared
//     CTAs each own a 32-wide slice of the shared expert: 32 gate/up row pairs ->
//     32 SwiGLU outputs (shared memory) -> their split-K contribution to all H down
//     rows (a contiguous column-chunk block of the down matrix), kept in shared memory.
//     Every CTA also copies its share of h_l into the next residual buffer.
//  -- barrier --
//  B  every CTA computes the softmax top-k from the logits (one warp, redundantly).
//     Routed CTAs each own (slot, 32-wide slice): they issue all loads of their unit
//     at once (gate/up rows and the down block, ~110 KB per CTA for Flint), compute
//     the slice's SwiGLU outputs, and red.add w_slot * (down block x h slice) into the
//     next residual; shared CTAs red.add their contribution.
//  -- barrier --
//
// After the last layer the head GEMV (optional) runs over the whole grid, each CTA
// keeps its best (logit, index), and CTA 0 reduces them after one more barrier.
// Barrier waits are bounded by %globaltimer: on expiry the kernel records
// FLINT_ERR_TIMEOUT, raises an abort flag that releases every other wait, and runs to
// the end without hanging.
#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kPWarps = 16;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kSlice = 32;          // SwiGLU outputs per unit (one code chunk of down)

// ---------------------------------------------------------------- grid barrier
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// bar[0]: arrivals (monotonic), bar[1]: generation released, bar[2]: abort flag.
__device__ __forceinline__ void grid_sync(unsigned* bar, unsigned& gen) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = ++gen;
    __threadfence();
    const unsigned arrived = atomicAdd(&bar[0], 1u) + 1u;
    if (arrived == target * gridDim.x) {
      st_release_gpu(&bar[1], target);
    } else {
      const unsigned long long t0 = globaltimer();
      unsigned polls = 0;
      while (ld_acquire_gpu(&bar[1]) < target) {
        if ((++polls & 255u) == 0) {
          if (ld_acquire_gpu(&bar[2])) break;
          if (globaltimer() - t0 > kWaitLimitNs) {
            raise_status(FLINT_ERR_TIMEOUT);
            atomicExch(&bar[2], 1u);
            break;
          }
        }
      }
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- vector atomics
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// ---------------------------------------------------------------- activation staging
// Warp-redundant RMSNorm: every warp reads the whole residual h (fp32, L2) in its
// chunk order, sums squares (identical order in every warp), and returns the bf16
// x = bf16(h / sqrt(mean(h^2) + eps)) as bf16x2 pairs of the lane's chunks.
template <int CPL>
__device__ __forceinline__ void rmsnorm_bf16_pairs(uint32_t (&xb)[CPL * 16], const float* h, int H,
                                                   float eps, int sl, int LPR) {
  float v[CPL * 32];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const float4* src = reinterpret_cast<const float4*>(h + 32 * (sl + LPR * i));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 f = __ldcg(src + j);
      v[i * 32 + 4 * j] = f.x; v[i * 32 + 4 * j + 1] = f.y;
      v[i * 32 + 4 * j + 2] = f.z; v[i * 32 + 4 * j + 3] = f.w;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < CPL * 32; ++q) ss = fmaf(v[q], v[q], ss);
  ss = sum_lanes_rt(ss, LPR);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
#pragma unroll
  for (int q = 0; q < CPL * 16; ++q)
    xb[q] = (uint32_t)f32_to_bf16_rn(v[2 * q] * r) | ((uint32_t)f32_to_bf16_rn(v[2 * q + 1] * r) << 16);
}

template <int CPL>
__device__ __forceinline__ void load_bf16_pairs(uint32_t (&xb)[CPL * 16], const uint16_t* x, int sl,
                                                int LPR) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(x + 32 * (sl + LPR * i));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = __ldcg(src + j);
      xb[i * 16 + 4 * j] = q.x; xb[i * 16 + 4 * j + 1] = q.y;
      xb[i * 16 + 4 * j + 2] = q.z; xb[i * 16 + 4 * j + 3] = q.w;
    }
  }
}

// bf16 pairs -> f16 pairs scaled by 2^k (exact), amax over the slice
template <int CPL>
__device__ __forceinline__ void stage_from_pairs(XStage<CPL, 1>& xs, const uint32_t (&xb)[CPL * 16],
                                                 int LPR) {
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < CPL * 16; ++q) {
    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(xb[q] & 0xFFFFu)));
    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(xb[q] >> 16)));
  }
  amax = max_lanes_rt(amax, LPR);
  const int k = f16_stage_exponent(amax);
  const float s = exp2i(k);
  xs.unscale = exp2i(-k);
#pragma unroll
  for (int q = 0; q < CPL * 16; ++q)
    xs.p[0][q] = pack_f16x2_rn(bf16_bits_to_f32(xb[q] & 0xFFFFu) * s, bf16_bits_to_f32(xb[q] >> 16) * s);
}

// A 32-value slice (shared memory) staged as hi/lo f16 pairs: every lane holds all 32.
__device__ __forceinline__ void stage_slice(XStage<1, 2>& hs, const float* s_h) {
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < kSlice; ++q) amax = fmaxf(amax, fabsf(s_h[q]));
  const int k = f16_stage_exponent(amax);
  const float s = exp2i(k);
  hs.unscale = exp2i(-k);
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float a = s_h[2 * q] * s, b = s_h[2 * q + 1] * s;
    const uint32_t hi = pack_f16x2_rn(a, b);
    float ha, hb;
    f16x2_to_f32x2(hi, ha, hb);
    hs.p[0][q] = hi;
    hs.p[1][q] = pack_f16x2_rn(a - ha, b - hb);
  }
}

// ---------------------------------------------------------------- per-layer units
struct UnitLoads {
  RowRegs<1> dn[4];    // down block rows (4 consecutive rows per lane per pass)
};

// One 32-wide SwiGLU slice of one expert: gate/up rows [j0, j0+32) of (gate, up) stacks
// (matrix `mat`), then the split-K contribution of the down column chunk j0/32 to all
// H rows.  The contribution, times `wgt`, is either red.added into acc (direct) or
// accumulated into the CTA's shared partial s_part[H].
template <int CPL>
__device__ __forceinline__ void swiglu_slice_unit(const PersistArgs& a, const NVPtr& gate,
                                                  const NVPtr& up, const uint8_t* dcc_codes,
                                                  const uint8_t* dcc_scales, float dtsc,
                                                  size_t mat, int width, int j0, float wgt,
                                                  const XStage<CPL, 1>& xs, float* s_h,
                                                  float* acc, float* s_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const size_t cb = H / 2, sb = H / 16;
  // --- issue all loads: gate/up pairs of this warp, then the down rows
  constexpr int kPairs = 2;  // pair passes per warp (32 pairs / 16 warps for RPP = 1)
  RowRegs<CPL> g[kPairs], u[kPairs];
  int pj[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    int p = (warp * RPP + slice) + kPWarps * RPP * i;
    pj[i] = p;
    const int pr = p < kSlice ? p : 0;
    const size_t row = mat * width + j0 + pr;
    load_row<CPL>(g[i], gate.codes + row * cb, gate.scales + row * sb, sl, LPR);
    load_row<CPL>(u[i], up.codes + row * cb, up.scales + row * sb, sl, LPR);
  }
  // down block: chunk c = j0/32 of matrix `mat` -> rows [0, H) contiguous
  const int rows_per_warp = H / kPWarps;
  const size_t chunk = (size_t)mat * (width / 32) + j0 / 32;
  const uint8_t* dc = dcc_codes + chunk * H * 16;
  const uint8_t* ds = dcc_scales + chunk * H * 2;
  const int nbase = warp * rows_per_warp;
  // every lane owns 4 consecutive rows per 128-row group
  UnitLoads L;
  const int r0 = 4 * lane;
  const bool have = r0 < rows_per_warp;   // rows_per_warp >= 4 always (H >= 64)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = nbase + (have ? r0 + q : 0);
    L.dn[q].q[0] = ldg_stream(dc + (size_t)n * 16);
    L.dn[q].s[0] = ldg_stream_u16(ds + (size_t)n * 2);
  }
  // --- SwiGLU outputs of the slice
  const float gs = gate.tsc[mat] * xs.unscale, us = up.tsc[mat] * xs.unscale;
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const float vg = sum_lanes_rt(dot_row<CPL, 1>(g[i], xs), LPR);
    const float vu = sum_lanes_rt(dot_row<CPL, 1>(u[i], xs), LPR);
    if (sl == 0 && pj[i] < kSlice) s_h[pj[i]] = silu(vg * gs) * (vu * us);
  }
  __syncthreads();
  XStage<1, 2> hs;
  stage_slice(hs, s_h);
  const float scale = dtsc * hs.unscale * wgt;
  float part[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) part[q] = dot_row<1, 2>(L.dn[q], hs) * scale;
  // remaining row groups (only when H / 16 > 128, i.e. H > 2048)
  if (have) {
    if (s_part) {
#pragma unroll
      for (int q = 0; q < 4; ++q) s_part[nbase + r0 + q] += part[q];
    } else {
      red_add_v4(acc + nbase + r0, part[0], part[1], part[2], part[3]);
    }
  }
  for (int rb = 128; rb < rows_per_warp; rb += 128) {
    const int rr = rb + r0;
    if (rr < rows_per_warp) {
      RowRegs<1> d4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        d4[q].q[0] = ldg_stream(dc + (size_t)(nbase + rr + q) * 16);
        d4[q].s[0] = ldg_stream_u16(ds + (size_t)(nbase + rr + q) * 2);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) part[q] = dot_row<1, 2>(d4[q], hs) * scale;
      if (s_part) {
#pragma unroll
        for (int q = 0; q < 4; ++q) s_part[nbase + rr + q] += part[q];
      } else {
        red_add_v4(acc + nbase + rr, part[0], part[1], part[2], part[3]);
      }
    }
  }
  __syncthreads();   // s_h is reused by the next unit
}

// Softmax top-k by one warp (see flint.h): largest logit first, ties to the lower index.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ void topk_warp(const float* logits, int E, int K, int* s_sel, float* s_w) {
  const int lane = threadIdx.x & 31;
  constexpr int kMaxPerLane = FLINT_MAX_EXPERTS / 32;
  unsigned key[kMaxPerLane];
  float val[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    float l = (e < E) ? __ldcg(logits + e) : -INFINITY;
    l = (l == l) ? l : -INFINITY;
    val[i] = l;
    key[i] = (e < E) ? order_key(l) : 0u;      // padding never beats a real expert
  }
  float top0 = 0.f, z = 0.f;
  for (int s = 0; s < K; ++s) {
    // this lane's best candidate: largest key, then lowest index (retired keys are 0,
    // every live key is >= 1, so a candidate always exists while s < K <= E)
    unsigned bk = 0u;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && key[i] != 0u && (key[i] > bk || (key[i] == bk && e < bi))) {
        bk = key[i];
        bi = e;
      }
    }
    const unsigned wk = __reduce_max_sync(0xffffffffu, bk);
    const int we = (int)__reduce_min_sync(0xffffffffu, (unsigned)(bk == wk ? bi : 0x7FFFFFFF));
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (lane + 32 * i == we) { mine = val[i]; key[i] = 0u; }
    const float wl = __shfl_sync(0xffffffffu, mine, we & 31);
    if (s == 0) top0 = wl;
    const float p = expf(wl - top0);
    z += p;
    if (lane == 0) { s_sel[s] = we; s_w[s] = p; }
  }
  __syncwarp();
  if (lane < K) s_w[lane] = s_w[lane] / z;
}

// ---------------------------------------------------------------- head phase
template <int CPL>
__device__ __forceinline__ void head_rows(const PersistArgs& a, const XStage<CPL, 1>& xs, int t,
                                          float& bv, int& bi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = a.H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const size_t cb = a.H / 2, sb = a.H / 16;
  constexpr int NR = 4;
  const int gw = blockIdx.x * kPWarps + warp, nw = gridDim.x * kPWarps;
  const int per_task = RPP * NR;
  const int n_tasks = (a.V + per_task - 1) / per_task;
  const float tsc = a.head.tsc[0] * xs.unscale;
  for (int task = gw; task < n_tasks; task += nw) {
    RowRegs<CPL> r[NR];
#pragma unroll
    for (int p = 0; p < NR; ++p) {
      int row = task * per_task + p * RPP + slice;
      row = row < a.V ? row : a.V - 1;
      load_row<CPL>(r[p], a.head.codes + row * cb, a.head.scales + row * sb, sl, LPR);
    }
#pragma unroll
    for (int p = 0; p < NR; ++p) {
      const int row = task * per_task + p * RPP + slice;
      const float v = sum_lanes_rt(dot_row<CPL, 1>(r[p], xs), LPR) * tsc;
      if (row < a.V) {
        if (sl == 0 && a.logits) a.logits[(size_t)t * a.V + row] = v;
        const float vv = (v == v) ? v : -INFINITY;
        if (vv > bv || (vv == bv && row < bi)) { bv = vv; bi = row; }
      }
    }
  }
}

__device__ __forceinline__ void best_reduce_warp(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

// ---------------------------------------------------------------- the kernel
template <int CPL>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const __grid_constant__ PersistArgs a) {
  __shared__ float s_h[kSlice];
  __shared__ int s_sel[FLINT_MAX_TOP_K];
  __shared__ float s_w[FLINT_MAX_TOP_K];
  __shared__ float s_bv[kPWarps];
  __shared__ int s_bi[kPWarps];
  extern __shared__ float s_part[];            // [H]: shared-expert partials of this CTA
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nC = gridDim.x, c = blockIdx.x;
  const int H = a.H;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int n_sh = a.Fs / kSlice;
  const int n_rt = a.K * (a.F / kSlice);
  const int router_per_cta = kPWarps * RPP;
  const int n_rcta = (a.E + router_per_cta - 1) / router_per_cta;
  unsigned* bar = a.bar;
  unsigned gen = 0;
  int cur = 0;                                  // acc buffer holding h after layer >= 1
  for (int t = 0; t < a.T; ++t) {
    for (int l = 0; l < a.L; ++l) {
      const LayerPtrs& P = a.layer[l];
      float* acc_cur = a.acc + cur * H;
      float* acc_next = a.acc + (cur ^ 1) * H;
      // ---------------- A
      // x_l as bf16 pairs (every warp)
      uint32_t xb[CPL * 16];
      if (l == 0) load_bf16_pairs<CPL>(xb, a.x + (size_t)t * H, sl, LPR);
      else rmsnorm_bf16_pairs<CPL>(xb, acc_cur, H, a.eps, sl, LPR);
      // next residual buffer <- h_l (this CTA's rows)
      for (int n = c * kPThreads + threadIdx.x; n < H; n += nC * kPThreads) {
        float hv;
        if (l > 0) hv = __ldcg(acc_cur + n);
        else if (a.residual) hv = a.residual[(size_t)t * H + n];
        else hv = bf16_bits_to_f32(a.x[(size_t)t * H + n]);
        acc_next[n] = hv;
      }
      bool has_shared = false;
      for (int n = threadIdx.x; n < H; n += kPThreads) s_part[n] = 0.f;
      __syncthreads();
      // router rows
      const int rc0 = ((c - (n_sh + n_rt)) % nC + nC) % nC;
      for (int rc = rc0; rc < n_rcta; rc += nC) {
        const int row = rc * router_per_cta + warp * RPP + slice;
        XRawBF16<CPL> xr;
#pragma unroll
        for (int q = 0; q < CPL * 16; ++q) xr.p[q] = xb[q];
        RowBF16<CPL> r;
        load_row_bf16<CPL>(r, P.router_w + (size_t)(row < a.E ? row : 0) * H, sl, LPR);
        const float v = sum_lanes_rt(dot_row_bf16<CPL>(r, xr), LPR);
        if (row < a.E && sl == 0) a.logits_ws[row] = v + (P.router_bias ? P.router_bias[row] : 0.f);
      }
      // shared units
      if (c < n_sh || n_sh > nC) {
        XStage<CPL, 1> xs;
        stage_from_pairs<CPL>(xs, xb, LPR);
        for (int u = c; u < n_sh; u += nC) {
          has_shared = true;
          swiglu_slice_unit<CPL>(a, P.sh_gate, P.sh_up, P.sh_dcc_codes, P.sh_dcc_scales,
                                 P.sh_down_tsc[0], 0, a.Fs, u * kSlice, 1.0f, xs, s_h, nullptr,
                                 s_part);
        }
      }
      grid_sync(bar, gen);
      // ---------------- B
      if (warp == 0) topk_warp(a.logits_ws, a.E, a.K, s_sel, s_w);
      __syncthreads();
      if (c == 0 && threadIdx.x < a.K) {
        const size_t o = ((size_t)t * a.L + l) * a.K + threadIdx.x;
        if (a.idx_out) a.idx_out[o] = s_sel[threadIdx.x];
        if (a.w_out) a.w_out[o] = s_w[threadIdx.x];
      }
      if (has_shared) {
        for (int n = 4 * threadIdx.x; n < H; n += 4 * kPThreads)
          red_add_v4(acc_next + n, s_part[n], s_part[n + 1], s_part[n + 2], s_part[n + 3]);
      }
      {
        int u0 = (c - n_sh) % nC;
        if (u0 < 0) u0 += nC;
        if (u0 < n_rt) {
          XStage<CPL, 1> xs;
          stage_from_pairs<CPL>(xs, xb, LPR);
          const int per_slot = a.F / kSlice;
          for (int u = u0; u < n_rt; u += nC) {
            const int s = u / per_slot, j = u % per_slot;
            int e = s_sel[s];
            if (e < 0 || e >= a.E) { raise_status(FLINT_ERR_INVALID_ARG); e = 0; }
            swiglu_slice_unit<CPL>(a, P.gate, P.up, P.dcc_codes, P.dcc_scales, P.down_tsc[e],
                                   (size_t)e, a.F, j * kSlice, s_w[s], xs, s_h, acc_next,
                                   nullptr);
          }
        }
      }
      grid_sync(bar, gen);
      cur ^= 1;
    }
    // ---------------- outputs of token t
    const float* hfin = a.acc + cur * H;
    if (a.out)
      for (int n = c * kPThreads + threadIdx.x; n < H; n += nC * kPThreads)
        a.out[(size_t)t * H + n] = __ldcg(hfin + n);
    if (a.x_out || a.head.codes) {
      uint32_t xb[CPL * 16];
      rmsnorm_bf16_pairs<CPL>(xb, hfin, H, a.eps, sl, LPR);
      if (a.x_out && c == 0 && warp == 0) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(a.x_out + (size_t)t * H);
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
          for (int q = 0; q < 16; ++q) dst[16 * (sl + LPR * i) + q] = xb[i * 16 + q];
      }
      if (a.head.codes) {
        XStage<CPL, 1> xs;
        stage_from_pairs<CPL>(xs, xb, LPR);
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        head_rows<CPL>(a, xs, t, bv, bi);
        best_reduce_warp(bv, bi);
        if (lane == 0) { s_bv[warp] = bv; s_bi[warp] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
          for (int w = 1; w < kPWarps; ++w)
            if (s_bv[w] > bv || (s_bv[w] == bv && s_bi[w] < bi)) { bv = s_bv[w]; bi = s_bi[w]; }
          a.best_v[c] = bv;
          a.best_i[c] = bi;
        }
        grid_sync(bar, gen);
        if (c == 0 && warp == 0) {
          float v = -INFINITY;
          int i = 0x7FFFFFFF;
          for (int k = lane; k < nC; k += 32) {
            const float kv = __ldcg(a.best_v + k);
            const int ki = __ldcg(a.best_i + k);
            if (kv > v || (kv == v && ki < i)) { v = kv; i = ki; }
          }
          best_reduce_warp(v, i);
          if (lane == 0 && a.argmax) a.argmax[t] = (i < a.V) ? i : 0;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- column-chunk repack
__global__ void k_column_chunks(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                int rows, int cols, uint8_t* __restrict__ codes_cc,
                                uint8_t* __restrict__ scales_cc) {
  const int m = blockIdx.y;
  const int nch = cols / 32;
  const int64_t n = (int64_t)rows * nch;
  const uint8_t* cm = codes + (size_t)m * rows * (cols / 2);
  const uint8_t* sm = scales + (size_t)m * rows * (cols / 16);
  uint8_t* co = codes_cc + (size_t)m * rows * (cols / 2);
  uint8_t* so = scales_cc + (size_t)m * rows * (cols / 16);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nch, ch = i % nch;        // source: row r, chunk ch
    const uint4 v = *reinterpret_cast<const uint4*>(cm + r * (cols / 2) + ch * 16);
    const uint16_t s = *reinterpret_cast<const uint16_t*>(sm + r * (cols / 16) + ch * 2);
    *reinterpret_cast<uint4*>(co + (ch * rows + r) * 16) = v;
    *reinterpret_cast<uint16_t*>(so + (ch * rows + r) * 2) = s;
  }
}

cudaError_t launch_column_chunks(const uint8_t* codes, const uint8_t* scales, int n_mat, int rows,
                                 int cols, uint8_t* codes_cc, uint8_t* scales_cc, cudaStream_t st) {
  const int64_t n = (int64_t)rows * (cols / 32);
  int g = (int)((n + 255) / 256);
  if (g > 4096) g = 4096;
  k_column_chunks<<<dim3(g, n_mat), 256, 0, st>>>(codes, scales, rows, cols, codes_cc, scales_cc);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host side
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr int kMaxCtas = 1024;

size_t decode_workspace_bytes(int H, int E) {
  return align256(sizeof(float) * E) + align256(sizeof(float) * 2 * H) + 256 +
         align256(kMaxCtas * (sizeof(float) + sizeof(int)));
}

void decode_carve(PersistArgs& a, void* ws) {
  char* p = static_cast<char*>(ws);
  a.bar = reinterpret_cast<unsigned*>(p); p += 256;
  a.logits_ws = reinterpret_cast<float*>(p); p += align256(sizeof(float) * a.E);
  a.acc = reinterpret_cast<float*>(p); p += align256(sizeof(float) * 2 * a.H);
  a.best_v = reinterpret_cast<float*>(p); p += align256(kMaxCtas * sizeof(float));
  a.best_i = reinterpret_cast<int*>(p);
}

template <int CPL>
static cudaError_t launch_persistent_cpl(const PersistArgs& a, cudaStream_t st) {
  static int grid = 0;
  const size_t smem = sizeof(float) * a.H;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<CPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(float) * FLINT_MAX_HIDDEN));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_persistent<CPL>, kPThreads,
                                                      sizeof(float) * FLINT_MAX_HIDDEN);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    grid = sms < kMaxCtas ? sms : kMaxCtas;   // one CTA per SM
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_persistent<CPL>, a);
}

cudaError_t launch_persistent(const PersistArgs& a, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.bar, 0, 256, st);
  if (e != cudaSuccess) return e;
  if (a.H <= 1024) return launch_persistent_cpl<1>(a, st);
  if (a.H <= 2048) return launch_persistent_cpl<2>(a, st);
  return launch_persistent_cpl<4>(a, st);
}

}  // namespace flint
