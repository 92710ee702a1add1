// decode.cu -- persistent decode kernel: T tokens x L chained Flint MoE layers (+ head)
// in one cooperative launch (one CTA per SM).
//
// The layer ("Flint: 125 tokens a second is what 2.5B active parameters buy at 273
// GB/s", section "The shape, read from the headers"; "Recursive Releases Flint, a 40B
// MoE Coding Model That Runs Locally at 125 Tokens per Second", section "How does
// Flint's architecture work?") needs every active weight once per token and has one
// dependency no schedule can hide: which experts are read depends on the router.
//
// CTA roles (fixed for the launch).  With n_sh = Fs/32 shared-expert slices and
// n_rt = k*F/32 routed slices ("units": 32 SwiGLU outputs and their down block):
//   shared CTAs  [0, n_sh)              one shared-expert unit each
//   routed CTAs  [n_sh, n_sh + n_rt)    one (slot, slice) unit of the selected experts
//   router CTAs  the rest               router rows, and the copy of h_l into the next
//                                       residual buffer
// Step s = one layer of one token.  Two monotonic counters replace grid barriers:
//   logits(s) -- bumped by each router CTA once its logits and its share of the
//                residual copy are written;
//   done(s)   -- bumped by each unit CTA once its down contribution is red.added.
// Every CTA waits for done(s-1) (h_l complete) and stages x_l = bf16(RMSNorm(h_l)) in
// registers from one CTA-wide read of h_l.  Router CTAs compute logits and signal.
// Shared CTAs compute their unit right away (it needs only x_l), then wait for
// logits(s) before red.adding.  Routed CTAs wait for logits(s), compute the softmax
// top-k, then stream their unit.  Unit and router weights move global -> shared
// memory by TMA bulk copies (cp.async.bulk + mbarrier); router rows and shared units
// do not depend on the data, so the copies for step s+1 are issued as soon as step s
// has consumed the buffer.  The down projection of a unit is a split-K contribution to
// all H rows (a contiguous column-chunk block, see flint.h), summed into the next
// residual with red.global.add.v4.f32.
//
// After the last layer of a token the head GEMV (optional) runs over all CTAs; each
// CTA posts its best (logit, index) and CTA 0 reduces them.  Every wait is bounded by
// %globaltimer: on expiry the kernel records FLINT_ERR_TIMEOUT, raises an abort flag
// that releases all other waits, and runs to the end without hanging.
#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kPWarps = 16;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kSlice = 32;          // SwiGLU outputs per unit (one code chunk of down)
constexpr int kMaxCtas = 1024;
// Sync words, each on its own 128-byte line.
constexpr int kSyncLogits = 0, kSyncDone = 32, kSyncHead = 64, kSyncAbort = 96;
constexpr int kSyncWords = 128;

// ---------------------------------------------------------------- sync primitives
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 spins (bounded) until *cnt >= target; the CTA then proceeds together.
__device__ __forceinline__ void wait_count(unsigned* sync, int which, unsigned target) {
  if (threadIdx.x == 0) {
    const unsigned* cnt = sync + which;
    unsigned polls = 0;
    unsigned long long t0 = 0;
    while (ld_acquire_gpu(cnt) < target) {
      if ((++polls & 127u) == 0) {
        if (ld_acquire_gpu(sync + kSyncAbort)) break;
        const unsigned long long now = globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kWaitLimitNs) {
          raise_status(FLINT_ERR_TIMEOUT);
          atomicExch(sync + kSyncAbort, 1u);
          break;
        }
      }
    }
  }
  __syncthreads();
}

// Publishes every write of this CTA made before the call, then bumps the counter.
__device__ __forceinline__ void signal_count(unsigned* sync, int which) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(sync + which, 1u);
  }
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// ---------------------------------------------------------------- TMA bulk copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
               "selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(smem_addr(b)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for a bulk-copy phase; on expiry records FLINT_ERR_TIMEOUT.
__device__ __forceinline__ void mbar_wait(uint64_t* b, uint32_t parity, unsigned* sync) {
  unsigned long long t0 = 0;
  unsigned polls = 0;
  while (!mbar_try(b, parity)) {
    if ((++polls & 63u) == 0) {
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        raise_status(FLINT_ERR_TIMEOUT);
        atomicExch(sync + kSyncAbort, 1u);
        break;
      }
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------- activation staging
// x_l is built once per CTA (thread t owns elements [4t, 4t+4); H <= 4 * 512):
//   h    fp32 residual (global, L2) -> s_hx (kept for the residual copy)
//   x    bf16(h * r), r = 1/sqrt(mean(h^2) + eps)  (r = 1 for a layer-0 input, which
//        is bf16 already)                            -> s_xb
//   xf   f16(x * 2^k), the GEMV operand; 2^k puts max|x| in [2^14, 2^15) -> s_xf
// Sum of squares and max|h| come from one fixed-order block reduction, so every CTA
// derives the same r and k (max|bf16(h r)| = bf16(max|h| r): rounding is monotone).
struct Staged {
  float unscale;    // 2^-k
};

__device__ __forceinline__ Staged cta_stage(const float* h_f32, const uint16_t* x_bf16, int H,
                                            float eps, float* s_hx, uint16_t* s_xb,
                                            uint16_t* s_xf, float* s_red) {
  const int n = 4 * threadIdx.x;
  const bool own = n < H;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (own) {
    if (h_f32) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(h_f32 + n));
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
      const uint2 b = __ldcg(reinterpret_cast<const uint2*>(x_bf16 + n));
      v[0] = bf16_bits_to_f32(b.x & 0xFFFFu); v[1] = bf16_bits_to_f32(b.x >> 16);
      v[2] = bf16_bits_to_f32(b.y & 0xFFFFu); v[3] = bf16_bits_to_f32(b.y >> 16);
    }
    *reinterpret_cast<float4*>(s_hx + n) = make_float4(v[0], v[1], v[2], v[3]);
  }
  float ss = 0.f, am = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) { ss = fmaf(v[q], v[q], ss); am = fmaxf(am, fabsf(v[q])); }
  ss = sum_lanes<32>(ss);
#pragma unroll
  for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((threadIdx.x & 31) == 0) { s_red[threadIdx.x >> 5] = ss; s_red[kPWarps + (threadIdx.x >> 5)] = am; }
  __syncthreads();
  float tot = 0.f, amax = 0.f;
#pragma unroll
  for (int w = 0; w < kPWarps; ++w) { tot += s_red[w]; amax = fmaxf(amax, s_red[kPWarps + w]); }
  const float r = h_f32 ? 1.0f / sqrtf(tot / (float)H + eps) : 1.0f;
  const float xmax = bf16_bits_to_f32(f32_to_bf16_rn(amax * r));
  const int k = f16_stage_exponent(xmax);
  const float s = exp2i(k);
  if (own) {
    uint16_t b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = f32_to_bf16_rn(v[q] * r);
    *reinterpret_cast<uint2*>(s_xb + n) =
        make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16), (uint32_t)b[2] | ((uint32_t)b[3] << 16));
    const uint32_t f01 = pack_f16x2_rn(bf16_bits_to_f32(b[0]) * s, bf16_bits_to_f32(b[1]) * s);
    const uint32_t f23 = pack_f16x2_rn(bf16_bits_to_f32(b[2]) * s, bf16_bits_to_f32(b[3]) * s);
    *reinterpret_cast<uint2*>(s_xf + n) = make_uint2(f01, f23);
  }
  __syncthreads();
  return Staged{exp2i(-k)};
}

// The lane's chunk pairs from a staged 16-bit vector (bf16 or f16) in shared memory.
template <int CPL>
__device__ __forceinline__ void pairs_from_smem(uint32_t (&p)[CPL * 16], const uint16_t* s_v,
                                                int sl, int LPR) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(s_v + 32 * (sl + LPR * i));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = src[j];
      p[i * 16 + 4 * j] = q.x; p[i * 16 + 4 * j + 1] = q.y;
      p[i * 16 + 4 * j + 2] = q.z; p[i * 16 + 4 * j + 3] = q.w;
    }
  }
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

// ---------------------------------------------------------------- shared-memory rows
template <int CPL>
__device__ __forceinline__ void lds_row(RowRegs<CPL>& r, const uint8_t* codes_row,
                                        const uint8_t* scales_row, int sl, int LPR) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = sl + LPR * i;
    r.q[i] = *reinterpret_cast<const uint4*>(codes_row + 16 * c);
    r.s[i] = *reinterpret_cast<const uint16_t*>(scales_row + 2 * c);
  }
}

template <int CPL>
__device__ __forceinline__ void lds_row_bf16(RowBF16<CPL>& r, const uint16_t* row, int sl, int LPR) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(row + 32 * (sl + LPR * i));
#pragma unroll
    for (int j = 0; j < 4; ++j) r.q[i * 4 + j] = src[j];
  }
}

// ---------------------------------------------------------------- units
// Shared-memory image of one unit: 32 gate rows, 32 up rows (codes then scales) and
// the down block (H rows x one 32-column chunk).
struct UnitLayout {
  uint32_t gc, gs, uc, us, dc, ds, bytes;
  __host__ __device__ static UnitLayout of(int H) {
    UnitLayout u;
    u.gc = 0;
    u.gs = u.gc + kSlice * (H / 2);
    u.uc = u.gs + kSlice * (H / 16);
    u.us = u.uc + kSlice * (H / 2);
    u.dc = u.us + kSlice * (H / 16);
    u.ds = u.dc + H * 16;
    u.bytes = u.ds + H * 2;
    return u;
  }
};

// Issues the bulk copies of one unit (thread 0 only): gate/up rows [row0, row0+32) of
// the stacks and the down column-chunk block `chunk`.
__device__ __forceinline__ void issue_unit_copy(uint8_t* buf, uint64_t* bar, int H, const NVPtr& gate,
                                                const NVPtr& up, const uint8_t* dcc_codes,
                                                const uint8_t* dcc_scales, size_t row0,
                                                size_t chunk) {
  const UnitLayout L = UnitLayout::of(H);
  mbar_expect_tx(bar, L.bytes);
  bulk_g2s(buf + L.gc, gate.codes + row0 * (H / 2), kSlice * (H / 2), bar);
  bulk_g2s(buf + L.gs, gate.scales + row0 * (H / 16), kSlice * (H / 16), bar);
  bulk_g2s(buf + L.uc, up.codes + row0 * (H / 2), kSlice * (H / 2), bar);
  bulk_g2s(buf + L.us, up.scales + row0 * (H / 16), kSlice * (H / 16), bar);
  bulk_g2s(buf + L.dc, dcc_codes + chunk * H * 16, H * 16, bar);
  bulk_g2s(buf + L.ds, dcc_scales + chunk * H * 2, H * 2, bar);
}

// Computes one unit from shared memory: 32 SwiGLU outputs, then the down contribution
// (times wgt) of all H rows, added into s_part[H].
template <int CPL>
__device__ __forceinline__ void unit_compute(const uint8_t* buf, int H, float gate_tsc,
                                             float up_tsc, float down_tsc, float wgt,
                                             const XStage<CPL, 1>& xs, float* s_h,
                                             float* s_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const UnitLayout U = UnitLayout::of(H);
  const float gs = gate_tsc * xs.unscale, us = up_tsc * xs.unscale;
  // SwiGLU outputs: pair p handled by (warp, slice)
  for (int p0 = warp * RPP; p0 < kSlice; p0 += kPWarps * RPP) {
    const int p = p0 + slice;
    const int pr = p < kSlice ? p : 0;
    RowRegs<CPL> g, u;
    lds_row<CPL>(g, buf + U.gc + pr * (H / 2), buf + U.gs + pr * (H / 16), sl, LPR);
    lds_row<CPL>(u, buf + U.uc + pr * (H / 2), buf + U.us + pr * (H / 16), sl, LPR);
    const float vg = sum_lanes_rt(dot_row<CPL, 1>(g, xs), LPR);
    const float vu = sum_lanes_rt(dot_row<CPL, 1>(u, xs), LPR);
    if (sl == 0 && p < kSlice) s_h[p] = silu(vg * gs) * (vu * us);
  }
  __syncthreads();
  XStage<1, 2> hs;
  stage_slice(hs, s_h);
  const float scale = down_tsc * hs.unscale * wgt;
  // down block: consecutive lanes take consecutive rows (conflict-free shared loads)
  for (int n = warp * 32 + lane; n < H; n += kPWarps * 32) {
    RowRegs<1> d;
    d.q[0] = *reinterpret_cast<const uint4*>(buf + U.dc + n * 16);
    d.s[0] = *reinterpret_cast<const uint16_t*>(buf + U.ds + n * 2);
    s_part[n] += dot_row<1, 2>(d, hs) * scale;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- top-k
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Softmax top-k by one warp (see flint.h): largest logit first, ties to the lower index.
template <int kMaxPerLane>
__device__ void topk_warp(const float* logits, int E, int K, int* s_sel, float* s_w) {
  const int lane = threadIdx.x & 31;
  unsigned key[kMaxPerLane];
  float val[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    float l = (e < E) ? logits[e] : -INFINITY;
    l = (l == l) ? l : -INFINITY;
    val[i] = l;
    key[i] = (e < E) ? order_key(l) : 0u;      // every live key is >= 1
  }
  float top0 = 0.f, z = 0.f;
  for (int s = 0; s < K; ++s) {
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
  __syncwarp();
}

__device__ __forceinline__ void topk_dispatch(const float* logits, int E, int K, int* s_sel,
                                              float* s_w) {
  const int per_lane = (E + 31) / 32;
  if (per_lane <= 1) topk_warp<1>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 2) topk_warp<2>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 4) topk_warp<4>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 8) topk_warp<8>(logits, E, K, s_sel, s_w);
  else topk_warp<16>(logits, E, K, s_sel, s_w);
}

// ---------------------------------------------------------------- head
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
enum Role { kRoleShared = 0, kRoleRouted = 1, kRoleRouter = 2 };

template <int CPL>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const __grid_constant__ PersistArgs a) {
  __shared__ float s_h[kSlice];
  __shared__ int s_sel[FLINT_MAX_TOP_K];
  __shared__ float s_w[FLINT_MAX_TOP_K];
  __shared__ float s_bv[kPWarps];
  __shared__ int s_bi[kPWarps];
  __shared__ float s_red[2 * kPWarps];
  __shared__ float s_logits[FLINT_MAX_EXPERTS];
  __shared__ __align__(8) uint64_t s_bar;
  extern __shared__ __align__(128) uint8_t s_dyn[];
  float* s_hx = reinterpret_cast<float*>(s_dyn);                       // [H] residual h
  float* s_part = s_hx + a.H;                                          // [H] down partials
  uint16_t* s_xb = reinterpret_cast<uint16_t*>(s_part + a.H);          // [H] x, bf16
  uint16_t* s_xf = s_xb + a.H;                                         // [H] x * 2^k, f16
  uint8_t* s_wbuf = reinterpret_cast<uint8_t*>(s_xf + a.H);            // weight buffer

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, nC = gridDim.x;
  const int H = a.H;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int n_sh = a.Fs / kSlice;
  const int per_slot = a.F / kSlice;
  const int n_rt = a.K * per_slot;
  const int n_units = n_sh + n_rt;
  const int nR = nC - n_units;                       // router CTAs (host checks >= 1)
  const Role role = c < n_sh ? kRoleShared : (c < n_units ? kRoleRouted : kRoleRouter);
  const int ridx = c - n_units;                      // router CTA index
  const int rows_per_router = (a.E + nR - 1) / nR;
  const int r_lo = role == kRoleRouter ? min(a.E, ridx * rows_per_router) : 0;
  const int r_hi = role == kRoleRouter ? min(a.E, r_lo + rows_per_router) : 0;
  unsigned* sync = a.bar;
  uint32_t phase = 0;                                // parity of the weight-buffer mbarrier
  (void)lane;

  if (threadIdx.x == 0) {
    mbar_init(&s_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // Data-independent weight copies of a layer: router rows or this CTA's shared unit.
  auto issue_static = [&](int l) {
    if (threadIdx.x != 0) return;
    const LayerPtrs& P = a.layer[l];
    if (role == kRoleShared) {
      issue_unit_copy(s_wbuf, &s_bar, H, P.sh_gate, P.sh_up, P.sh_dcc_codes, P.sh_dcc_scales,
                      (size_t)c * kSlice, (size_t)c);
    } else if (role == kRoleRouter && r_hi > r_lo) {
      const uint32_t bytes = (uint32_t)(r_hi - r_lo) * H * 2;
      mbar_expect_tx(&s_bar, bytes);
      bulk_g2s(s_wbuf, P.router_w + (size_t)r_lo * H, bytes, &s_bar);
    }
  };
  issue_static(0);

  unsigned step = 0;                                 // global layer step
  for (int t = 0; t < a.T; ++t) {
    for (int l = 0; l < a.L; ++l, ++step) {
      const LayerPtrs& P = a.layer[l];
      float* acc_cur = a.acc + (step & 1) * H;
      float* acc_next = a.acc + ((step + 1) & 1) * H;
      const int l_next = (l + 1 < a.L) ? l + 1 : 0;
      const bool more = (l + 1 < a.L) || (t + 1 < a.T);
      // ---- h_l complete: stage x_l
      if (step > 0) wait_count(sync, kSyncDone, (unsigned)n_units * step);
      const Staged stg = cta_stage(l == 0 ? nullptr : acc_cur, a.x + (size_t)t * H, H, a.eps, s_hx,
                                   s_xb, s_xf, s_red);

      if (role == kRoleRouter) {
        // next residual buffer <- h_l (router CTAs share the rows)
        for (int n = ridx * kPThreads + threadIdx.x; n < H; n += nR * kPThreads)
          acc_next[n] = (l == 0 && a.residual) ? a.residual[(size_t)t * H + n] : s_hx[n];
        if (r_hi > r_lo) {
          mbar_wait(&s_bar, phase, sync);
          phase ^= 1;
          XRawBF16<CPL> xr;
          pairs_from_smem<CPL>(xr.p, s_xb, sl, LPR);
          for (int r0 = r_lo + warp * RPP; r0 < r_hi; r0 += kPWarps * RPP) {
            const int row = r0 + slice;
            RowBF16<CPL> rw;
            lds_row_bf16<CPL>(rw, reinterpret_cast<const uint16_t*>(s_wbuf) +
                                      (size_t)((row < r_hi ? row : r_lo) - r_lo) * H, sl, LPR);
            const float v = sum_lanes_rt(dot_row_bf16<CPL>(rw, xr), LPR);
            if (row < r_hi && sl == 0) a.logits_ws[row] = v + (P.router_bias ? P.router_bias[row] : 0.f);
          }
        }
        signal_count(sync, kSyncLogits);
        __syncthreads();                       // buffer reads done before it is refilled
        if (more) issue_static(l_next);
      } else if (role == kRoleShared) {
        XStage<CPL, 1> xs;
        pairs_from_smem<CPL>(xs.p[0], s_xf, sl, LPR);
        xs.unscale = stg.unscale;
        for (int n = threadIdx.x; n < H; n += kPThreads) s_part[n] = 0.f;
        mbar_wait(&s_bar, phase, sync);
        phase ^= 1;
        unit_compute<CPL>(s_wbuf, H, P.sh_gate.tsc[0], P.sh_up.tsc[0], P.sh_down_tsc[0], 1.0f, xs,
                          s_h, s_part);
        if (more) issue_static(l_next);         // unit_compute ended with a CTA barrier
        wait_count(sync, kSyncLogits, (unsigned)nR * (step + 1));
        for (int n = 4 * threadIdx.x; n < H; n += 4 * kPThreads)
          red_add_v4(acc_next + n, s_part[n], s_part[n + 1], s_part[n + 2], s_part[n + 3]);
        signal_count(sync, kSyncDone);
      } else {  // routed
        XStage<CPL, 1> xs;
        pairs_from_smem<CPL>(xs.p[0], s_xf, sl, LPR);
        xs.unscale = stg.unscale;
        for (int n = threadIdx.x; n < H; n += kPThreads) s_part[n] = 0.f;
        wait_count(sync, kSyncLogits, (unsigned)nR * (step + 1));
        for (int e = threadIdx.x; e < a.E; e += kPThreads) s_logits[e] = __ldcg(a.logits_ws + e);
        __syncthreads();
        if (warp == 0) topk_dispatch(s_logits, a.E, a.K, s_sel, s_w);
        __syncthreads();
        const int u = c - n_sh;
        const int sslot = u / per_slot, j = u % per_slot;
        int e = s_sel[sslot];
        if (e < 0 || e >= a.E) { raise_status(FLINT_ERR_INVALID_ARG); e = 0; }
        if (threadIdx.x == 0)
          issue_unit_copy(s_wbuf, &s_bar, H, P.gate, P.up, P.dcc_codes, P.dcc_scales,
                          (size_t)e * a.F + (size_t)j * kSlice, (size_t)e * per_slot + j);
        if (u == 0 && threadIdx.x < a.K) {
          const size_t o = ((size_t)t * a.L + l) * a.K + threadIdx.x;
          if (a.idx_out) a.idx_out[o] = s_sel[threadIdx.x];
          if (a.w_out) a.w_out[o] = s_w[threadIdx.x];
        }
        mbar_wait(&s_bar, phase, sync);
        phase ^= 1;
        unit_compute<CPL>(s_wbuf, H, P.gate.tsc[e], P.up.tsc[e], P.down_tsc[e], s_w[sslot], xs, s_h,
                          s_part);
        for (int n = 4 * threadIdx.x; n < H; n += 4 * kPThreads)
          red_add_v4(acc_next + n, s_part[n], s_part[n + 1], s_part[n + 2], s_part[n + 3]);
        signal_count(sync, kSyncDone);
      }
    }
    // ---------------- outputs of token t
    wait_count(sync, kSyncDone, (unsigned)n_units * step);
    const float* hfin = a.acc + (step & 1) * H;
    if (a.out)
      for (int n = c * kPThreads + threadIdx.x; n < H; n += nC * kPThreads)
        a.out[(size_t)t * H + n] = __ldcg(hfin + n);
    if (a.x_out || a.head.codes) {
      const Staged stg = cta_stage(hfin, nullptr, H, a.eps, s_hx, s_xb, s_xf, s_red);
      if (a.x_out && c == 0)
        for (int n = 4 * threadIdx.x; n < H; n += 4 * kPThreads)
          *reinterpret_cast<uint2*>(a.x_out + (size_t)t * H + n) = *reinterpret_cast<const uint2*>(s_xb + n);
      if (a.head.codes) {
        XStage<CPL, 1> xs;
        pairs_from_smem<CPL>(xs.p[0], s_xf, sl, LPR);
        xs.unscale = stg.unscale;
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        head_rows<CPL>(a, xs, t, bv, bi);
        best_reduce_warp(bv, bi);
        if ((threadIdx.x & 31) == 0) { s_bv[warp] = bv; s_bi[warp] = bi; }
        __syncthreads();
        float* best_v = a.best_v + (t & 1) * kMaxCtas;
        int* best_i = a.best_i + (t & 1) * kMaxCtas;
        if (threadIdx.x == 0) {
          for (int w = 1; w < kPWarps; ++w)
            if (s_bv[w] > bv || (s_bv[w] == bv && s_bi[w] < bi)) { bv = s_bv[w]; bi = s_bi[w]; }
          best_v[c] = bv;
          best_i[c] = bi;
        }
        signal_count(sync, kSyncHead);
        if (c == 0) {
          wait_count(sync, kSyncHead, (unsigned)nC * (t + 1));
          if (warp == 0) {
            const int ln = threadIdx.x & 31;
            float v = -INFINITY;
            int i = 0x7FFFFFFF;
            for (int k = ln; k < nC; k += 32) {
              const float kv = __ldcg(best_v + k);
              const int ki = __ldcg(best_i + k);
              if (kv > v || (kv == v && ki < i)) { v = kv; i = ki; }
            }
            best_reduce_warp(v, i);
            if (ln == 0 && a.argmax) a.argmax[t] = (i < a.V) ? i : 0;
          }
        }
      }
    }
  }
  // No bulk copy is in flight at exit: copies are issued only while `more` holds, and
  // every issued copy is waited for in the step that follows.
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

size_t decode_workspace_bytes(int H, int E) {
  return sizeof(unsigned) * kSyncWords + align256(sizeof(float) * E) +
         align256(sizeof(float) * 2 * H) + 2 * align256(2 * kMaxCtas * sizeof(float));
}

void decode_carve(PersistArgs& a, void* ws) {
  char* p = static_cast<char*>(ws);
  a.bar = reinterpret_cast<unsigned*>(p); p += sizeof(unsigned) * kSyncWords;
  a.logits_ws = reinterpret_cast<float*>(p); p += align256(sizeof(float) * a.E);
  a.acc = reinterpret_cast<float*>(p); p += align256(sizeof(float) * 2 * a.H);
  a.best_v = reinterpret_cast<float*>(p); p += align256(2 * kMaxCtas * sizeof(float));
  a.best_i = reinterpret_cast<int*>(p);
}

static int g_sms = 0;
int decode_grid() {
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms > kMaxCtas) g_sms = kMaxCtas;
  }
  return g_sms;
}

size_t decode_smem_bytes(int H, int E, int nR) {
  const size_t unit = UnitLayout::of(H).bytes;
  const size_t router = (size_t)((E + nR - 1) / nR) * H * 2;
  return (2 * sizeof(float) + 2 * sizeof(uint16_t)) * H + (unit > router ? unit : router);
}

template <int CPL>
static cudaError_t launch_persistent_cpl(const PersistArgs& a, cudaStream_t st) {
  const int grid = decode_grid();
  const int nR = grid - (a.Fs / kSlice + a.K * (a.F / kSlice));
  const size_t smem = decode_smem_bytes(a.H, a.E, nR);
  cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<CPL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
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
  cudaError_t e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned) * kSyncWords, st);
  if (e != cudaSuccess) return e;
  if (a.H <= 1024) return launch_persistent_cpl<1>(a, st);
  return launch_persistent_cpl<2>(a, st);
}

}  // namespace flint
