// decode.cu -- persistent decode kernel: T tokens x L chained Flint MoE layers (+ head)
// in one cooperative launch (one CTA per SM).
//
// The layer ("Flint: 125 tokens a second is what 2.5B active parameters buy at 273
// GB/s", section "The shape, read from the headers"; "Recursive Releases Flint, a 40B
// MoE Coding Model That Runs Locally at 125 Tokens per Second", section "How does
// Flint's architecture work?") needs every active weight once per token and has one
// dependency no schedule can hide: which experts are read depends on the router.
//
// Work split (fixed for the launch; G CTAs, every CTA runs the same code).  A "unit"
// is 8 consecutive SwiGLU outputs of one expert with the down-projection column chunk
// they feed; the decode-unit copy of the weights (flint.h) stores each unit as one
// contiguous block, fetched by one TMA bulk copy.  CTA c owns
//   router rows   e = c, c + G, ...        (of E)
//   shared units  s = G-1-c, G-1-c + G, ... (of Fs/8)
//   routed units  r = c, c + G, ...        (of k*F/8: unit r % (F/8) of slot r / (F/8))
// Step s = one layer of one token:
//   1. wait until done(s-1) = G*s (h_l complete) and stage x_l = bf16(RMSNorm(h_l))
//      in shared memory from one fixed-order CTA reduction (identical in every CTA);
//   2. compute the router rows and post each logit, tagged with s+1, to every copy of
//      a logit board (one 64-bit store: no fence, no counter);
//   3. warps 0-7 poll all E logits on this CTA's board copy and select the top k
//      exactly (threshold from the warp maxima, then ranks); warp 0 issues the routed
//      units' copies, warp 1 computes the routing weights and the selected experts'
//      tensor scales; meanwhile warps 8-15 compute the shared units' gate/up;
//   4. the shared units' SwiGLU and down pass run while the routed copies are in
//      flight; each routed unit's gate/up runs as soon as its copy lands, then their
//      SwiGLU and down pass;
//   5. the CTA's down contributions (all H rows) are red.added (fp32) into the next
//      residual buffer, and done(s) is bumped with a release add.
// Router rows and shared units do not depend on the data: their copies for step s+1
// are issued as soon as step s has consumed the buffers.  The per-layer pointer table,
// shared tensor scales and router bias are prefetched into shared memory a step ahead.
// The loops of the step stay rolled: the step runs far more distinct instructions
// than the instruction caches hold, so its time follows its code size.
//
// After the last layer of a token the head GEMV (optional) runs over all CTAs; each
// CTA posts its best (logit, index) and CTA 0 reduces them.  Every wait is bounded by
// %globaltimer: on expiry the kernel records FLINT_ERR_TIMEOUT, raises an abort flag
// that releases all other waits, and runs to the end without hanging.
#include <atomic>

#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kPWarps = 16;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kUnit = 8;            // SwiGLU outputs per unit (one 8-column chunk of down)
constexpr int kMaxRouterRows = kPThreads / 64;   // router rows per CTA (64 threads each)
static_assert((kMaxRouterRows & (kMaxRouterRows - 1)) == 0, "router rows: a power of two");
constexpr int kMaxRoutedUnits = 5;  // routed units per CTA and step (6 pieces each <= 32 lanes)
constexpr int kMaxSharedUnits = 4;  // shared units per CTA
constexpr int kMaxUnits = kMaxRoutedUnits + kMaxSharedUnits;
constexpr size_t kMaxDecodeSmem = 216 * 1024;   // dynamic; the static arrays take about 9 KB of the 227 KB
constexpr int kMaxCtas = 512;
// Sync words, each on its own 128-byte line.
constexpr int kSyncDone = 32, kSyncHead = 64, kSyncAbort = 96;
constexpr int kSyncWords = 128;
// Copies of the residual accumulator: unit u adds into copy u % kAccCopies, which
// spreads the atomic traffic; readers sum the copies in a fixed order.
constexpr int kAccCopies = 2;
constexpr int kTagBoardBytes = 128 * 1024;   // logit board copies (see decode_tag_copies)

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

// Publishes every write of this CTA made before the call, then bumps the counter
// (the barrier orders the CTA's writes before thread 0's release-add).
__device__ __forceinline__ void signal_count(unsigned* sync, int which) {
  __syncthreads();
  if (threadIdx.x == 0)
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(sync + which) : "memory");
}

// Router logits travel as tagged 64-bit words {value bits, step + 1}; a reader that
// sees its tag has the value written with it (one single-copy-atomic word), so no
// counter and no fence are needed.  The tags are cleared before each launch.
__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Waits (bounded) until *p carries `tag` and returns its value.
__device__ __forceinline__ float wait_tagged(const unsigned long long* p, unsigned tag, unsigned* sync) {
  unsigned polls = 0;
  unsigned long long t0 = 0;
  for (;;) {
    const unsigned long long v = ld_relaxed_u64(p);
    if ((unsigned)(v >> 32) == tag) return __uint_as_float((unsigned)v);
    if ((++polls & 63u) == 0) {
      if (ld_acquire_gpu(sync + kSyncAbort)) return 0.f;
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        raise_status(FLINT_ERR_TIMEOUT);
        atomicExch(sync + kSyncAbort, 1u);
        return 0.f;
      }
    }
  }
}

// Barrier `id` (1-15) over the first `n` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
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
// x_l is built once per CTA (thread t owns elements [4t, 4t+4); H <= 4 * 512).  Every
// CTA keeps the residual h_l in s_hx, bit-identical across CTAs:
//   layer 0:   x_0 = x[t] (bf16, used as is); h_0 = residual[t], or x[t]
//   layer l:   h_l = h_{l-1} + sum of the accumulator copies (fixed order);
//              x_l = bf16(h_l * r), r = 1/sqrt(mean(h_l^2) + eps)
// and the GEMV operand xf = f16(x_l * 2^k), 2^k putting max|x_l| in [2^14, 2^15).
// Sum of squares and max|h| come from one fixed-order block reduction, so every CTA
// derives the same r and k (max|bf16(h r)| = bf16(max|h| r): rounding is monotone).
struct Staged {
  float unscale;    // 2^-k
};

__device__ __forceinline__ Staged cta_stage(const float* acc, const uint16_t* x_bf16,
                                            const float* residual, int H, float eps, float* s_hx,
                                            uint16_t* s_xb, uint16_t* s_xf, float* s_red) {
  const int n = 4 * threadIdx.x;
  const bool own = n < H;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (own) {
    if (acc) {
      float4 f[kAccCopies];
#pragma unroll
      for (int c = 0; c < kAccCopies; ++c) f[c] = __ldcg(reinterpret_cast<const float4*>(acc + c * H + n));
      const float4 h = *reinterpret_cast<const float4*>(s_hx + n);
      v[0] = h.x; v[1] = h.y; v[2] = h.z; v[3] = h.w;
#pragma unroll
      for (int c = 0; c < kAccCopies; ++c) { v[0] += f[c].x; v[1] += f[c].y; v[2] += f[c].z; v[3] += f[c].w; }
      *reinterpret_cast<float4*>(s_hx + n) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      const uint2 b = __ldcg(reinterpret_cast<const uint2*>(x_bf16 + n));
      v[0] = bf16_bits_to_f32(b.x & 0xFFFFu); v[1] = bf16_bits_to_f32(b.x >> 16);
      v[2] = bf16_bits_to_f32(b.y & 0xFFFFu); v[3] = bf16_bits_to_f32(b.y >> 16);
      *reinterpret_cast<float4*>(s_hx + n) =
          residual ? make_float4(__ldcg(residual + n), __ldcg(residual + n + 1), __ldcg(residual + n + 2),
                                 __ldcg(residual + n + 3))
                   : make_float4(v[0], v[1], v[2], v[3]);
    }
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
  const float r = acc ? 1.0f / sqrtf(tot / (float)H + eps) : 1.0f;
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

// ---------------------------------------------------------------- units
// A unit is kUnit = 8 consecutive SwiGLU outputs of one expert (routed or shared): 8
// gate rows, 8 up rows, and the matching 8-column chunk of the down matrix (H rows x
// 4 code bytes, plus the H scale bytes of the 16-column block that holds it).  The
// decode-unit copy (flint.h) stores each unit as one block in this layout, which is
// also its shared-memory image:
struct UnitLayout {
  uint32_t gc, gs, uc, us, dc, ds, bytes;
  __host__ __device__ static UnitLayout of(int H) {
    UnitLayout u;
    u.gc = 0;
    u.gs = u.gc + kUnit * (H / 2);
    u.uc = u.gs + kUnit * (H / 16);
    u.us = u.uc + kUnit * (H / 2);
    u.dc = u.us + kUnit * (H / 16);
    u.ds = u.dc + H * 4;
    u.bytes = u.ds + H;
    return u;
  }
};

// Gate/up of n units from shared memory (unit u at buf + u * ub): their 16 n row dot
// products, by warps [w0, w0 + nw), with tensor scales (unit u: gate tsc[2 u s],
// up tsc[2 u s + 1], s = tsc_stride) and 2^-k applied, into s_gu[16 u + row].  A warp
// takes up to kGURows rows per pass and interleaves them, so that their load, FMA and
// shuffle latencies overlap.  No barrier.
constexpr int kGURows = 3;
template <int CPL>
__device__ __forceinline__ void units_gateup(const uint8_t* buf, uint32_t ub, int n, int H, const float* tsc,
                                             int tsc_stride, const XStage<CPL, 1>& xs, float* s_gu, int w0,
                                             int nw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const UnitLayout U = UnitLayout::of(H);
  const int R = 2 * kUnit * n, step = nw * RPP;
#pragma unroll 1
  for (int b0 = (warp - w0) * RPP; b0 < R; b0 += kGURows * step) {
    RowRegs<CPL> w[kGURows];
#pragma unroll
    for (int k = 0; k < kGURows; ++k) {
      const int r = b0 + k * step + slice;
      const int rc = r < R ? r : 0;
      const int q = rc % (2 * kUnit);
      const uint8_t* ubuf = buf + (size_t)(rc / (2 * kUnit)) * ub;
      const bool up = q >= kUnit;
      const int row = up ? q - kUnit : q;
      lds_row<CPL>(w[k], ubuf + (up ? U.uc : U.gc) + row * (H / 2), ubuf + (up ? U.us : U.gs) + row * (H / 16),
                   sl, LPR);
    }
    float v[kGURows];
#pragma unroll
    for (int k = 0; k < kGURows; ++k) v[k] = dot_row<CPL, 1>(w[k], xs);
#pragma unroll 1
    for (int o = LPR / 2; o; o >>= 1)
#pragma unroll
      for (int k = 0; k < kGURows; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
#pragma unroll
    for (int k = 0; k < kGURows; ++k) {
      const int r = b0 + k * step + slice;
      if (sl == 0 && r < R) {
        const int u = r / (2 * kUnit), q = r % (2 * kUnit);
        s_gu[r] = v[k] * tsc[2 * u * tsc_stride + (q >= kUnit ? 1 : 0)] * xs.unscale;
      }
    }
  }
}

// SwiGLU values of n units (warp 0; lane 8u + j holds output j of unit u), staged as
// hi/lo f16 pairs scaled by 2^k per unit: s_hs[u][0..4) hi pairs, [4..8) lo pairs,
// [8] the unit's down scale (down tensor scale x routing weight x 2^-k).
__device__ __forceinline__ void stage_swiglu(int n, const float* s_gu, const float* s_dscale,
                                             uint32_t* s_hs) {
  const int lane = threadIdx.x & 31;
  #pragma unroll 1
  for (int u0 = 0; u0 < n; u0 += 32 / kUnit) {
    const int u = u0 + lane / kUnit, j = lane % kUnit;
    const bool live = u < n;
    const float hj = live ? silu(s_gu[u * 2 * kUnit + j]) * s_gu[u * 2 * kUnit + kUnit + j] : 0.f;
    float amax = fabsf(hj);
#pragma unroll
    for (int o = kUnit / 2; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int k = f16_stage_exponent(amax);
    const float v = hj * exp2i(k);
    const float w = __shfl_down_sync(0xffffffffu, v, 1);      // the odd partner
    if (live && (j & 1) == 0) {
      const uint32_t hi = pack_f16x2_rn(v, w);
      float ha, hb;
      f16x2_to_f32x2(hi, ha, hb);
      s_hs[u * (kUnit + 1) + j / 2] = hi;
      s_hs[u * (kUnit + 1) + kUnit / 2 + j / 2] = pack_f16x2_rn(v - ha, w - hb);
    }
    if (live && j == 0) s_hs[u * (kUnit + 1) + kUnit] = __float_as_uint(s_dscale[u] * exp2i(-k));
  }
}

// Down contributions of one unit to this thread's rows [4t, 4t + 4), added into part[].
__device__ __forceinline__ void unit_down(const uint8_t* buf, int H, const uint32_t* hs, float (&part)[4]) {
  const UnitLayout U = UnitLayout::of(H);
  const int n0 = 4 * threadIdx.x;
  if (n0 >= H) return;
  uint32_t hh[kUnit / 2], hl[kUnit / 2];
#pragma unroll
  for (int q = 0; q < kUnit / 2; ++q) { hh[q] = hs[q]; hl[q] = hs[kUnit / 2 + q]; }
  const float scale = __uint_as_float(hs[kUnit]);
  const uint4 cw = *reinterpret_cast<const uint4*>(buf + U.dc + 4 * n0);
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(buf + U.ds + n0);
  const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t f[4];
    e2m1x8_to_f16x2x4(wv[q], f[0], f[1], f[2], f[3]);
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      fma2_f16(a0, a1, f[i], hh[i]);
      fma2_f16(b0, b1, f[i], hl[i]);
    }
    float s0, s1;
    f16x2_to_f32x2(e4m3x2_to_f16x2((sw >> (8 * q)) & 0xFFu), s0, s1);
    part[q] = fmaf((a0 + a1) + (b0 + b1), s0 * scale, part[q]);
  }
}

// ---------------------------------------------------------------- top-k
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// (key, index) a comes before b: larger key, or equal key and lower index.
__device__ __forceinline__ bool before(unsigned ka, int ia, unsigned kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Bitonic network over N register pairs, leaving them in `before` order.
template <int N>
__device__ __forceinline__ void sort_pairs(unsigned (&k)[N], int (&ix)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool first_half = (i & size) == 0;
          const bool swap = first_half ? before(k[j], ix[j], k[i], ix[i]) : before(k[i], ix[i], k[j], ix[j]);
          const unsigned tk = swap ? k[j] : k[i];
          const int ti = swap ? ix[j] : ix[i];
          k[j] = swap ? k[i] : k[j];
          ix[j] = swap ? ix[i] : ix[j];
          k[i] = tk;
          ix[i] = ti;
        }
      }
    }
  }
}

// Exact softmax top-k by one warp (see flint.h): the K largest logits, ties to the
// lower index, in that order; weights exp(l_i - l_0) / sum over the selected.  Lane l
// holds logits [PER*l, PER*l + PER) sorted; each round the warp takes the best head
// (one max-reduction; a second reduction only when heads tie) and its lane pops it.
template <int PER>
__device__ __noinline__ void topk_exact(const float* logits, int E, int K, int* s_sel, float* s_w) {
  const int lane = threadIdx.x & 31;
  unsigned key[PER];
  int idx[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    float l = (e < E) ? logits[e] : -INFINITY;
    l = (l == l) ? l : -INFINITY;
    key[i] = (e < E) ? order_key(l) : 0u;      // every live key is >= 1
    idx[i] = e;
  }
  if (PER > 1) sort_pairs<PER>(key, idx);
  unsigned my_key = 0u;
  int my_sel = 0;
  for (int s = 0; s < K; ++s) {
    const unsigned wk = __reduce_max_sync(0xffffffffu, key[0]);
    unsigned tie = __ballot_sync(0xffffffffu, key[0] == wk);
    if (tie & (tie - 1u)) {
      const unsigned wi = __reduce_min_sync(0xffffffffu, key[0] == wk ? (unsigned)idx[0] : 0xFFFFFFFFu);
      tie = __ballot_sync(0xffffffffu, key[0] == wk && (unsigned)idx[0] == wi);
    }
    const int wl = __ffs(tie) - 1;
    const int we = __shfl_sync(0xffffffffu, idx[0], wl);
    if (lane == s) { my_key = wk; my_sel = we; }
    if (lane == wl) {
#pragma unroll
      for (int i = 0; i + 1 < PER; ++i) { key[i] = key[i + 1]; idx[i] = idx[i + 1]; }
      key[PER - 1] = 0u;
      idx[PER - 1] = 0x7FFFFFFF;
    }
  }
  const float l = key_value(my_key);
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  const float p = lane < K ? expf(l - l0) : 0.f;
  float z = p;
#pragma unroll
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < K) { s_sel[lane] = my_sel; s_w[lane] = p / z; }
  __syncwarp();
}

// Fast path for E <= 256: one 32-bit key per logit = (upper 24 bits of the order key,
// 255 - index), so a single max-reduction per round yields both the winner and its
// index, and ties go to the lower index.  Dropping the low 8 bits of the order key can
// only misorder logits that agree in their upper 24 bits; such a pair among the K + 1
// best shows up as two consecutive winners with equal upper bits, and the exact path
// then decides.  Returns false (warp-uniform) in that case.
template <int PER>
__device__ __forceinline__ bool topk_fast(const float* logits, int E, int K, int* s_sel, float* s_w) {
  const int lane = threadIdx.x & 31;
  unsigned pk[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    float l = (e < E) ? logits[e] : -INFINITY;
    l = (l == l) ? l : -INFINITY;
    pk[i] = (e < E) ? ((order_key(l) & 0xFFFFFF00u) | (unsigned)(255 - e)) : 0u;
  }
  unsigned prev = 0u;
  bool exact = true;
  int my_sel = 0;
  for (int s = 0; s <= K; ++s) {                    // round K only checks the boundary
    unsigned m = pk[0];
#pragma unroll
    for (int i = 1; i < PER; ++i) m = max(m, pk[i]);
    const unsigned w = __reduce_max_sync(0xffffffffu, m);
    if (s > 0 && (w >> 8) == (prev >> 8) && w != 0u) exact = false;
    prev = w;
    if (s == K) break;
    const int e = 255 - (int)(w & 255u);
    if (lane == s) my_sel = e;
    if (lane == e / PER) {
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (i == e % PER) pk[i] = 0u;
    }
  }
  if (!exact) return false;
  float l = lane < K ? logits[my_sel] : 0.f;
  l = (l == l) ? l : -INFINITY;
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  const float p = lane < K ? expf(l - l0) : 0.f;
  float z = p;
#pragma unroll
  for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < K) { s_sel[lane] = my_sel; s_w[lane] = p / z; }
  __syncwarp();
  return true;
}

template <int PER>
__device__ __forceinline__ void topk_per(const float* logits, int E, int K, int* s_sel, float* s_w) {
  if (PER <= 8 && E <= 256 && topk_fast<PER>(logits, E, K, s_sel, s_w)) return;
  topk_exact<PER>(logits, E, K, s_sel, s_w);
}

__device__ __forceinline__ void topk_dispatch(const float* logits, int E, int K, int* s_sel,
                                              float* s_w) {
  const int per_lane = (E + 31) / 32;
  if (per_lane <= 1) topk_per<1>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 2) topk_per<2>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 4) topk_per<4>(logits, E, K, s_sel, s_w);
  else if (per_lane <= 8) topk_per<8>(logits, E, K, s_sel, s_w);
  else topk_per<16>(logits, E, K, s_sel, s_w);
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

// ---------------------------------------------------------------- copy issue (warp 0)
// Data-independent copies of a layer for CTA c: its router rows e = c, c + G, ...
__device__ __forceinline__ void issue_router_rows(const LayerPtrs& P, uint8_t* s_router, uint64_t* bar, int H,
                                               int c, int G, int my_rows) {
  const int lane = threadIdx.x & 31;
  if (my_rows == 0) return;
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)my_rows * H * 2);
  __syncwarp();
  if (lane < my_rows)
    bulk_g2s(s_router + (size_t)lane * H * 2, P.router_w + (size_t)(c + lane * G) * H, H * 2, bar);
}

// Shared units of a layer (warp 0; lane i fetches shared unit s_su[i] into buffer i):
// data-independent, issued one layer ahead.
__device__ __forceinline__ void issue_shared(const LayerPtrs& P, uint8_t* s_static, uint64_t* bar,
                                             const int* s_su, int my_sh, uint32_t unit_bytes) {
  const int lane = threadIdx.x & 31;
  if (my_sh == 0) return;
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)my_sh * unit_bytes);
  __syncwarp();
  if (lane < my_sh)
    bulk_g2s(s_static + (size_t)lane * unit_bytes, P.sh_units + (size_t)s_su[lane] * unit_bytes, unit_bytes, bar);
}

// ---------------------------------------------------------------- layer tables
// The per-layer values every step reads, held in shared memory one layer ahead (the
// kernel parameter's table sits in the constant bank, where each layer's first use
// would miss): the pointer table, the shared expert's three tensor scales and this
// CTA's router bias entries.
struct LayerSmem {
  LayerPtrs p;
  float sh_tsc[3];              // shared gate, up, down tensor scales
  float bias[kMaxRouterRows];   // router bias of rows c, c + G, ...
};
constexpr int kLayerWords = (int)(sizeof(LayerPtrs) / 8);
static_assert(sizeof(LayerPtrs) % 8 == 0 && kLayerWords <= 32, "layer table: at most 32 words");

// One warp: layer `l` into `dst`.
__device__ __forceinline__ void load_layer(const PersistArgs& a, int l, LayerSmem* dst, int c, int G,
                                           int my_rows) {
  const int lane = threadIdx.x & 31;
  const LayerPtrs& P = a.layer[l];
  if (lane < kLayerWords)
    reinterpret_cast<unsigned long long*>(&dst->p)[lane] = reinterpret_cast<const unsigned long long*>(&P)[lane];
  if (lane < 3) dst->sh_tsc[lane] = __ldg(lane == 0 ? P.sh_gate.tsc : lane == 1 ? P.sh_up.tsc : P.sh_down_tsc);
  if (lane < my_rows) dst->bias[lane] = P.router_bias ? __ldg(P.router_bias + c + lane * G) : 0.f;
}

// ---------------------------------------------------------------- the kernel
// Work of CTA c (of G) in every layer step, all CTAs running the same code:
//   router rows      e = c, c + G, ...                       (< E)
//   shared units     s = G-1-c, G-1-c + G, ...               (< Fs/8)
//   routed units     r = c, c + G, ...                       (< K*F/8)
// Routed units fill CTAs from the front and shared units from the back, so the
// busiest CTAs hold at most one unit more than the least busy.  Router rows and
// shared units do not depend on the data: their copies for the next step are issued
// as soon as this step has consumed them.
// Residual accumulators rotate over three buffers: step s adds its down contributions
// into B(s) = (s + 1) % 3, which the next step's staging reads; B(s + 1) is cleared
// by step s (each CTA a share), ordered before step s + 1's additions by the done
// counter.
template <int CPL>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const __grid_constant__ PersistArgs a) {
  __shared__ float s_gu[kMaxUnits * 2 * kUnit];
  __shared__ uint32_t s_hs[kMaxUnits * (kUnit + 1)];
  __shared__ float s_dscale[kMaxUnits];
  __shared__ float s_rp[kPWarps];
  __shared__ int s_sel[FLINT_MAX_TOP_K];
  __shared__ float s_w[FLINT_MAX_TOP_K];
  __shared__ float s_lsel[FLINT_MAX_TOP_K];
  __shared__ unsigned s_wmax[8];
  __shared__ int s_nc;
  __shared__ int s_slot[kMaxRoutedUnits], s_jrt[kMaxRoutedUnits], s_su[kMaxSharedUnits];
  __shared__ float s_bv[kPWarps];
  __shared__ int s_bi[kPWarps];
  __shared__ float s_red[2 * kPWarps];
  __shared__ float s_val[FLINT_MAX_EXPERTS];
  __shared__ unsigned long long s_c64[FLINT_MAX_EXPERTS];
  __shared__ LayerSmem s_ly[2];                      // layer tables, by step parity
  __shared__ float s_tsc[FLINT_MAX_TOP_K][3];         // selected experts: gate, up, down x weight
  __shared__ float s_rtsc[kMaxRoutedUnits][2];        // routed units: gate, up tensor scales
  __shared__ __align__(8) uint64_t s_bar_rr, s_bar_sh;
  __shared__ __align__(8) uint64_t s_bar_rt[kMaxRoutedUnits];
  extern __shared__ __align__(128) uint8_t s_dyn[];
  const int H = a.H;
  const UnitLayout U = UnitLayout::of(H);
  float* s_hx = reinterpret_cast<float*>(s_dyn);                       // [H] residual h
  uint16_t* s_xb = reinterpret_cast<uint16_t*>(s_hx + H);              // [H] x, bf16
  uint16_t* s_xf = s_xb + H;                                           // [H] x * 2^k, f16
  uint8_t* s_router = reinterpret_cast<uint8_t*>(s_xf + H);            // [RR][H] bf16 rows
  uint8_t* s_static = s_router + (size_t)a.max_router_rows * H * 2;   // shared units
  uint8_t* s_routed = s_static + (size_t)a.max_shared_units * U.bytes; // routed units
  float* s_etsc = reinterpret_cast<float*>(s_routed + (size_t)a.max_routed_units * U.bytes);  // [3][E]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, G = gridDim.x;
  const int LPR = H / (32 * CPL), sl = lane % LPR;
  const int n_sh = a.Fs / kUnit;                    // shared units
  const int per_slot = a.F / kUnit;                 // routed units per selected expert
  const int n_rt = a.K * per_slot;                  // routed units
  const int my_rows = c < a.E ? (a.E - 1 - c) / G + 1 : 0;
  const int my_sh = (G - 1 - c) < n_sh ? (n_sh - 1 - (G - 1 - c)) / G + 1 : 0;
  const int my_rt = c < n_rt ? (n_rt - 1 - c) / G + 1 : 0;
  const int nw_e = (a.E + 31) / 32;
  const int npw = nw_e < 8 ? nw_e : 8;              // warps that poll the logits; the rest
                                                    // run the shared gate/up meanwhile
  const unsigned long long* board = a.logits_tag + (size_t)(c % a.tag_copies) * a.tag_stride;
  unsigned* sync = a.bar;
  uint32_t ph_rr = 0, ph_sh = 0, ph_rt = 0;         // mbarrier parities

  if (warp == kPWarps - 1) load_layer(a, 0, &s_ly[0], c, G, my_rows);
  if (threadIdx.x == 0) {
    mbar_init(&s_bar_rr, 1);
    mbar_init(&s_bar_sh, 1);
    for (int i = 0; i < kMaxRoutedUnits; ++i) mbar_init(&s_bar_rt[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // this CTA's units: routed unit i is unit j of the expert in slot `slot`; shared
  // unit i is unit s_su[i] of the shared expert
  if (threadIdx.x < my_rt) {
    const int r = c + threadIdx.x * G;
    s_slot[threadIdx.x] = r / per_slot;
    s_jrt[threadIdx.x] = r % per_slot;
  }
  if (threadIdx.x < my_sh) s_su[threadIdx.x] = (G - 1 - c) + threadIdx.x * G;
  __syncthreads();

  if (warp == 0) {
    issue_router_rows(a.layer[0], s_router, &s_bar_rr, H, c, G, my_rows);
    issue_shared(a.layer[0], s_static, &s_bar_sh, s_su, my_sh, U.bytes);
  }

  unsigned step = 0;                                 // global layer step
  for (int t = 0; t < a.T; ++t) {
#pragma unroll 1
    for (int l = 0; l < a.L; ++l, ++step) {
      const LayerSmem& LY = s_ly[step & 1];
      const LayerPtrs& P = LY.p;
      float* acc_cur = a.acc + (step % 3) * (kAccCopies * H);         // B(step - 1)
      float* acc_out = a.acc + ((step + 1) % 3) * (kAccCopies * H);   // B(step)
      float* acc_clr = a.acc + ((step + 2) % 3) * (kAccCopies * H);   // B(step + 1)
      const int l_next = (l + 1 < a.L) ? l + 1 : 0;
      const bool more = (l + 1 < a.L) || (t + 1 < a.T);
      const unsigned tag = step + 1;
      if (threadIdx.x == 0) s_nc = 0;                // read after the barriers below
      // ---- h_l complete: stage x_l
      if (step > 0) wait_count(sync, kSyncDone, (unsigned)G * step);
      const Staged stg = cta_stage(l == 0 ? nullptr : acc_cur, a.x + (size_t)t * H,
                                   (l == 0 && a.residual) ? a.residual + (size_t)t * H : nullptr,
                                   H, a.eps, s_hx, s_xb, s_xf, s_red);
      // ---- clear this CTA's share of B(step + 1) (published by this step's done signal)
#pragma unroll 1
      for (int n = 4 * (c + G * threadIdx.x); n < H; n += 4 * G * kPThreads)
#pragma unroll
        for (int cp = 0; cp < kAccCopies; ++cp)
          *reinterpret_cast<float4*>(acc_clr + cp * H + n) = make_float4(0.f, 0.f, 0.f, 0.f);
      // ---- router rows -> tagged logits; row r takes threads [64 r, 64 r + 64)
      if (my_rows > 0) {
        mbar_wait(&s_bar_rr, ph_rr, sync);
        ph_rr ^= 1;
        const int r = threadIdx.x >> 6, tr = threadIdx.x & 63;
        float acc = 0.f;
        if (r < my_rows) {
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          const uint16_t* row = reinterpret_cast<const uint16_t*>(s_router) + (size_t)r * H;
#pragma unroll 1
          for (int e = 8 * tr; e < H; e += 8 * 64) {
            const uint4 wv = *reinterpret_cast<const uint4*>(row + e);
            const uint4 xv = *reinterpret_cast<const uint4*>(s_xb + e);
            fma2_bf16(a0, a1, wv.x, xv.x);
            fma2_bf16(a2, a3, wv.y, xv.y);
            fma2_bf16(a0, a1, wv.z, xv.z);
            fma2_bf16(a2, a3, wv.w, xv.w);
          }
          acc = (a0 + a1) + (a2 + a3);
        }
        acc = sum_lanes<32>(acc);
        if (lane == 0) s_rp[warp] = acc;
        __syncthreads();
        // every board copy gets the rows (thread 8 q + rr: copy q, row rr); readers
        // spread their polls over the copies
        const int rr = threadIdx.x & (kMaxRouterRows - 1);
        if (rr < my_rows) {
          const float v = (s_rp[2 * rr] + s_rp[2 * rr + 1]) + LY.bias[rr];
          const unsigned long long word = ((unsigned long long)tag << 32) | __float_as_uint(v);
#pragma unroll 1
          for (int cp = threadIdx.x / kMaxRouterRows; cp < a.tag_copies; cp += kPThreads / kMaxRouterRows)
            st_tagged(a.logits_tag + (size_t)cp * a.tag_stride + c + rr * G, word);
        }
      }
      XStage<CPL, 1> xs;
      pairs_from_smem<CPL>(xs.p[0], s_xf, sl, LPR);
      xs.unscale = stg.unscale;
      if (warp < npw) {
        // ---- top-k.  Warps [0, npw) poll the logits (thread i: logits i, i + 32 npw, ...).
        // The K-th largest warp maximum is a threshold that the K best logits all reach
        // (at least K warps hold a logit at or above it); the logits at or above it are
        // ranked exactly by (value, lower index first).
        unsigned wmax = 0u;                            // every logit's order key is >= 1
#pragma unroll 1
        for (int e = threadIdx.x; e < a.E; e += npw * 32) {
          // the expert's tensor scales load while its logit is awaited
          const float tg = __ldg(P.gate.tsc + e), tu = __ldg(P.up.tsc + e), td = __ldg(P.down_tsc + e);
          float v = wait_tagged(board + e, tag, sync);
          s_etsc[e] = tg;
          s_etsc[a.E + e] = tu;
          s_etsc[2 * a.E + e] = td;
          v = (v == v) ? v : -INFINITY;
          s_val[e] = v;
          wmax = max(wmax, order_key(v));
        }
        wmax = __reduce_max_sync(0xffffffffu, wmax);
        if (lane == 0) s_wmax[warp] = wmax;
        named_bar(1, npw * 32);
        unsigned thr = 0u;
        if (npw >= a.K) {
          const unsigned m = lane < npw ? s_wmax[lane] : 0u;
          int ge = 0;
#pragma unroll 1
          for (int u = 0; u < npw; ++u) ge += __shfl_sync(0xffffffffu, m, u) >= m ? 1 : 0;
          thr = __reduce_max_sync(0xffffffffu, (lane < npw && ge >= a.K) ? m : 0u);
        }
#pragma unroll 1
        for (int e0 = warp * 32; e0 < a.E; e0 += npw * 32) {
          const int e = e0 + lane;
          const unsigned key = e < a.E ? order_key(s_val[e]) : 0u;
          const bool cand = key != 0u && key >= thr;
          const unsigned bal = __ballot_sync(0xffffffffu, cand);
          int base = 0;
          if (lane == 0 && bal) base = atomicAdd(&s_nc, __popc(bal));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (cand) s_c64[base + __popc(bal & ((1u << lane) - 1u))] = ((unsigned long long)key << 32) | (unsigned)(~e);
        }
        named_bar(1, npw * 32);
        const int n = s_nc;
#pragma unroll 1
        for (int j = threadIdx.x; j < n; j += npw * 32) {
          const unsigned long long ck = s_c64[j];
          int rank = 0;
#pragma unroll 1
          for (int m = 0; m < n; ++m) rank += s_c64[m] > ck ? 1 : 0;
          if (rank < a.K) {
            const int e = (int)(~(unsigned)ck);
            s_sel[rank] = e;
            s_lsel[rank] = s_val[e];
          }
        }
        named_bar(1, npw * 32);
        if (warp == 0) {
          // routed copies first: they gate the critical path
          if (lane < my_rt) mbar_expect_tx(&s_bar_rt[lane], U.bytes);
          __syncwarp();
          if (lane < my_rt) {
            int e = s_sel[s_slot[lane]];
            if (e < 0 || e >= a.E) { raise_status(FLINT_ERR_INVALID_ARG); e = 0; }
            bulk_g2s(s_routed + (size_t)lane * U.bytes,
                     P.units + ((size_t)e * per_slot + s_jrt[lane]) * U.bytes, U.bytes, &s_bar_rt[lane]);
          }
        }
        if (warp == (npw > 1 ? 1 : 0)) {
          // routing weights: the selected scores (softmax or sigmoid), renormalised
          const float lv = lane < a.K ? s_lsel[lane] : 0.f;
          const float l0 = __shfl_sync(0xffffffffu, lv, 0);
          const float pr = lane >= a.K ? 0.f
                           : P.router_score == FLINT_ROUTER_SIGMOID ? 1.0f / (1.0f + expf(-lv))
                                                                    : expf(lv - l0);
          float z = pr;
#pragma unroll
          for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
          if (lane < a.K) {
            const int e = s_sel[lane];
            const bool ok = e >= 0 && e < a.E;
            s_w[lane] = pr / z;
            s_tsc[lane][0] = ok ? s_etsc[e] : 0.f;
            s_tsc[lane][1] = ok ? s_etsc[a.E + e] : 0.f;
            s_tsc[lane][2] = ok ? s_etsc[2 * a.E + e] * (pr / z) : 0.f;
          }
          __syncwarp();
          if (lane < my_rt) {
            s_rtsc[lane][0] = s_tsc[s_slot[lane]][0];
            s_rtsc[lane][1] = s_tsc[s_slot[lane]][1];
          }
        }
      } else {
        // ---- shared units' gate/up by the warps that do not poll; the last of them
        // then fetches the next layer's table
        if (my_sh > 0) {
          mbar_wait(&s_bar_sh, ph_sh, sync);
          units_gateup<CPL>(s_static, U.bytes, my_sh, H, LY.sh_tsc, 0, xs, s_gu, npw, kPWarps - npw);
        }
        if (more && warp == kPWarps - 1) load_layer(a, l_next, &s_ly[(step + 1) & 1], c, G, my_rows);
      }
      if (my_sh > 0) ph_sh ^= 1;
      if (threadIdx.x < my_sh) s_dscale[threadIdx.x] = LY.sh_tsc[2];
      __syncthreads();                               // s_sel, s_w and the shared s_gu visible
      const LayerPtrs& PN = s_ly[(step + 1) & 1].p;   // next layer (written before the barrier above)
      if (more && warp == 0) issue_router_rows(PN, s_router, &s_bar_rr, H, c, G, my_rows);
      if (c == 0 && threadIdx.x < a.K) {
        const size_t o = ((size_t)t * a.L + l) * a.K + threadIdx.x;
        if (a.idx_out) a.idx_out[o] = s_sel[threadIdx.x];
        if (a.w_out) a.w_out[o] = s_w[threadIdx.x];
      }
      // ---- group 0: the shared units (SwiGLU and down while the routed copies are in
      // flight); group 1: the routed units, each gate/up as soon as its copy lands
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        const int n = g ? my_rt : my_sh;
        const int off = g ? my_sh : 0;
        const uint8_t* ubase = g ? s_routed : s_static;
        if (g) {
          // all routed units at once (they land close together; the interleaved rows
          // hide each other's latency)
#pragma unroll 1
          for (int i = 0; i < my_rt; ++i) mbar_wait(&s_bar_rt[i], ph_rt, sync);
          units_gateup<CPL>(s_routed, U.bytes, my_rt, H, &s_rtsc[0][0], 1, xs, s_gu + my_sh * 2 * kUnit, 0, kPWarps);
          if (threadIdx.x < my_rt) s_dscale[my_sh + threadIdx.x] = s_tsc[s_slot[threadIdx.x]][2];
          ph_rt ^= 1;
          __syncthreads();
          // the shared-unit buffers are free again
          if (more && warp == 0) issue_shared(PN, s_static, &s_bar_sh, s_su, my_sh, U.bytes);
        }
        if (n > 0) {
          if (warp == 0) stage_swiglu(n, s_gu + off * 2 * kUnit, s_dscale + off, s_hs + off * (kUnit + 1));
          __syncthreads();
#pragma unroll 1
          for (int u = 0; u < n; ++u) unit_down(ubase + (size_t)u * U.bytes, H, s_hs + (off + u) * (kUnit + 1), part);
        }
      }
      if (my_sh + my_rt > 0 && 4 * threadIdx.x < H)
        red_add_v4(acc_out + (c % kAccCopies) * H + 4 * threadIdx.x, part[0], part[1], part[2], part[3]);
      signal_count(sync, kSyncDone);                 // begins with a CTA barrier
    }
    // ---------------- outputs of token t
    wait_count(sync, kSyncDone, (unsigned)G * step);
    const float* hfin = a.acc + (step % 3) * (kAccCopies * H);         // B(step - 1)
    const Staged stg = cta_stage(hfin, nullptr, nullptr, H, a.eps, s_hx, s_xb, s_xf, s_red);
    if (a.out)
      for (int n = c * kPThreads + threadIdx.x; n < H; n += G * kPThreads) a.out[(size_t)t * H + n] = s_hx[n];
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
        wait_count(sync, kSyncHead, (unsigned)G * (t + 1));
        if (warp == 0) {
          const int ln = threadIdx.x & 31;
          float v = -INFINITY;
          int i = 0x7FFFFFFF;
          for (int k = ln; k < G; k += 32) {
            const float kv = __ldcg(best_v + k);
            const int ki = __ldcg(best_i + k);
            if (kv > v || (kv == v && ki < i)) { v = kv; i = ki; }
          }
          best_reduce_warp(v, i);
          if (ln == 0 && a.argmax) a.argmax[t] = (i < a.V) ? i : 0;
        }
      }
    }
    __syncthreads();                                 // s_hx is rewritten by the next token
  }
  // No bulk copy is in flight at exit: copies are issued only while `more` holds (or
  // for the current step), and every issued copy is waited for in the step it serves.
}

// ---------------------------------------------------------------- decode-unit pack
// CTA (q, m) builds units 4q .. 4q + 3 of matrix m (see UnitLayout): gate/up rows
// 32q .. 32q + 31 split by 8, and the down codes of columns 32q .. 32q + 31 (16 bytes
// per row) with the scales of blocks 2q, 2q + 1 spread over the four units.
__device__ __forceinline__ void copy16(uint8_t* dst, const uint8_t* src, uint32_t bytes) {
  for (uint32_t i = threadIdx.x; i < bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
}

__global__ void k_unit_pack(NVPtr gate, NVPtr up, NVPtr down, int H, int F, uint8_t* __restrict__ units) {
  const int m = blockIdx.y, q = blockIdx.x;
  const UnitLayout L = UnitLayout::of(H);
  uint8_t* out = units + ((size_t)m * (F / kUnit) + 4 * q) * L.bytes;
#pragma unroll 1
  for (int u = 0; u < 4; ++u) {
    uint8_t* o = out + (size_t)u * L.bytes;
    const size_t row0 = (size_t)m * F + 32 * q + kUnit * u;
    copy16(o + L.gc, gate.codes + row0 * (H / 2), kUnit * (H / 2));
    copy16(o + L.gs, gate.scales + row0 * (H / 16), kUnit * (H / 16));
    copy16(o + L.uc, up.codes + row0 * (H / 2), kUnit * (H / 2));
    copy16(o + L.us, up.scales + row0 * (H / 16), kUnit * (H / 16));
  }
  for (int r = threadIdx.x; r < H; r += blockDim.x) {
    const size_t row = (size_t)m * H + r;
    const uint4 v = *reinterpret_cast<const uint4*>(down.codes + row * (F / 2) + 16 * q);
    const uint8_t s0 = down.scales[row * (F / 16) + 2 * q], s1 = down.scales[row * (F / 16) + 2 * q + 1];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      *reinterpret_cast<uint32_t*>(out + (size_t)u * L.bytes + L.dc + 4 * r) = w[u];
      out[(size_t)u * L.bytes + L.ds + r] = u < 2 ? s0 : s1;
    }
  }
}

cudaError_t launch_unit_pack(const NVPtr& gate, const NVPtr& up, const NVPtr& down, int n_mat, int H,
                             int F, uint8_t* units, cudaStream_t st) {
  k_unit_pack<<<dim3(F / 32, n_mat), 256, 0, st>>>(gate, up, down, H, F, units);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host side
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes at the start of the workspace that every launch clears: sync words + tags.
// Copies of the logit board: each logit is written to every copy and CTA c polls copy
// c % copies, so the polls of all CTAs do not pile onto the same few L2 lines.
int decode_tag_stride(int E) { return (E + 15) & ~15; }   // 128-byte rows
int decode_tag_copies(int E) {
  const int c = kTagBoardBytes / (8 * decode_tag_stride(E));
  return c < 1 ? 1 : (c > kMaxCtas ? kMaxCtas : c);
}

static size_t decode_cleared_bytes(int H, int E, int copies) {
  return sizeof(unsigned) * kSyncWords +
         align256(sizeof(unsigned long long) * decode_tag_stride(E) * copies) +
         align256(sizeof(float) * 3 * kAccCopies * H);
}

size_t decode_workspace_bytes(int H, int E, int copies) {
  return decode_cleared_bytes(H, E, copies) + 2 * align256(2 * kMaxCtas * sizeof(float));
}

void decode_carve(PersistArgs& a, void* ws) {
  char* p = static_cast<char*>(ws);
  a.bar = reinterpret_cast<unsigned*>(p); p += sizeof(unsigned) * kSyncWords;
  a.tag_stride = decode_tag_stride(a.E);
  a.logits_tag = reinterpret_cast<unsigned long long*>(p);
  p += align256(sizeof(unsigned long long) * a.tag_stride * a.tag_copies);
  a.acc = reinterpret_cast<float*>(p); p += align256(sizeof(float) * 3 * kAccCopies * a.H);
  a.best_v = reinterpret_cast<float*>(p); p += align256(2 * kMaxCtas * sizeof(float));
  a.best_i = reinterpret_cast<int*>(p);
}

// SM count of each device, looked up on the first launch from that device (the value
// is the same for every thread that stores it, so a relaxed atomic is enough).
constexpr int kMaxDevices = 64;
static std::atomic<int> g_sms[kMaxDevices];
int decode_grid() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (n > kMaxCtas) n = kMaxCtas;
    g_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

DecodePlan decode_plan(int H, int E, int K, int F, int Fs, int G) {
  DecodePlan p = {};
  if (G <= 0) return p;                              // no device
  p.router_rows = (E + G - 1) / G;
  p.shared_units = (Fs / kUnit + G - 1) / G;
  p.routed_units = (K * (F / kUnit) + G - 1) / G;
  p.smem = (size_t)H * (4 + 2 + 2) + (size_t)p.router_rows * H * 2 +
           (size_t)(p.shared_units + p.routed_units) * UnitLayout::of(H).bytes +
           (size_t)3 * E * sizeof(float);
  p.ok = p.router_rows <= kMaxRouterRows && p.routed_units <= kMaxRoutedUnits &&
         p.shared_units <= kMaxSharedUnits &&
         p.smem <= kMaxDecodeSmem && F % (2 * kUnit) == 0 && Fs % (2 * kUnit) == 0;
  return p;
}

template <int CPL>
static cudaError_t launch_persistent_cpl(const PersistArgs& a, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<CPL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(decode_grid());
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

// a.max_router_rows / a.max_shared_units must hold decode_plan's counts.
cudaError_t launch_persistent(const PersistArgs& a, cudaStream_t st) {
  const DecodePlan p = decode_plan(a.H, a.E, a.K, a.F, a.Fs, decode_grid());
  if (!p.ok || a.max_router_rows != p.router_rows || a.max_shared_units != p.shared_units ||
      a.max_routed_units != p.routed_units)
    return cudaErrorInvalidConfiguration;
  if (a.tag_copies < 1) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.bar, 0, decode_cleared_bytes(a.H, a.E, a.tag_copies), st);
  if (e != cudaSuccess) return e;
  if (a.H <= 1024) return launch_persistent_cpl<1>(a, p.smem, st);
  return launch_persistent_cpl<2>(a, p.smem, st);
}

}  // namespace flint
