// decode.cu -- persistent decode kernel: T tokens x L chained Flint MoE layers (+ head)
// in one launch of clusters of 16 CTAs (one CTA per SM).
//
// The layer ("Flint: 125 tokens a second is what 2.5B active parameters buy at 273
// GB/s", section "The shape, read from the headers"; "Recursive Releases Flint, a 40B
// MoE Coding Model That Runs Locally at 125 Tokens per Second", section "How does
// Flint's architecture work?") reads every active weight once per token and has one
// dependency no schedule can hide: which experts are read depends on the router.  At
// batch 1 the step is a chain of latencies, so the design minimises the exchanges
// between SMs on that chain:
//
//   * The work of a layer is a set of groups: one per selected expert, plus the shared
//     expert (a run of parts of width F).  Cluster c runs its groups (the routed
//     clusters one selected expert each, the last cluster the shared expert).  The
//     cluster's 16 CTAs split each part's gate/up rows (n = W/16 SwiGLU outputs each),
//     swap the SwiGLU values through distributed shared memory, and each CTA then
//     applies the group's down columns to its own H/16 output rows.  Gate/up rows and
//     down rows are contiguous pieces of the row-major NVFP4 stacks, moved by TMA bulk
//     copies (a group that does not span whole down rows takes them by cp.async).
//   * Every routed cluster computes all E router logits itself (E/16 rows per CTA,
//     staged in shared memory a step ahead) and swaps them through distributed shared
//     memory, so routing needs no exchange between clusters.  The top-k runs in every
//     CTA of the cluster on the same logits.
//   * The only exchange between clusters is the residual: CTA (c, j) posts its partial
//     sums of rows R_j = [j H/16, (j+1) H/16) as tagged 64-bit words {value, step + 1}
//     (no fence, no counter, no atomics); CTA j of every cluster reads all clusters'
//     words of R_j and adds them in one fixed order, so every cluster computes
//     bit-identical h rows, which the cluster then gathers through distributed shared
//     memory.  Every sum has a fixed order: runs repeat bit for bit.
//   * The head: after a token's last layer every CTA streams its share of the head rows
//     through a two-slot ring of TMA bulk copies; each posts its best (value, index) and
//     the last CTA reduces them.
//
// Within a cluster every hand-off (logits, SwiGLU values, h) is st.async into the
// receivers' shared memory, completing bytes on their mbarriers: a CTA waits for the
// data it needs, not for the cluster, and no cluster barrier remains in a step.  The
// copies of the next step that do not depend on its data go out a step ahead, and a
// routed expert's copies are described before the top-k ends.  Every wait on another
// CTA or on a copy is bounded by %globaltimer: on expiry the kernel records
// FLINT_ERR_TIMEOUT, raises an abort flag that releases every other wait, stops issuing
// copies and runs to its end.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {
namespace dc {

constexpr int kCS = kDecCluster;
constexpr int kThreads = kDecThreads;
constexpr int kWarps = kThreads / 32;
static_assert(kWarps >= 8 && (kWarps & (kWarps - 1)) == 0, "warps per CTA: a power of two, at least 8");
constexpr int kRouterBytes = 64 * 1024;   // router rows of one CTA
constexpr int kBigBytes = 172 * 1024;     // router rows + group buffer, or the head ring
constexpr int kMaxW = 1024;               // down columns of a group (one 32-column chunk per lane)
constexpr int kMaxE = 256;                // experts of a routed layer
constexpr int kMaxRR = kMaxE / kDecCluster;   // router rows per CTA
constexpr int kMaxN = 64;                 // SwiGLU outputs per CTA and part
constexpr int kMaxParts = 16;             // parts of a group (at least 4 SwiGLU values per CTA and part)
static_assert(kMaxParts * 4 * kDecCluster >= kMaxW, "parts of a group");
constexpr int kMaxG = kDecMaxClusters * kCS;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders the cluster's shared-memory writes
// before the barrier against its reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void* local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}
// One float to `dst` in CTA `peer`, completing 4 bytes on that CTA's barrier `bar`.
__device__ __forceinline__ void st_async1(float* dst, float v, uint64_t* bar, int peer) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               :: "r"(peer_addr(dst, peer)), "r"(__float_as_uint(v)), "r"(peer_addr(bar, peer)) : "memory");
}
// n 16-byte pieces of `src` (local shared memory) to `dst` in every CTA of the cluster,
// each completing its bytes on that CTA's barrier `bar` (st.async: the receiver waits on
// bar instead of a cluster barrier).
__device__ __forceinline__ void to_cluster_async(float* dst, const float* src, int n, uint64_t* bar) {
#pragma unroll 1
  for (int i = threadIdx.x; i < kCS * n; i += kThreads) {
    const int peer = i / n, k = i - peer * n;
    const float4 v = *reinterpret_cast<const float4*>(src + 4 * k);
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(peer_addr(dst + 4 * k, peer)), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w),
                    "r"(peer_addr(bar, peer)) : "memory");
  }
}
__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_abort(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void give_up(unsigned* sync) {
  raise_status(FLINT_ERR_TIMEOUT);
  atomicExch(sync, 1u);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(smem_addr(b)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for a copy phase (every thread that reads the data waits itself).
// ... a phase completed by other CTAs' st.async (acquire at cluster scope).
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(smem_addr(b)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __noinline__ void mbar_wait_cluster(uint64_t* b, uint32_t parity, unsigned* sync, unsigned long long limit) {
  unsigned long long t0 = 0;
  for (unsigned polls = 1; !mbar_try_cluster(b, parity); ++polls) {
    if ((polls & 63u) == 0) {
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit) {
        give_up(sync);
        return;
      }
    }
  }
}
__device__ __noinline__ void mbar_wait(uint64_t* b, uint32_t parity, unsigned* sync, unsigned long long limit) {
  unsigned long long t0 = 0;
  for (unsigned polls = 1; !mbar_try(b, parity); ++polls) {
    if ((polls & 63u) == 0) {
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit) {
        give_up(sync);
        return;
      }
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst)), "l"(src) : "memory");
}
// This thread's earlier cp.asyncs count as one arrival on b once they have landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_addr(b)) : "memory");
}
// ... the same without counting as an arrival: it only holds the phase open until they land.
__device__ __forceinline__ void cp_async_arrive_hold(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(smem_addr(b)) : "memory");
}
__host__ __device__ __forceinline__ uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }

// ---------------------------------------------------------------- staging
// x operand of the row dots, lane-major: with LPR lanes per row and chunk c = sl + LPR i
// (32 elements) taken by lane sl, s_xl[(4 i + w) LPR + sl] holds the f16 pairs of
// elements [32 c + 8 w, 32 c + 8 w + 8) -- one conflict-free 16-byte load per word.
__device__ __forceinline__ int xl_index(int e, int LPR) {
  const int cidx = e >> 5, w = (e >> 3) & 3;
  return ((4 * (cidx / LPR) + w) * LPR + cidx % LPR) * 4 + ((e & 7) >> 1);
}

// Thread t owns elements [4t, 4t + 4) (H <= 4 * kThreads).  One fixed-order block
// reduction: every CTA derives the same scale from the same data.
//   input: x = x[t] as given, h = residual[t] (or x[t])      (a token's first layer)
//   else:  x = bf16(h / sqrt(mean(h^2) + eps)), gain 1        (later layers, the head)
// s_xb = x; s_xl = f16(x * 2^k) as above, 2^k putting max|x| in [2^14, 2^15) (max|bf16(h
// r)| = bf16(max|h| r): rounding is monotone).  Returns 2^-k.
__device__ __forceinline__ float stage(const uint16_t* xg, const float* rg, bool input, int H, int LPR, float eps,
                                    float* s_h, uint16_t* s_xb, uint32_t* s_xl, float* s_red) {
  const int n = 4 * threadIdx.x;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  uint16_t b[4] = {0, 0, 0, 0};
  if (n < H) {
    if (input) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(xg + n));
      b[0] = (uint16_t)(w.x & 0xFFFFu); b[1] = (uint16_t)(w.x >> 16);
      b[2] = (uint16_t)(w.y & 0xFFFFu); b[3] = (uint16_t)(w.y >> 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = bf16_bits_to_f32(b[q]);
      const float4 h = rg ? make_float4(__ldg(rg + n), __ldg(rg + n + 1), __ldg(rg + n + 2), __ldg(rg + n + 3))
                          : make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(s_h + n) = h;
    } else {
      const float4 h = *reinterpret_cast<const float4*>(s_h + n);
      v[0] = h.x; v[1] = h.y; v[2] = h.z; v[3] = h.w;
    }
  }
  float ss = 0.f, am = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) { ss = fmaf(v[q], v[q], ss); am = fmaxf(am, fabsf(v[q])); }
  ss = sum_lanes<32>(ss);
#pragma unroll
  for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { s_red[warp] = ss; s_red[kWarps + warp] = am; }
  __syncthreads();
  // the kWarps partials in 16-byte loads, summed in one fixed order
  const float4* r4 = reinterpret_cast<const float4*>(s_red);
  float4 q[kWarps / 2];
#pragma unroll
  for (int i = 0; i < kWarps / 2; ++i) q[i] = r4[i];
  float ps[kWarps / 4], pm[kWarps / 4];
#pragma unroll
  for (int i = 0; i < kWarps / 4; ++i) {
    ps[i] = (q[i].x + q[i].y) + (q[i].z + q[i].w);
    const float4 m = q[kWarps / 4 + i];
    pm[i] = fmaxf(fmaxf(m.x, m.y), fmaxf(m.z, m.w));
  }
#pragma unroll
  for (int w = kWarps / 8; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) { ps[i] += ps[i + w]; pm[i] = fmaxf(pm[i], pm[i + w]); }
  const float tot = ps[0], amax = pm[0];
  float xmax = amax;
  if (!input) {
    const float r = rsqrtf(__fdividef(tot, (float)H) + eps);
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = f32_to_bf16_rn(v[q] * r);
    xmax = bf16_bits_to_f32(f32_to_bf16_rn(amax * r));
  }
  const int k = f16_stage_exponent(xmax);
  const float s = exp2i(k);
  if (n < H) {
    *reinterpret_cast<uint2*>(s_xb + n) =
        make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16), (uint32_t)b[2] | ((uint32_t)b[3] << 16));
    const uint32_t f01 = pack_f16x2_rn(bf16_bits_to_f32(b[0]) * s, bf16_bits_to_f32(b[1]) * s);
    const uint32_t f23 = pack_f16x2_rn(bf16_bits_to_f32(b[2]) * s, bf16_bits_to_f32(b[3]) * s);
    *reinterpret_cast<uint2*>(s_xl + xl_index(n, LPR)) = make_uint2(f01, f23);
  }
  __syncthreads();
  return exp2i(-k);
}

// ---------------------------------------------------------------- row dots
// Rows [0, nrows) of an NVFP4 block in shared memory (codes rows of H/2 bytes, then, at
// `scales`, rows of H/16 bytes) dotted with x (s_xl); out[r] = dot * (r < nsplit ? s0 :
// s1).  A warp takes four rows at a time (slices of LPR lanes) and walks their 32-element
// chunks; one copy serves the gate/up parts and the head.
template <int CPL>
__device__ __noinline__ void rows_dot(const uint8_t* codes, const uint8_t* scales, int nrows, int nsplit, float s0,
                                      float s1, int H, const uint4* s_xl, float* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = H / (32 * CPL), RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int step = kWarps * RPP;
#pragma unroll 1
  for (int b0 = warp * RPP; b0 < nrows; b0 += 4 * step) {
    int row[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = b0 + k * step + slice;
      row[k] = r < nrows ? r : 0;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int cidx = sl + LPR * i;
      uint32_t xp[16];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 q = s_xl[(4 * i + w) * LPR + sl];
        xp[4 * w] = q.x; xp[4 * w + 1] = q.y; xp[4 * w + 2] = q.z; xp[4 * w + 3] = q.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 cw = *reinterpret_cast<const uint4*>(codes + (size_t)row[k] * (H / 2) + 16 * cidx);
        const uint32_t sw = *reinterpret_cast<const uint16_t*>(scales + (size_t)row[k] * (H / 16) + 2 * cidx);
        const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
        float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t h[4];
          e2m1x8_to_f16x2x4(wv[w], h[0], h[1], h[2], h[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) fma2_f16(a[w >> 1][0], a[w >> 1][1], h[e], xp[4 * w + e]);
        }
        float c0, c1;
        f16x2_to_f32x2(e4m3x2_to_f16x2(sw), c0, c1);
        acc[k] = fmaf(a[0][0] + a[0][1], c0, acc[k]);
        acc[k] = fmaf(a[1][0] + a[1][1], c1, acc[k]);
      }
    }
#pragma unroll 1
    for (int m = LPR / 2; m; m >>= 1)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], m);
    if (sl == 0)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = b0 + k * step + slice;
        if (r < nrows) out[r] = acc[k] * (r < nsplit ? s0 : s1);
      }
  }
}

// ---------------------------------------------------------------- router and top-k
// Router rows [r0, r0 + nr) (nr <= kMaxRR) from shared memory, bf16 x bf16 with fp32
// accumulation, plus the bias; every CTA of the cluster receives them (4 bytes each on
// its bar_lg).  Thread t takes
// columns [4 q, 4 q + 4), q = t, t + kThreads, ..., of every row (x read once per CTA);
// a warp reduces its sixteen row partials by halving exchanges (lane pair 2 m, 2 m + 1
// ends with row m), the warps' partials meet in s_rp in a fixed order.
// One halving exchange: lanes with bit O set keep rows [Hh, 2 Hh) of their current 2 Hh,
// the others rows [0, Hh); each adds its partner's copy of the rows it keeps.
template <int O, int Hh>
__device__ __forceinline__ void halve_rows(float (&p)[kMaxRR], int lane) {
  const bool up = (lane & O) != 0;
#pragma unroll
  for (int i = 0; i < Hh; ++i) {
    const float send = up ? p[i] : p[i + Hh];
    const float keep = up ? p[i + Hh] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}
__device__ __noinline__ void router_rows(const uint16_t* s_router, const uint16_t* s_xb, int H, int r0, int nr,
                                         const float* bias, float* s_rp, float* s_lg, uint64_t* bar_lg) {
  static_assert(kMaxRR == 16 && kWarps * kMaxRR <= 256, "router partials");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float p[kMaxRR], ph[kMaxRR];
#pragma unroll
  for (int r = 0; r < kMaxRR; ++r) { p[r] = 0.f; ph[r] = 0.f; }
#pragma unroll 1
  for (int q = threadIdx.x; q < H / 4; q += kThreads) {
    const uint2 x = *reinterpret_cast<const uint2*>(s_xb + 4 * q);
#pragma unroll
    for (int r = 0; r < kMaxRR; ++r)
      if (r < nr) {
        const uint2 w = *reinterpret_cast<const uint2*>(s_router + (size_t)r * H + 4 * q);
        fma2_bf16(p[r], ph[r], w.x, x.x);
        fma2_bf16(p[r], ph[r], w.y, x.y);
      }
  }
#pragma unroll
  for (int r = 0; r < kMaxRR; ++r) p[r] += ph[r];
  halve_rows<16, 8>(p, lane);
  halve_rows<8, 4>(p, lane);
  halve_rows<4, 2>(p, lane);
  halve_rows<2, 1>(p, lane);
  p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
  if ((lane & 1) == 0) s_rp[warp * kMaxRR + (lane >> 1)] = p[0];
  __syncthreads();
  if (threadIdx.x < kMaxRR * kCS) {
    const int r = threadIdx.x % kMaxRR, peer = threadIdx.x / kMaxRR;
    if (r < nr) {
      float v[kWarps];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v[w] = s_rp[w * kMaxRR + r];
#pragma unroll
      for (int h = kWarps / 2; h; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) v[i] += v[i + h];
      st_async1(s_lg + r0 + r, v[0] + bias[r], bar_lg, peer);
    }
  }
}

__device__ __forceinline__ unsigned order_key(float v) {
  v = (v == v) ? v : -INFINITY;                 // NaN counts as -inf
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Softmax (or sigmoid) top-k of the E <= kMaxE logits, ties to the lower index, exact.
// Warp 0 alone: lane l holds the keys of logits l + 32 i; each of K rounds takes the
// largest key by one warp max-reduction, the lowest index holding it by one
// min-reduction, and retires it.  Weights: the selected scores over their sum.  Every
// thread calls this (one barrier at the end).
__device__ __forceinline__ void best_of_lane(const unsigned (&key)[kMaxE / 32], unsigned& b, int& bi) {
  unsigned k2[kMaxE / 64];
  int i2[kMaxE / 64];
#pragma unroll
  for (int i = 0; i < kMaxE / 64; ++i) {           // pairs, then a tree: ties keep the lower i
    const bool hi = key[2 * i + 1] > key[2 * i];
    k2[i] = hi ? key[2 * i + 1] : key[2 * i];
    i2[i] = hi ? 2 * i + 1 : 2 * i;
  }
#pragma unroll
  for (int w = kMaxE / 128; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const bool hi = k2[i + w] > k2[i];
      k2[i] = hi ? k2[i + w] : k2[i];
      i2[i] = hi ? i2[i + w] : i2[i];
    }
  b = k2[0];
  bi = i2[0];
}
__device__ __noinline__ void topk(const float* s_lg, int E, int K, int score, int* s_sel, float* s_w) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned key[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? order_key(s_lg[e]) : 0u;  // every live key is >= 1
    }
    unsigned mine = 0u;                           // lane r < K: round r's key and index
    int mine_e = 0;
#pragma unroll 1
    for (int r = 0; r < K; ++r) {
      unsigned b;
      int bi;
      best_of_lane(key, b, bi);
      const unsigned wk = __reduce_max_sync(0xffffffffu, b);
      const int wi = (int)__reduce_min_sync(0xffffffffu, b == wk ? (unsigned)(lane + 32 * bi) : 0xFFFFFFFFu);
      if (lane == r) { mine = wk; mine_e = wi; }
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i)
        if (lane + 32 * i == wi) key[i] = 0u;
    }
    const float l = lane < K ? key_value(mine) : 0.f;
    const float l0 = __shfl_sync(0xffffffffu, l, 0);
    const float p = lane >= K ? 0.f : score == FLINT_ROUTER_SIGMOID ? 1.0f / (1.0f + expf(-l)) : expf(l - l0);
    float z = p;
#pragma unroll
    for (int o = FLINT_MAX_TOP_K / 2; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < K) {
      s_sel[lane] = mine_e;
      s_w[lane] = __fdividef(p, z);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- groups
// Group g of cluster c in layer D: routed (rank >= 0: the expert of that rank, one part
// of F outputs) or parts [p0, p0 + np) of the shared expert (parts of Wsh outputs).
struct GroupDims {
  int rank, n, Wp, np, W, contiguous;
};
__device__ __forceinline__ GroupDims group_dims(const DecLayer& D, int c, int g) {
  GroupDims d;
  d.rank = D.rank[c][g];
  d.Wp = d.rank >= 0 ? D.F : D.Wsh;
  d.np = d.rank >= 0 ? 1 : D.np[c][g];
  d.W = d.Wp * d.np;
  d.n = d.Wp / kCS;
  d.contiguous = d.rank >= 0 || d.W == D.Fs;
  return d;
}
// Group buffer: two slots.  Part p's gate/up rows go to slot p % 2: codes [2n][H/2] (gate
// rows, then up rows) and scales [2n][H/16].  The down rows (codes [R16][W/2], scales
// [R16][W/16]) go to slot 1 for a one-part group, and for a longer group to the slot of
// part np - 2 once that part has been used; each slot holds whichever it receives.
struct GroupOff {
  uint32_t slot0, bytes;
  __host__ __device__ static GroupOff of(int n, int W, int np, int H) {
    GroupOff o;
    const uint32_t part = a16(2 * n * H / 2) + a16(2 * n * H / 16);
    const uint32_t down = a16(H / 16 * W / 2) + a16(H / 16 * W / 16);
    const uint32_t s0 = np >= 2 ? (part > down ? part : down) : part;
    o.slot0 = s0;
    o.bytes = s0 + (np >= 2 ? s0 : down);
    return o;
  }
  __host__ __device__ uint32_t slot(int k) const { return k ? slot0 : 0u; }
  __host__ __device__ uint32_t down_slot(int np) const { return slot(np >= 2 ? (np - 2) % 2 : 1); }
};

// A group's contiguous copies, one per warp (lane 0 of warp w0 + k makes copy k: the
// lanes of one warp issue bulk copies one after another, different warps side by side):
//   what >= 0: part `what` -- this CTA's n gate rows and n up rows (codes, then scales)
//              into `dst`; part 0 also brings the group's three tensor scales into tsc;
//   what <  0: the group's down rows R_j (all its W columns: the group spans whole rows).
// Copy 0's thread posts the byte count on `bar` (its one arrival); the copies land on it.
// A copy is described before the expert is known: source base + e * stride (e the routed
// expert, 0 for a shared group), `bytes` (0: none) to dst, a bulk copy (kind 0) or a
// 4-byte cp.async that holds bar's phase open until it lands (kind 1).
struct CopyDesc {
  const uint8_t* base;
  unsigned long long stride;
  uint32_t dst, bar, bytes, kind;
};
constexpr int kCopyWarps = 7;                 // copies of one call: warps w0 .. w0 + 6
constexpr int kDownW0 = 8;                    // first warp of the down-row copies
static_assert(kDownW0 >= kCopyWarps && kDownW0 + kCopyWarps <= kWarps, "copy warps");

// Copy k (0 <= k < kCopyWarps) of a group; *expect: the byte count copy 0 posts.
__device__ __forceinline__ CopyDesc copy_desc(const DecLayer& D, int c, int g, int what, int k, int j, int H,
                                              uint8_t* dst, float* tsc, uint64_t* bar, uint32_t* expect) {
  CopyDesc cd;
  cd.base = nullptr;
  cd.stride = 0;
  cd.dst = smem_addr(dst);
  cd.bar = smem_addr(bar);
  cd.bytes = 0;
  cd.kind = 0;
  const GroupDims d = group_dims(D, c, g);
  const bool routed = d.rank >= 0;
  if (what >= 0) {
    const size_t row0 = routed ? (size_t)d.n * j : (size_t)(D.p0[c][g] + what) * D.Wsh + (size_t)d.n * j;
    const size_t rows_e = routed ? (size_t)D.F : 0;          // rows per expert
    const NVPtr& P = (k & 1) ? (routed ? D.up : D.sh_up) : (routed ? D.gate : D.sh_gate);
    const uint32_t cb = d.n * H / 2, sb = d.n * H / 16;
    *expect = 2 * (cb + sb);
    if (k < 2) {                                  // codes: gate, up
      cd.base = P.codes + row0 * (H / 2);
      cd.stride = rows_e * (H / 2);
      cd.dst += k * cb;
      cd.bytes = cb;
    } else if (k < 4) {                           // scales: gate, up
      cd.base = P.scales + row0 * (H / 16);
      cd.stride = rows_e * (H / 16);
      cd.dst += a16(2 * cb) + (k - 2) * sb;
      cd.bytes = sb;
    } else if (what == 0 && k < 7) {              // tensor scales of gate, up, down
      const NVPtr& T = k == 4 ? (routed ? D.gate : D.sh_gate) : k == 5 ? (routed ? D.up : D.sh_up)
                                                                       : (routed ? D.down : D.sh_down);
      cd.base = reinterpret_cast<const uint8_t*>(T.tsc);
      cd.stride = routed ? 4 : 0;
      cd.dst = smem_addr(tsc + (k - 4));
      cd.bytes = 4;
      cd.kind = 1;
    }
  } else {
    const int R16 = H / 16;
    const size_t drow0 = (size_t)R16 * j;
    const size_t rows_e = routed ? (size_t)H : 0;
    const NVPtr& Dn = routed ? D.down : D.sh_down;
    const uint32_t dcb = R16 * d.W / 2, dsb = R16 * d.W / 16;
    *expect = dcb + dsb;
    if (k == 0) {
      cd.base = Dn.codes + drow0 * (d.W / 2);
      cd.stride = rows_e * (d.W / 2);
      cd.bytes = dcb;
    } else if (k == 1) {
      cd.base = Dn.scales + drow0 * (d.W / 16);
      cd.stride = rows_e * (d.W / 16);
      cd.dst += a16(dcb);
      cd.bytes = dsb;
    }
  }
  return cd;
}
__device__ __forceinline__ void copy_go(const CopyDesc& cd, int e) {
  if (!cd.bytes) return;
  const uint8_t* src = cd.base + (size_t)e * cd.stride;
  if (cd.kind == 0) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(cd.dst), "l"(src), "r"(cd.bytes), "r"(cd.bar) : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(cd.dst), "l"(src) : "memory");
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(cd.bar) : "memory");
  }
}
// The copies of a group issued now (e: the routed expert); every thread calls this.
__device__ __noinline__ void issue_copies(const DecLayer& D, int c, int g, int what, int e, int j, int H,
                                          uint8_t* dst, float* tsc, uint64_t* bar, int w0) {
  const int k = (threadIdx.x & 31) == 0 ? (int)(threadIdx.x >> 5) - w0 : -1;   // this thread's copy
  if (k < 0 || k >= kCopyWarps) return;
  uint32_t expect = 0;
  const CopyDesc cd = copy_desc(D, c, g, what, k, j, H, dst, tsc, bar, &expect);
  if (k == 0) mbar_expect_tx(bar, expect);
  copy_go(cd, e);
}
// ... described now, issued later by prepared_go (a shared group: e = 0); copy 0 posts
// the byte count at once.  Every thread calls this.
__device__ __noinline__ void prepare_copies(const DecLayer& D, int c, int g, int what, int j, int H, uint8_t* dst,
                                            float* tsc, uint64_t* bar, int w0, CopyDesc* s_cp) {
  const int k = (threadIdx.x & 31) == 0 ? (int)(threadIdx.x >> 5) - w0 : -1;
  if (k < 0 || k >= kCopyWarps) return;
  uint32_t expect = 0;
  s_cp[threadIdx.x >> 5] = copy_desc(D, c, g, what, k, j, H, dst, tsc, bar, &expect);
  if (k == 0) mbar_expect_tx(bar, expect);
}
// A routed group's first copies described before its expert is known, for expert 0
// (prepared_go adds e * stride): part 0 (copies 0..6, warps 0..6) into buf, the down rows
// (copies 0..1, warps kDownW0..) into slot 1.  The routed buffer sits at the start of the
// big region and holds one part, so none of this depends on which group it is.  Copy 0
// of each posts its byte count at once (the phase then waits for the copies).  Every
// thread calls this.
__device__ __noinline__ void prepare_routed_copies(const DecLayer& D, int j, int H, uint8_t* buf, float* tsc,
                                                   uint64_t* bar_gu, uint64_t* bar_dn, CopyDesc* s_cp) {
  if (threadIdx.x & 31) return;
  const int w = threadIdx.x >> 5;
  const bool part = w < kCopyWarps, down = w >= kDownW0 && w < kDownW0 + kCopyWarps;
  if (!part && !down) return;
  const int F = D.F, n = F / kCS, R16 = H / 16;
  const uint32_t cb = n * H / 2, sb = n * H / 16;
  CopyDesc cd;
  cd.base = nullptr;
  cd.stride = 0;
  cd.bytes = 0;
  cd.kind = 0;
  if (part) {
    const int k = w;
    cd.bar = smem_addr(bar_gu);
    cd.dst = smem_addr(buf);
    if (k < 4) {                                  // codes gate, up; scales gate, up
      const NVPtr& P = (k & 1) ? D.up : D.gate;
      const bool sc = k >= 2;
      const uint32_t row = sc ? H / 16 : H / 2;
      cd.base = (sc ? P.scales : P.codes) + (size_t)n * j * row;
      cd.stride = (unsigned long long)F * row;
      cd.dst += sc ? a16(2 * cb) + (k - 2) * sb : k * cb;
      cd.bytes = sc ? sb : cb;
    } else {                                      // tensor scales of gate, up, down
      const NVPtr& T = k == 4 ? D.gate : k == 5 ? D.up : D.down;
      cd.base = reinterpret_cast<const uint8_t*>(T.tsc);
      cd.stride = 4;
      cd.dst = smem_addr(tsc + (k - 4));
      cd.bytes = 4;
      cd.kind = 1;
    }
    if (k == 0) mbar_expect_tx(bar_gu, 2 * (cb + sb));
  } else {
    const int k = w - kDownW0;
    const uint32_t dcb = R16 * F / 2, dsb = R16 * F / 16;
    cd.bar = smem_addr(bar_dn);
    cd.dst = smem_addr(buf) + a16(2 * cb) + a16(2 * sb);   // slot 1 of a one-part group
    if (k < 2) {                                  // codes, scales
      const uint32_t row = k ? F / 16 : F / 2;
      cd.base = (k ? D.down.scales : D.down.codes) + (size_t)R16 * j * row;
      cd.stride = (unsigned long long)H * row;
      cd.dst += k ? a16(dcb) : 0u;
      cd.bytes = k ? dsb : dcb;
    }
    if (k == 0) mbar_expect_tx(bar_dn, dcb + dsb);
  }
  s_cp[w] = cd;
}
__device__ __forceinline__ void prepared_go(const CopyDesc* s_cp, int e, int w0) {
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0 && w >= w0 && w < w0 + kCopyWarps) copy_go(s_cp[w], e);
}

// ... strided down rows (a shared group spanning part of the columns): cp.async from every
// thread, completing on bar (one arrival per thread).
__device__ __noinline__ void issue_down_strided(const DecLayer& D, int c, int g, int j, int H, uint8_t* dst,
                                                uint64_t* bar) {
  const GroupDims d = group_dims(D, c, g);
  const int R16 = H / 16;
  const int o0 = D.p0[c][g] * D.Wsh;
  const uint8_t* dc = D.sh_down.codes + (size_t)R16 * j * (D.Fs / 2) + o0 / 2;
  const uint8_t* ds = D.sh_down.scales + (size_t)R16 * j * (D.Fs / 16) + o0 / 16;
  const uint32_t dcb = R16 * d.W / 2;
  const int cpr = d.W / 32;                    // 16-byte code chunks per row
#pragma unroll 1
  for (int i = threadIdx.x; i < R16 * cpr; i += kThreads) {
    const int r = i / cpr, k = i - r * cpr;
    cp_async16(dst + r * (d.W / 2) + 16 * k, dc + (size_t)r * (D.Fs / 2) + 16 * k);
  }
  const int spr = d.W / 64;                    // 4-byte scale chunks per row
#pragma unroll 1
  for (int i = threadIdx.x; i < R16 * spr; i += kThreads) {
    const int r = i / spr, k = i - r * spr;
    cp_async4(dst + a16(dcb) + r * (d.W / 16) + 4 * k, ds + (size_t)r * (D.Fs / 16) + 4 * k);
  }
  cp_async_arrive_noinc(bar);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// D (16 x 8, fp32) += A (16 x 16, f16, row) . B (16 x 8, f16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Down columns of a group: this CTA's R16 rows (codes [R16][W/2], scales [R16][W/16] in
// shared memory) times the group's W SwiGLU values hsw (whose producers' maxima are in
// hmax), added (times `scale`) into s_part.  Every thread calls this.
//
// hsw is split into two f16 terms under one power-of-two scale 2^k (max |hsw| 2^k in
// [2^14, 2^15)): hi = f16(v 2^k), lo = f16(v 2^k - hi), about 22 bits of every value.
// They are columns 0 and 1 of the B operand of mma.sync m16n8k16 (f16 x f16 products are
// exact, accumulation fp32); the weights are decoded to f16 (cvt.rn.f16x2.e2m1x2) and
// multiplied by their E4M3 block scale (exact in f16: |e2m1 x e4m3| lies in [2^-10,
// 2688]).  A warp takes 16 rows and a range of 128-column chunk sets; lane (g, t) of the
// mma fragments holds rows g and g + 8 and reads 32-column chunk 4 c + t of each, so the
// order of the columns within an mma is a fixed permutation that the B operand (read by
// the same lane from the same chunk) follows.
__device__ __noinline__ void group_down(const uint8_t* dcodes, const uint8_t* dscales, int W, int R16,
                                        const float* hsw, const float* hmax, int nmax, uint32_t* s_hh,
                                        uint32_t* s_hl, float* s_acc, float scale, float* s_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // 1. one scale for the group: the max of the producers' maxima (hmax[i], i < nmax:
  // every part's CTAs sent theirs with their values; non-negative floats order as
  // their bit patterns)
  float am = 0.f;
#pragma unroll 1
  for (int i = lane; i < nmax; i += 32) am = fmaxf(am, hmax[i]);
  am = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(am)));
  const int k = f16_stage_exponent(am);
  const float s2k = exp2i(k);
  // 2. the hi / lo terms, f16 pairs in column order
#pragma unroll 1
  for (int i = threadIdx.x; i < W / 2; i += kThreads) {
    const float2 v = *reinterpret_cast<const float2*>(hsw + 2 * i);
    const float a = v.x * s2k, b = v.y * s2k;
    const uint32_t hi = pack_f16x2_rn(a, b);
    float ha, hb;
    f16x2_to_f32x2(hi, ha, hb);
    s_hh[i] = hi;
    s_hl[i] = pack_f16x2_rn(a - ha, b - hb);
  }
  __syncthreads();
  // 3. 16-row tiles x chunk-set ranges over the warps
  const int g = lane >> 2, t = lane & 3;
  const int tiles = R16 / 16, csets = (W + 127) / 128, qmax = W / 32;
  int ksegs = kWarps / tiles;
  ksegs = ksegs < 1 ? 1 : (ksegs > csets ? csets : ksegs);
  const int per = (csets + ksegs - 1) / ksegs;
  const uint32_t* bsrc = g == 1 ? s_hl : s_hh;         // B column 1 (lanes 4-7) = lo, column 0 = hi
#pragma unroll 1
  for (int item = warp; item < tiles * ksegs; item += kWarps) {
    const int tile = item % tiles, ks = item / tiles;
    const uint8_t* ra = dcodes + (size_t)(16 * tile + g) * (W / 2);
    const uint8_t* rb = ra + (size_t)8 * (W / 2);
    const uint8_t* sa = dscales + (size_t)(16 * tile + g) * (W / 16);
    const uint8_t* sb = sa + (size_t)8 * (W / 16);
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int c1 = min(csets, (ks + 1) * per);
#pragma unroll 1
    for (int c = ks * per; c < c1; ++c) {
      const int q = 4 * c + t;
      uint4 wa = make_uint4(0u, 0u, 0u, 0u), wb = wa, x0 = wa, x1 = wa, x2 = wa, x3 = wa;
      uint32_t fa = 0u, fb = 0u;
      if (q < qmax) {
        wa = *reinterpret_cast<const uint4*>(ra + 16 * q);
        wb = *reinterpret_cast<const uint4*>(rb + 16 * q);
        fa = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sa + 2 * q));
        fb = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sb + 2 * q));
        const uint4* xp = reinterpret_cast<const uint4*>(bsrc + 16 * q);
        x0 = xp[0]; x1 = xp[1]; x2 = xp[2]; x3 = xp[3];
      }
      const uint32_t SA[2] = {__byte_perm(fa, 0, 0x1010), __byte_perm(fa, 0, 0x3232)};
      const uint32_t SB[2] = {__byte_perm(fb, 0, 0x1010), __byte_perm(fb, 0, 0x3232)};
      const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                               x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
      const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w}, wbv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {                    // word h of the chunk: mmas 2h, 2h + 1
        uint32_t a[4], b[4];
        e2m1x8_to_f16x2x4(wav[h], a[0], a[1], a[2], a[3]);
        e2m1x8_to_f16x2x4(wbv[h], b[0], b[1], b[2], b[3]);
        const uint32_t S_a = SA[h >> 1], S_b = SB[h >> 1];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int j = 2 * h + m;
          mma16816(d[m], hmul2(a[2 * m], S_a), hmul2(b[2 * m], S_b), hmul2(a[2 * m + 1], S_a),
                   hmul2(b[2 * m + 1], S_b), xv[2 * j], xv[2 * j + 1]);
        }
      }
    }
    if (t == 0) {
      s_acc[ks * R16 + 16 * tile + g] = (d[0][0] + d[0][1]) + (d[1][0] + d[1][1]);
      s_acc[ks * R16 + 16 * tile + g + 8] = (d[0][2] + d[0][3]) + (d[1][2] + d[1][3]);
    }
  }
  __syncthreads();
  const float unscale = exp2i(-k) * scale;
#pragma unroll 1
  for (int r = threadIdx.x; r < R16; r += kThreads) {
    float v = 0.f;
#pragma unroll 1
    for (int ks = 0; ks < ksegs; ++ks) v += s_acc[ks * R16 + r];
    s_part[r] += v * unscale;
  }
}

// ---------------------------------------------------------------- residual exchange
// post_rows posts this CTA's partial rows.  exchange waits (bounded) until every word it
// reads carries `tag`: word i = c' * H/16 + r is row r of R_j from cluster c'; two per
// thread, both in flight at once.  Then h_{l+1}[R_j] = h_l[R_j] + the
// clusters' partials summed pairwise in a fixed order, into s_hn, which goes to every
// CTA of the cluster (h_nxt, completing on each one's bar_nxt) and, when `out` is given,
// to out.  Thread 0 also refreshes *s_abort (its load completes during the poll).  Every
// thread calls this.
__device__ __forceinline__ void post_rows(unsigned long long* bd, int c, int H, int j, unsigned tag,
                                          const float* s_part) {
  const int R16 = H / 16;
#pragma unroll 1
  for (int r = threadIdx.x; r < R16; r += kThreads)
    st_tagged(bd + (size_t)c * H + (size_t)R16 * j + r, ((unsigned long long)tag << 32) | __float_as_uint(s_part[r]));
}
__device__ __noinline__ void exchange(const unsigned long long* bd, int NC, int H, int j, unsigned tag,
                                      float* s_pp, const float* h_cur, float* s_hn, float* h_nxt, uint64_t* bar_nxt,
                                      float* out, unsigned* sync, unsigned long long limit, int* s_abort) {
  const int R16 = H / 16;
  const unsigned ab = threadIdx.x == 0 ? ld_abort(sync) : 0u;
  const int N = NC * R16;
  const int i0 = threadIdx.x, i1 = threadIdx.x + kThreads;
  bool n0 = i0 < N, n1 = i1 < N;
  const unsigned long long* p0 = bd + (size_t)(n0 ? i0 / R16 : 0) * H + (size_t)R16 * j + (n0 ? i0 % R16 : 0);
  const unsigned long long* p1 = bd + (size_t)(n1 ? i1 / R16 : 0) * H + (size_t)R16 * j + (n1 ? i1 % R16 : 0);
  unsigned long long w0 = n0 ? ld_relaxed(p0) : 0ull, w1 = n1 ? ld_relaxed(p1) : 0ull;
  unsigned long long t0 = 0;
#pragma unroll 1
  for (unsigned polls = 1;; ++polls) {
    if (n0 && (unsigned)(w0 >> 32) == tag) { s_pp[i0] = __uint_as_float((unsigned)w0); n0 = false; }
    if (n1 && (unsigned)(w1 >> 32) == tag) { s_pp[i1] = __uint_as_float((unsigned)w1); n1 = false; }
    if (!n0 && !n1) break;
    if ((polls & 15u) == 0) {
      if (ld_abort(sync)) break;
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit) {
        give_up(sync);
        break;
      }
    }
    if (n0) w0 = ld_relaxed(p0);
    if (n1) w1 = ld_relaxed(p1);
  }
  if (threadIdx.x == 0) *s_abort = (int)ab;
  __syncthreads();
#pragma unroll 1
  for (int r = threadIdx.x; r < R16; r += kThreads) {
    float v[kDecMaxClusters];
#pragma unroll
    for (int k = 0; k < kDecMaxClusters; ++k) v[k] = k < NC ? s_pp[k * R16 + r] : 0.f;
#pragma unroll
    for (int w = kDecMaxClusters / 2; w; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) v[i] += v[i + w];
    const float h = h_cur[R16 * j + r] + v[0];
    s_hn[r] = h;
    if (out) out[R16 * j + r] = h;
  }
  __syncthreads();
  to_cluster_async(h_nxt + R16 * j, s_hn, R16 / 4, bar_nxt);
}

// ---------------------------------------------------------------- head
__device__ __forceinline__ void best_reduce_warp(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

// The last CTA reduces the CTAs' tagged maxima of token t (warp 0; bounded waits).
__device__ __noinline__ void head_argmax(const unsigned long long* best, int G, unsigned ttag, int V, int32_t* out,
                                         unsigned* sync, unsigned long long lim) {
  const int lane = threadIdx.x & 31;
  float v = -INFINITY;
  int i = 0x7FFFFFFF;
#pragma unroll 1
  for (int k = lane; k < G; k += 32) {
    unsigned long long wv = ld_relaxed(best + 2 * k), wi = ld_relaxed(best + 2 * k + 1);
    unsigned long long t0 = 0;
    for (unsigned polls = 1; (unsigned)(wv >> 32) != ttag || (unsigned)(wi >> 32) != ttag; ++polls) {
      if ((polls & 15u) == 0) {
        if (ld_abort(sync)) break;
        const unsigned long long now = globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > lim) {
          give_up(sync);
          break;
        }
      }
      wv = ld_relaxed(best + 2 * k);
      wi = ld_relaxed(best + 2 * k + 1);
    }
    const float kv = __uint_as_float((unsigned)wv);
    const int ki = (int)(unsigned)wi;
    if (kv > v || (kv == v && ki < i)) { v = kv; i = ki; }
  }
  best_reduce_warp(v, i);
  if (lane == 0 && out) *out = (i >= 0 && i < V) ? i : 0;
}

// ---------------------------------------------------------------- fused sampling
// ("Recursive Releases Flint, a 40B MoE Coding Model That Runs Locally at 125 Tokens per
// Second", section "How does Flint perform on coding benchmarks?": temperature 1.0,
// top-p 0.95, top-k 20.)  The K largest logits of the token are found in two levels --
// each CTA its own rows, then the last CTA over the CTAs' lists -- and the draw follows
// flint_sample_logits exactly.

// Candidates are (order key, index) pairs ranked by key, ties to the lower index; key 0
// is empty (index 0x7FFFFFFF).  prec(a, b): a ranks before b.
__device__ __forceinline__ bool prec(unsigned ka, int ia, unsigned kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}
__device__ __forceinline__ void cas(unsigned (&k)[8], int (&x)[8], int i, int j) {
  const bool sw = prec(k[j], x[j], k[i], x[i]);
  const unsigned ki = k[i], kj = k[j];
  const int xi = x[i], xj = x[j];
  k[i] = sw ? kj : ki; k[j] = sw ? ki : kj;
  x[i] = sw ? xj : xi; x[j] = sw ? xi : xj;
}
// This lane's eight candidates in rank order (Batcher's odd-even merge network).
__device__ __forceinline__ void lane_sort8(unsigned (&k)[8], int (&x)[8]) {
  cas(k, x, 0, 1); cas(k, x, 2, 3); cas(k, x, 4, 5); cas(k, x, 6, 7);
  cas(k, x, 0, 2); cas(k, x, 1, 3); cas(k, x, 4, 6); cas(k, x, 5, 7);
  cas(k, x, 1, 2); cas(k, x, 5, 6);
  cas(k, x, 0, 4); cas(k, x, 1, 5); cas(k, x, 2, 6); cas(k, x, 3, 7);
  cas(k, x, 2, 4); cas(k, x, 3, 5);
  cas(k, x, 1, 2); cas(k, x, 3, 4); cas(k, x, 5, 6);
}
// The K best of the warp's candidates (eight per lane, each lane's in rank order), in
// rank order into out_key / out_idx: each round takes the best lane head by two warp
// reductions (largest key, then lowest index holding it) and that lane moves on.
__device__ __forceinline__ void warp_topk8(unsigned (&k)[8], int (&x)[8], int K, unsigned* out_key, int* out_idx) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int s = 0; s < K; ++s) {
    const unsigned wk = __reduce_max_sync(0xffffffffu, k[0]);
    const int wi = (int)__reduce_min_sync(0xffffffffu, k[0] == wk ? (unsigned)x[0] : 0xFFFFFFFFu);
    if (lane == 0) { out_key[s] = wk; out_idx[s] = wi; }
    if (k[0] == wk && x[0] == wi) {
#pragma unroll
      for (int q = 0; q < 7; ++q) { k[q] = k[q + 1]; x[q] = x[q + 1]; }
      k[7] = 0u;
      x[7] = 0x7FFFFFFF;
    }
  }
}
// The K best of M <= 128 lists in rank order (list m: keys[m * ld + r], r < len), in
// rank order into out_key / out_idx; one warp (lane l holds lists l, l + 32, ...).
__device__ __noinline__ void merge_lists(const unsigned* keys, const int* idx, int M, int ld, int len, int K,
                                         unsigned* out_key, int* out_idx) {
  const int lane = threadIdx.x & 31;
  unsigned hk[4];
  int hx[4], hp[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int m = lane + 32 * q;
    hp[q] = 0;
    hk[q] = m < M && len > 0 ? keys[m * ld] : 0u;
    hx[q] = m < M && len > 0 ? (hk[q] ? idx[m * ld] : 0x7FFFFFFF) : 0x7FFFFFFF;
  }
#pragma unroll 1
  for (int s = 0; s < K; ++s) {
    unsigned bk = hk[0];
    int bx = hx[0], bq = 0;
#pragma unroll
    for (int q = 1; q < 4; ++q)
      if (prec(hk[q], hx[q], bk, bx)) { bk = hk[q]; bx = hx[q]; bq = q; }
    const unsigned wk = __reduce_max_sync(0xffffffffu, bk);
    const int wi = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (unsigned)bx : 0xFFFFFFFFu);
    if (lane == 0) { out_key[s] = wk; out_idx[s] = wi; }
    if (bk == wk && bx == wi && (wk != 0u || wi != 0x7FFFFFFF)) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == bq) {
          const int m = lane + 32 * q, r = ++hp[q];
          hk[q] = r < len ? keys[m * ld + r] : 0u;
          hx[q] = r < len && hk[q] ? idx[m * ld + r] : 0x7FFFFFFF;
        }
    }
  }
}

// The K (<= 32) largest of n <= kThreads * 8 candidates (order keys s_key, 0 = empty;
// indices s_idx, or base + i when s_idx is null), ties to the lower index, in rank
// order into out_key / out_idx.  Each warp ranks its slice (<= 256, eight per lane),
// then warp 0 merges the warps' K-lists.  Every thread calls this.
__device__ __noinline__ void block_topk(const unsigned* s_key, const int* s_idx, int n, int K, int base,
                                        unsigned* s_wk, int* s_wi, unsigned* out_key, int* out_idx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (n + kWarps - 1) / kWarps;
  const int b0 = warp * per, b1 = min(n, b0 + per);
  {
    unsigned key[8];
    int idx[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = b0 + lane + 32 * q;
      key[q] = i < b1 ? s_key[i] : 0u;
      idx[q] = i < b1 && key[q] ? (s_idx ? s_idx[i] : base + i) : 0x7FFFFFFF;
    }
    lane_sort8(key, idx);
    warp_topk8(key, idx, K, s_wk + warp * K, s_wi + warp * K);
  }
  __syncthreads();
  if (warp == 0) merge_lists(s_wk, s_wi, kWarps, K, K, K, out_key, out_idx);
  __syncthreads();
}

// The last CTA: every CTA's K candidates of token t (tagged words {tag, key},
// {tag, index}, waited for with a bound), their K best, and the draw with the caller's
// uniform u: p_i = exp((l_i - l_0) / temp) over the K, the shortest prefix whose p sum
// reaches top_p, the first i of it with u < (p_0 + ... + p_i) / (sum of the prefix).
// +inf / all -inf: rank 0.  Writes the token and the argmax (rank 0).  Every thread of
// the CTA calls this.
__device__ __noinline__ void head_sample(const unsigned long long* cand, int G, int K, unsigned tag, float temp,
                                         float top_p, float u, int V, int32_t* token, int32_t* amax,
                                         unsigned* s_ck, int* s_ci, unsigned* s_wk, int* s_wi, unsigned* s_fk,
                                         int* s_fi, unsigned* sync, unsigned long long lim) {
  const int n = G * K;
#pragma unroll 1
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const unsigned long long* w = cand + 2 * ((size_t)(i / K) * 32 + i % K);
    unsigned long long wk = ld_relaxed(w), wi = ld_relaxed(w + 1);
    unsigned long long t0 = 0;
    for (unsigned polls = 1; (unsigned)(wk >> 32) != tag || (unsigned)(wi >> 32) != tag; ++polls) {
      if ((polls & 15u) == 0) {
        if (ld_abort(sync)) break;
        const unsigned long long now = globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > lim) {
          give_up(sync);
          break;
        }
      }
      wk = ld_relaxed(w);
      wi = ld_relaxed(w + 1);
    }
    s_ck[i] = (unsigned)wk;
    s_ci[i] = (int)(unsigned)wi;
  }
  __syncthreads();
  // each CTA's K candidates are in rank order: one warp merges the G lists
  if (threadIdx.x < 32) merge_lists(s_ck, s_ci, G, K, K, K, s_fk, s_fi);
  __syncwarp();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int idx = lane < K ? s_fi[lane] : 0;
  const float l = lane < K ? key_value(s_fk[lane]) : -INFINITY;
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  int pick_lane = 0;
  if (l0 != -INFINITY && l0 != INFINITY) {
    float p = lane < K ? expf((l - l0) / temp) : 0.f;
    float z = p;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    p /= z;
    float c = p;                                       // inclusive prefix sums in rank order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float x = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) c += x;
    }
    const unsigned reach = __ballot_sync(0xffffffffu, lane < K && c >= top_p);
    const int m = reach ? __ffs(reach) : K;
    const float zm = __shfl_sync(0xffffffffu, c, m - 1);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < m && u < c / zm);
    pick_lane = hit ? __ffs(hit) - 1 : m - 1;
  }
  const int pick = __shfl_sync(0xffffffffu, idx, pick_lane);
  if (lane == 0) {
    *token = (pick >= 0 && pick < V) ? pick : 0;
    if (amax) *amax = (idx >= 0 && idx < V) ? idx : 0;
  }
}

// ---------------------------------------------------------------- the kernel
constexpr int kLayerWords = (int)(sizeof(DecLayer) / 8);
static_assert(sizeof(DecLayer) % 8 == 0 && kLayerWords <= 32, "layer table: at most 32 words");

// Shared-memory carve (bytes), the same on the host and the device.
struct Smem {
  uint32_t h, xb, xl, lg, hsw, hmax, tmp, part, pp, gu, hn, hv, hh, hl, acc, big, total;
  __host__ __device__ static Smem of(int H, int Emax) {
    Smem s;
    const int R16 = H / 16;
    s.h = 0;                                   // [2][H] fp32 residual h (by step parity)
    s.xb = s.h + 8 * H;                        // [H] bf16 x
    s.xl = s.xb + 2 * H;                       // [H/8] uint4 x operand, lane-major
    s.lg = s.xl + 2 * H;                       // [2][Emax] fp32 logits (by step parity)
    s.hsw = s.lg + a16(8 * Emax);              // [2][kMaxW] fp32 SwiGLU values (by group parity)
    s.hmax = s.hsw + 8 * kMaxW;                // [2][kMaxParts][kCS] fp32 the producers' max |value|
    s.tmp = s.hmax + 2 * 4 * kCS * kMaxParts;  // [kMaxN] fp32 this CTA's SwiGLU values / logits
    s.part = s.tmp + 4 * kMaxN;                // [H/16] fp32 partial sums of this CTA's rows
    s.pp = s.part + 4 * R16;                   // [kDecMaxClusters][H/16] polled partials
    s.gu = s.pp + 4 * kDecMaxClusters * R16;   // [2 kMaxN] gate/up values
    s.hn = s.gu + 8 * kMaxN;                   // [H/16] fp32 h_{l+1} rows of this CTA
    s.hv = s.hn + 4 * R16;                     // [256] fp32 head chunk values
    s.hh = s.hv + 4 * 256;                     // [kMaxW/2] f16 pairs: hi terms of the SwiGLU values
    s.hl = s.hh + 2 * kMaxW;                   // [kMaxW/2] f16 pairs: lo terms
    s.acc = s.hl + 2 * kMaxW;                  // [256] fp32 down partials (chunk-set range x row)
    s.big = (s.acc + 4 * 256 + 127) & ~127u;   // router rows + group buffer, or the head ring
    s.total = s.big + kBigBytes;
    return s;
  }
};

// Head rows per ring slot at hidden H: a multiple of 64, at most 256, two slots in the
// big region.
__host__ __device__ __forceinline__ int head_chunk_rows(int H) {
  int r = ((kBigBytes - 8192) / 2) / (H / 2 + H / 16);    // the last 8 KB: sampled logits
  r = r > 256 ? 256 : r;
  return r & ~63;
}

// The head for one token: this CTA's rows [v0, v1) stream through a two-slot ring of TMA
// bulk copies in s_big and are dotted with x (s_xl).  Writes the logits (optional; also
// into s_lv[v - v0] when s_lv is given) and leaves this thread's running best in
// (bv, bi).  Every thread calls this.
template <int CPL>
__device__ __noinline__ void head_phase(const DecodeArgs& a, int t, int v0, int v1, const uint4* s_xl,
                                        float unscale, uint8_t* s_big, float* s_hv, float* s_lv, uint64_t* bar_hd,
                                        uint32_t& ph_hd, unsigned& pend_hd, bool abort, float& bv, int& bi) {
  const int H = a.H;
  const int HR = head_chunk_rows(H);
  const uint32_t cbytes = (uint32_t)HR * (H / 2);
  const uint32_t slot_bytes = a16(cbytes + (uint32_t)HR * (H / 16));
  const int nch = (v1 - v0 + HR - 1) / HR;
  const float tsc = __ldg(a.head.tsc) * unscale;
#pragma unroll 1
  for (int k = -2; k < nch; ++k) {
    // iteration k issues chunk k + 2 (once slot (k + 2) % 2 is free) and consumes chunk k
    if (k >= 0) {
      const int sl = k & 1;
      const int r0 = v0 + k * HR, nr = min(HR, v1 - r0);
      const uint8_t* src = s_big + (size_t)sl * slot_bytes;
      if (pend_hd & (1u << sl)) {
        mbar_wait(&bar_hd[sl], (ph_hd >> sl) & 1u, a.sync, a.wait_ns);
        ph_hd ^= 1u << sl;
        pend_hd &= ~(1u << sl);
      }
      rows_dot<CPL>(src, src + cbytes, nr, nr, tsc, tsc, H, s_xl, s_hv);
      __syncthreads();                               // s_hv; slot sl is free
#pragma unroll 1
      for (int r = threadIdx.x; r < nr; r += kThreads) {
        const float v = s_hv[r];
        if (a.logits) a.logits[(size_t)t * a.V + r0 + r] = v;
        if (s_lv) s_lv[r0 - v0 + r] = v;
        const float vv = (v == v) ? v : -INFINITY;
        if (vv > bv || (vv == bv && r0 + r < bi)) { bv = vv; bi = r0 + r; }
      }
    }
    const int kn = k + 2;
    if (kn < nch && !abort) {
      const int sl = kn & 1;
      if (threadIdx.x == 0) {
        const int r0 = v0 + kn * HR, nr = min(HR, v1 - r0);
        uint8_t* dst = s_big + (size_t)sl * slot_bytes;
        mbar_expect_tx(&bar_hd[sl], (uint32_t)nr * (H / 2 + H / 16));
        bulk_g2s(dst, a.head.codes + (size_t)r0 * (H / 2), (uint32_t)nr * (H / 2), &bar_hd[sl]);
        bulk_g2s(dst + cbytes, a.head.scales + (size_t)r0 * (H / 16), (uint32_t)nr * (H / 16), &bar_hd[sl]);
      }
      pend_hd |= 1u << sl;
    }
    __syncthreads();                                 // s_hv is rewritten by the next chunk
  }
}

template <int CPL>
__global__ void __launch_bounds__(kThreads, 1) k_decode(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t s_dyn[];
  __shared__ __align__(16) DecLayer s_ly[3];         // layer tables of steps s, s + 1, s + 2 (by s % 3)
  __shared__ float s_bias[3][kMaxRR];
  __shared__ int s_sel[FLINT_MAX_TOP_K];
  __shared__ float s_w[FLINT_MAX_TOP_K];
  __shared__ __align__(16) float s_tsc[2][4];        // tensor scales of the shared / routed group in flight
  __shared__ __align__(16) CopyDesc s_cp[kWarps];      // prepared copies, by issuing warp
  __shared__ __align__(16) float s_red[2 * kWarps];
  __shared__ float s_bv[kWarps];
  __shared__ int s_bi[kWarps];
  // copy barriers: router rows, shared parts (two slots), shared down rows (bulk or
  // cp.async), routed part, routed down rows; head ring
  __shared__ __align__(8) uint64_t bars[7], bar_hd[2], bar_h[2];   // bar_h: h_{l+1} landed (by parity)
  // the peers' logits (by step parity) and SwiGLU values (by group parity) landed
  __shared__ __align__(8) uint64_t bar_c[4];
  uint64_t* bar_lg = bar_c;
  __shared__ int s_abort;                            // this CTA saw the abort flag (refreshed per step)

  const int H = a.H, R16 = H / 16;
  const int LPR = H / (32 * CPL);
  const Smem S = Smem::of(H, a.Emax);
  float* s_h = reinterpret_cast<float*>(s_dyn + S.h);
  uint16_t* s_xb = reinterpret_cast<uint16_t*>(s_dyn + S.xb);
  uint4* s_xl = reinterpret_cast<uint4*>(s_dyn + S.xl);
  float* s_lg = reinterpret_cast<float*>(s_dyn + S.lg);
  float* s_hsw = reinterpret_cast<float*>(s_dyn + S.hsw);
  float* s_tmp = reinterpret_cast<float*>(s_dyn + S.tmp);
  float* s_hmax = reinterpret_cast<float*>(s_dyn + S.hmax);
  float* s_part = reinterpret_cast<float*>(s_dyn + S.part);
  float* s_pp = reinterpret_cast<float*>(s_dyn + S.pp);
  float* s_gu = reinterpret_cast<float*>(s_dyn + S.gu);
  float* s_hn = reinterpret_cast<float*>(s_dyn + S.hn);
  float* s_hv = reinterpret_cast<float*>(s_dyn + S.hv);
  uint32_t* s_hh = reinterpret_cast<uint32_t*>(s_dyn + S.hh);
  uint32_t* s_hl = reinterpret_cast<uint32_t*>(s_dyn + S.hl);
  float* s_acc = reinterpret_cast<float*>(s_dyn + S.acc);
  uint8_t* s_big = s_dyn + S.big;
  uint16_t* s_router = reinterpret_cast<uint16_t*>(s_big);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j = (int)cluster_rank();
  const int c = blockIdx.x / kCS;
  const int G = gridDim.x;
  unsigned* sync = a.sync;
  const unsigned long long lim = a.wait_ns;
  const int n_steps = a.T * a.L;
  enum { B_RT, B_GU0, B_GU1, B_DN, B_DNA, B_RGU, B_RDN };
  // per barrier (a bit each): the parity of its current phase, and whether a copy is in
  // flight on it.  A wait happens only for an issued copy, and after an abort no new copy
  // is issued, so the kernel ends with nothing in flight.
  uint32_t ph = 0, pend = 0, ph_hd = 0, pend_hd = 0, ph_h = 0, ph_c = 0;
  unsigned grp_seq = 0;                              // groups run by this cluster
  unsigned pre = 0;                                  // this step's groups already in flight (a bit each)
  auto wait_bar = [&](int i) {
    if (pend & (1u << i)) {
      mbar_wait(&bars[i], (ph >> i) & 1u, sync, lim);
      ph ^= 1u << i;
      pend &= ~(1u << i);
    }
  };

  // the last warp: the layer table of step `st` and this CTA's router bias entries (the
  // parameter's table sits in the constant bank, where each layer's first use would
  // miss).  The loads are issued at a step's start and stored at its end; the staging
  // between them is inlined, so the first call that needs them settled comes late.
  unsigned long long ly_word = 0;
  float ly_bias = 0.f;
  auto load_layer = [&](int st) {
    if (warp != kWarps - 1 || st >= n_steps) return;
    const DecLayer& P = a.layer[st % a.L];
    if (lane < kLayerWords) ly_word = reinterpret_cast<const unsigned long long*>(&P)[lane];
    const int r0 = j * a.RR;
    ly_bias = (lane < a.RR && P.router_bias && r0 + lane < P.E) ? __ldg(P.router_bias + r0 + lane) : 0.f;
  };
  auto store_layer = [&](int st) {
    if (warp != kWarps - 1 || st >= n_steps) return;
    if (lane < kLayerWords) reinterpret_cast<unsigned long long*>(&s_ly[st % 3])[lane] = ly_word;
    if (lane < a.RR) s_bias[st % 3][lane] = ly_bias;
  };
  // (every thread calls these; uniform within the CTA)
  auto issue_router = [&](const DecLayer& D) {
    const int r0 = j * a.RR;
    const int nr = min(a.RR, D.E - r0);
    if (nr <= 0) return;
    pend |= 1u << B_RT;
    if (threadIdx.x != 0) return;
    mbar_expect_tx(&bars[B_RT], (uint32_t)nr * H * 2);
    bulk_g2s(s_router, D.router_w + (size_t)r0 * H, (uint32_t)nr * H * 2, &bars[B_RT]);
  };
  // a group's buffer: routed groups at the start of the big region (over the router
  // rows, which are consumed before a routed group is issued), shared groups after the
  // routed buffer in a routed cluster
  auto group_buf = [&](const DecLayer& D, int g) {
    return s_big + (D.rank[c][g] >= 0 ? 0u : (D.routed[c] ? D.sh_off : 0u));
  };
  // a group's copies: what >= 0 a part (into slot what % 2), what < 0 the down rows
  auto issue = [&](const DecLayer& D, int g, int what) {
    const GroupDims d = group_dims(D, c, g);
    const GroupOff o = GroupOff::of(d.n, d.W, d.np, H);
    const bool routed = d.rank >= 0;
    uint8_t* buf = group_buf(D, g);
    if (what < 0 && !d.contiguous) {
      issue_down_strided(D, c, g, j, H, buf + o.down_slot(d.np), &bars[B_DNA]);
      pend |= 1u << B_DNA;
      return;
    }
    const int b = what >= 0 ? (routed ? B_RGU : B_GU0 + (what & 1)) : (routed ? B_RDN : B_DN);
    issue_copies(D, c, g, what, routed ? s_sel[d.rank] : 0, j, H, buf + (what >= 0 ? o.slot(what & 1) : o.down_slot(d.np)),
                   s_tsc[routed], &bars[b], what >= 0 ? 0 : kDownW0);
    pend |= 1u << b;
  };
  // a group's first copies: part 0, and part 1 or else the down rows
  auto issue_start = [&](const DecLayer& D, int g) {
    issue(D, g, 0);
    issue(D, g, D.rank[c][g] < 0 && D.np[c][g] >= 2 ? 1 : -1);
  };
  // While this step's last group waits for its SwiGLU values, the next step's copies
  // that have room already: its router rows over this routed group's consumed part, and
  // for a next group like this one (shared, an even number >= 2 of parts, same buffer and
  // slots: this group's down rows sit in slot 0) its part 1 into the free slot 1, with
  // part 0 described for prepared_go once this group's down rows are used.  Returns
  // whether part 0 was described (bit 0) and the router rows issued (bit 1).
  auto issue_early = [&](const DecLayer& D, const DecLayer& DN, int g, const GroupDims& d, const GroupOff& o,
                         const uint8_t* buf) -> unsigned {
    unsigned r = 0;
    if (DN.routed[c] && d.rank >= 0 && (uint32_t)2 * a.RR * H <= o.slot0) {
      issue_router(DN);
      r |= 2u;
    }
    if (d.rank < 0 && d.np >= 2 && (d.np & 1) == 0 && DN.n_grp[c] > 0 && DN.rank[c][0] < 0 && group_buf(DN, 0) == buf) {
      const GroupDims dn = group_dims(DN, c, 0);
      const GroupOff on = GroupOff::of(dn.n, dn.W, dn.np, H);
      if (dn.np >= 2 && on.slot0 == o.slot0) {
        issue(DN, 0, 1);
        prepare_copies(DN, c, 0, 0, j, H, group_buf(DN, 0), s_tsc[0], &bars[B_GU0], 0, s_cp);
        pend |= 1u << B_GU0;
        r |= 1u;
      }
    }
    return r;
  };
  // a routed group's first copies (part 0 and the down rows), described before its
  // expert is known; prepared_go(s_cp, e) issues them
  auto prepare_routed = [&](const DecLayer& D) {
    prepare_routed_copies(D, j, H, s_big, s_tsc[1], &bars[B_RGU], &bars[B_RDN], s_cp);
    pend |= (1u << B_RGU) | (1u << B_RDN);
  };

  load_layer(0);
  store_layer(0);
  load_layer(1);
  store_layer(1);
  if (threadIdx.x < kWarps) s_cp[threadIdx.x].bytes = 0;
  if (threadIdx.x == 0) {
    s_abort = 0;
#pragma unroll 1
    for (int i = 0; i < 7; ++i) mbar_init(&bars[i], i == B_DNA ? kThreads : 1);
    mbar_init(&bar_hd[0], 1);
    mbar_init(&bar_hd[1], 1);
    mbar_init(&bar_h[0], 1);
    mbar_init(&bar_h[1], 1);
#pragma unroll 1
    for (int i = 0; i < 4; ++i) mbar_init(&bar_c[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync();                                   // every peer runs before any remote write

  unsigned step = 0;
#pragma unroll 1
  for (int t = 0; t < a.T; ++t) {
#pragma unroll 1
    for (int l = 0; l < a.L; ++l, ++step) {
      const int par = step & 1;
      const DecLayer& D = s_ly[step % 3];
      const DecLayer& DN = s_ly[(step + 1) % 3];     // valid when next_in_token
      const bool next_in_token = l + 1 < a.L;
      float* h_cur = s_h + par * H;
      float* lg = s_lg + par * a.Emax;
      load_layer(step + 2);                          // stored at the step's end
      // ---- a token's first step: the copies that were not made a step ahead (the
      // head used the buffers), and a router this cluster had no step ahead to fetch
      if (!s_abort) {
        if (D.routed[c] && !(pend & (1u << B_RT))) issue_router(D);
        if (l == 0 && D.n_grp[c] > 0 && D.rank[c][0] < 0) {
          issue_start(D, 0);
          pre = 1u;
        }
      }
      // ---- 1. stage x_l (and h_0 at a token's first layer)
      const float unscale = stage(a.x + (size_t)t * H, (l == 0 && a.residual) ? a.residual + (size_t)t * H : nullptr,
                                  l == 0, H, LPR, a.eps, h_cur, s_xb, reinterpret_cast<uint32_t*>(s_xl), s_red);
      if (c == 0 && j == 0) {
        const size_t o = ((size_t)t * a.L + l) * H;
        if (a.x_trace)
#pragma unroll 1
          for (int n = 4 * threadIdx.x; n < H; n += 4 * kThreads)
            *reinterpret_cast<uint2*>(a.x_trace + o + n) = *reinterpret_cast<const uint2*>(s_xb + n);
        if (a.h_trace)
#pragma unroll 1
          for (int n = 4 * threadIdx.x; n < H; n += 4 * kThreads)
            *reinterpret_cast<float4*>(a.h_trace + o + n) = *reinterpret_cast<const float4*>(h_cur + n);
      }
#pragma unroll 1
      for (int r = threadIdx.x; r < R16; r += kThreads) s_part[r] = 0.f;
      // ---- 2. router and top-k (routed clusters)
      int g_r = -1;                                  // the routed group issued after the top-k
      unsigned early = 0u;                           // the next step's copies made early (issue_early)
      if (D.routed[c]) {
        const int r0 = j * a.RR, nr = min(a.RR, D.E - r0);
        wait_bar(B_RT);
        if (nr > 0) router_rows(s_router, s_xb, H, r0, nr, s_bias[step % 3], s_acc, lg, &bar_lg[par]);
        // the first routed group's copies are described while the logits travel
#pragma unroll 1
        for (int g = 0; g < D.n_grp[c]; ++g)
          if (D.rank[c][g] >= 0) { g_r = g; break; }
        if (g_r >= 0 && s_abort) g_r = -1;
        if (g_r >= 0) prepare_routed(D);
        // all E logits in every CTA: E * 4 bytes on bar_lg
        if (threadIdx.x == 0) mbar_expect_tx(&bar_lg[par], (uint32_t)D.E * 4);
        mbar_wait_cluster(&bar_lg[par], (ph_c >> par) & 1u, sync, lim);
        ph_c ^= 1u << par;
        topk(lg, D.E, D.K, D.score, s_sel, s_w);
        // the first routed group's copies at once: the groups ahead of it (shared parts,
        // in flight already) run while they land
        if (g_r >= 0) {                              // its down rows once its part has landed
          prepared_go(s_cp, s_sel[D.rank[c][g_r]], 0);
          pre |= 1u << g_r;
        }
        if (c == 0 && j == 0 && threadIdx.x < D.K) {
          const size_t o = ((size_t)t * a.L + l) * a.Kmax + threadIdx.x;
          if (a.idx_out) a.idx_out[o] = s_sel[threadIdx.x];
          if (a.w_out) a.w_out[o] = s_w[threadIdx.x];
        }
      }
      // ---- 3. the cluster's groups
      const int ng = D.n_grp[c];
#pragma unroll 1
      for (int g = 0; g < ng; ++g, ++grp_seq) {
        const GroupDims d = group_dims(D, c, g);
        const GroupOff o = GroupOff::of(d.n, d.W, d.np, H);
        const bool routed = d.rank >= 0;
        const uint8_t* buf = group_buf(D, g);
        const float* tsc = s_tsc[routed];
        float* hsw = s_hsw + (grp_seq & 1) * kMaxW;
        float* hmax = s_hmax + (grp_seq & 1) * (kCS * kMaxParts);
        uint64_t* bar_sw = &bar_c[2 + (grp_seq & 1)];
        if (!(pre & (1u << g)) && !s_abort) issue_start(D, g);
#pragma unroll 1
        for (int part = 0; part < d.np; ++part) {
          const int sl = part & 1;
          wait_bar(routed ? B_RGU : B_GU0 + sl);
          if (g == g_r && part == 0) prepared_go(s_cp, s_sel[d.rank], kDownW0);
          const uint8_t* pb = buf + o.slot(sl);
          rows_dot<CPL>(pb, pb + a16(d.n * H), 2 * d.n, d.n, tsc[0] * unscale, tsc[1] * unscale, H, s_xl, s_gu);
          __syncthreads();
          if (threadIdx.x < d.n) s_tmp[threadIdx.x] = silu(s_gu[threadIdx.x]) * s_gu[d.n + threadIdx.x];
          __syncthreads();                           // s_tmp; this part's slot is free
          if (warp == 0) {
            // this CTA's max |value| of the part goes to every CTA with the values
            float m = 0.f;
#pragma unroll 1
            for (int i = lane; i < d.n; i += 32) m = fmaxf(m, fabsf(s_tmp[i]));
            m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
            if (lane < kCS) st_async1(hmax + part * kCS + j, m, bar_sw, lane);
          }
          if (!s_abort) {
            if (part + 2 < d.np) issue(D, g, part + 2);
            else if (d.np >= 2 && part == d.np - 2) issue(D, g, -1);
          }
          to_cluster_async(hsw + part * d.Wp + d.n * j, s_tmp, d.n / 4, bar_sw);
        }
        if (g == ng - 1 && next_in_token && !s_abort) early = issue_early(D, DN, g, d, o, buf);
        // the group's W SwiGLU values and the producers' maxima everywhere
        if (threadIdx.x == 0) mbar_expect_tx(bar_sw, (uint32_t)d.np * kCS * (4 * d.n + 4));
        mbar_wait_cluster(bar_sw, (ph_c >> (2 + (grp_seq & 1))) & 1u, sync, lim);
        ph_c ^= 1u << (2 + (grp_seq & 1));
        wait_bar(routed ? B_RDN : B_DN);
        wait_bar(B_DNA);
        const uint8_t* db = buf + o.down_slot(d.np);
        group_down(db, db + a16(R16 * d.W / 2), d.W, R16, hsw, hmax, d.np * kCS, s_hh, s_hl, s_acc,
                   tsc[2] * (routed ? s_w[d.rank] : 1.0f), s_part);
        __syncthreads();                             // the group buffer is free again
      }
      store_layer(step + 2);                         // read from the next step on
      // ---- 4. residual exchange.  A cluster that met no cluster barrier in this step
      // meets one here: then every one of its CTAs has staged its inputs before any of
      // them posts (out may alias residual).
      if (ng == 0 && !D.routed[c]) cluster_sync();
      unsigned long long* bd = a.board + (size_t)par * kDecMaxClusters * H;
      if (!(a.hold && step == 0 && blockIdx.x == 0)) post_rows(bd, c, H, j, step + 1, s_part);
      exchange(bd, a.NC, H, j, step + 1, s_pp, h_cur, s_hn, s_h + (par ^ 1) * H, &bar_h[par ^ 1],
               (!next_in_token && c == 0 && a.out) ? a.out + (size_t)t * H : nullptr, sync, lim, &s_abort);
      // the rest of the next step's copies that do not depend on its data (within a token;
      // at a token's end the head uses the buffers): the router rows, and the first group
      // when it is a shared one.  Issued after the exchange has read the clusters' words:
      // data streaming into the SM delays those reads.
      pre = 0u;
      if (early & 1u) {                              // part 1 is in flight already
        prepared_go(s_cp, 0, 0);
        pre = 1u;
      }
      if (next_in_token && !s_abort) {
        if (DN.routed[c] && !(early & 2u)) issue_router(DN);
        if (!(early & 1u) && DN.n_grp[c] > 0 && DN.rank[c][0] < 0) {
          issue_start(DN, 0);
          pre = 1u;
        }
      }
      // h_{l+1} complete here: the H * 4 bytes of the cluster's CTAs on bar_h (the barrier
      // each step meets earlier keeps a CTA from writing a buffer a peer still reads)
      if (threadIdx.x == 0) mbar_expect_tx(&bar_h[par ^ 1], (uint32_t)H * 4);
      mbar_wait_cluster(&bar_h[par ^ 1], (ph_h >> (par ^ 1)) & 1u, sync, lim);
      ph_h ^= 1u << (par ^ 1);
    }
    // ---------------- token t's outputs: x_L and the head
    if (!a.x_out && !a.head.codes) continue;
    const float unscale = stage(nullptr, nullptr, false, H, LPR, a.eps, s_h + (step & 1) * H, s_xb,
                                reinterpret_cast<uint32_t*>(s_xl), s_red);
    if (a.x_out && blockIdx.x == 0)
#pragma unroll 1
      for (int n = 4 * threadIdx.x; n < H; n += 4 * kThreads)
        *reinterpret_cast<uint2*>(a.x_out + (size_t)t * H + n) = *reinterpret_cast<const uint2*>(s_xb + n);
    if (!a.head.codes) continue;
    const int chunk = (a.V + G - 1) / G;
    const int v0 = min(a.V, blockIdx.x * chunk), v1 = min(a.V, v0 + chunk);
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    // the CTA's logits: the last 8 KB of the big region, past the head's ring (two slots
    // of at most kBigBytes / 2 - 8 KB each; peers never write the big region)
    float* s_lv = a.tokens ? reinterpret_cast<float*>(s_big + kBigBytes - 8192) : nullptr;
    head_phase<CPL>(a, t, v0, v1, s_xl, unscale, s_big, s_hv, s_lv, bar_hd, ph_hd, pend_hd, s_abort != 0, bv, bi);
    const unsigned ttag = (unsigned)t + 1;
    if (a.tokens) {
      // the CTA's K best logits, posted as tagged words; the last CTA draws the token
      unsigned* s_key = reinterpret_cast<unsigned*>(s_lv);
#pragma unroll 1
      for (int i = threadIdx.x; i < v1 - v0; i += kThreads) s_key[i] = order_key(s_lv[i]);
      __syncthreads();
      unsigned* s_wk = reinterpret_cast<unsigned*>(s_big);          // the head ring is drained
      int* s_wi = reinterpret_cast<int*>(s_big + 4 * kWarps * 32);
      unsigned* s_fk = reinterpret_cast<unsigned*>(s_big + 8 * kWarps * 32);
      int* s_fi = reinterpret_cast<int*>(s_big + 8 * kWarps * 32 + 128);
      block_topk(s_key, nullptr, v1 - v0, a.top_k, v0, s_wk, s_wi, s_fk, s_fi);
      unsigned long long* cand = a.cand + (size_t)(t & 1) * kMaxG * 64;
      if (threadIdx.x < a.top_k) {
        unsigned long long* w = cand + 2 * ((size_t)blockIdx.x * 32 + threadIdx.x);
        st_tagged(w, ((unsigned long long)ttag << 32) | s_fk[threadIdx.x]);
        st_tagged(w + 1, ((unsigned long long)ttag << 32) | (unsigned)s_fi[threadIdx.x]);
      }
      if (blockIdx.x == G - 1) {
        __syncthreads();
        unsigned* s_ck = reinterpret_cast<unsigned*>(s_big + 8 * kWarps * 32 + 256);
        int* s_ci = reinterpret_cast<int*>(s_big + 8 * kWarps * 32 + 256 + 4 * kMaxG * 32);
        head_sample(cand, G, a.top_k, ttag, a.temp, a.top_p, __ldg(a.uniforms + t), a.V, a.tokens + t,
                    a.argmax ? a.argmax + t : nullptr, s_ck, s_ci, s_wk, s_wi, s_fk, s_fi, sync, lim);
      }
    } else {
      best_reduce_warp(bv, bi);
      if (lane == 0) { s_bv[warp] = bv; s_bi[warp] = bi; }
      __syncthreads();
      unsigned long long* best = a.best + (size_t)(t & 1) * kMaxG * 2;
      if (threadIdx.x == 0) {
#pragma unroll 1
        for (int w = 1; w < kWarps; ++w)
          if (s_bv[w] > bv || (s_bv[w] == bv && s_bi[w] < bi)) { bv = s_bv[w]; bi = s_bi[w]; }
        st_tagged(best + 2 * blockIdx.x, ((unsigned long long)ttag << 32) | __float_as_uint(bv));
        st_tagged(best + 2 * blockIdx.x + 1, ((unsigned long long)ttag << 32) | (unsigned)bi);
      }
      // the last CTA (in the cluster with the most slack) reduces the CTAs' maxima
      if (blockIdx.x == G - 1 && warp == 0)
        head_argmax(best, G, ttag, a.V, a.argmax ? a.argmax + t : nullptr, sync, lim);
    }
    __syncthreads();                                 // s_xb / s_xl are restaged next
  }
  // Copies are issued only for a step that follows and waited for in the step they
  // serve, so normally nothing is in flight here; after an abort, what a skipped wait
  // left in flight is drained (bounded) before the CTA exits.  The last remote writes
  // (the last step's h rows) have landed: each CTA waited for them on bar_h.
#pragma unroll 1
  for (int i = 0; i < 7; ++i) wait_bar(i);
#pragma unroll 1
  for (int k = 0; k < 2; ++k)
    if (pend_hd & (1u << k)) mbar_wait(&bar_hd[k], (ph_hd >> k) & 1u, sync, lim);
}

// ---------------------------------------------------------------- host side
static std::atomic<int> g_clusters[64];

template <int CPL>
static cudaError_t prepare(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(k_decode<CPL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode<CPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// The largest carve any accepted shape needs.
static size_t max_smem() { return Smem::of(2048, kMaxE).total; }

}  // namespace dc

// Clusters of 16 this device runs at once with the decode kernel's resources (at most
// kDecMaxClusters); 0 when there is no device or the query fails.
int decode_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = dc::g_clusters[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  const size_t smem = dc::max_smem();
  if (dc::prepare<1>(smem) != cudaSuccess || dc::prepare<2>(smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dc::kCS * kDecMaxClusters);
  cfg.blockDim = dim3(dc::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = dc::kCS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int m = 0;
  if (cudaOccupancyMaxActiveClusters(&m, dc::k_decode<2>, &cfg) != cudaSuccess) return 0;
  n = m < kDecMaxClusters ? m : kDecMaxClusters;
  if (n > 0) dc::g_clusters[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Router rows per CTA for E experts: a multiple of 4, so that every CTA's logits are
// whole 16-byte pieces; the logit array holds 16 of them.
int decode_router_rows(int E) { return (((E + dc::kCS - 1) / dc::kCS) + 3) & ~3; }

size_t decode_workspace_bytes(int H) {
  return 256 + (size_t)2 * kDecMaxClusters * H * 8 + (size_t)2 * dc::kMaxG * 2 * 8 +
         (size_t)2 * dc::kMaxG * 64 * 8;
}

size_t decode_smem_bytes(int H, int Emax) { return dc::Smem::of(H, Emax).total; }

void decode_carve(DecodeArgs& a, void* ws) {
  char* p = static_cast<char*>(ws);
  a.sync = reinterpret_cast<unsigned*>(p);
  p += 256;
  a.board = reinterpret_cast<unsigned long long*>(p);
  p += (size_t)2 * kDecMaxClusters * a.H * 8;
  a.best = reinterpret_cast<unsigned long long*>(p);
  p += (size_t)2 * dc::kMaxG * 2 * 8;
  a.cand = reinterpret_cast<unsigned long long*>(p);
}

bool decode_plan_layer(DecLayer& d, int H, int NC) {
  if (NC < 1 || NC > kDecMaxClusters) return false;
  if (H < 256 || H > 2048 || (H & (H - 1))) return false;
  std::memset(d.rank, -1, sizeof(d.rank));
  std::memset(d.np, 0, sizeof(d.np));
  std::memset(d.p0, 0, sizeof(d.p0));
  std::memset(d.n_grp, 0, sizeof(d.n_grp));
  std::memset(d.routed, 0, sizeof(d.routed));
  if (d.Fs < 0 || d.K < 0 || d.E < 0) return false;
  if (d.K > 0) {
    const int RR = decode_router_rows(d.E);
    if (d.E > dc::kMaxE || d.K > d.E || d.K > FLINT_MAX_TOP_K) return false;
    if (RR > dc::kMaxRR || (size_t)2 * RR * H > (size_t)dc::kRouterBytes) return false;
    const int n = d.F / dc::kCS;
    if (d.F < 64 || (d.F & (d.F - 1)) || n > dc::kMaxN || d.F > dc::kMaxW) return false;
  }
  // Routed experts on clusters [0, NR), one cluster per selected expert when there are
  // enough (a cluster takes a second one otherwise).
  int NR = 0;
  if (d.K > 0) {
    NR = d.K < (d.Fs > 0 ? NC - 1 : NC) ? d.K : (d.Fs > 0 ? NC - 1 : NC);
    if (NR < 1) NR = 1;
  }
  int n_routed[kDecMaxClusters] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int s = 0; s < d.K; ++s) ++n_routed[s % NR];
  for (int cc = 0; cc < NC; ++cc)
    if (n_routed[cc] > kDecMaxGroups) return false;
  // The shared expert in parts of Wsh outputs, as contiguous runs on the clusters
  // without a routed expert (a group costs a few microseconds of fixed latency, so few
  // large groups beat many small ones); with no such cluster, on the routed clusters
  // with a free group, ahead of their routed groups.
  int sh_np[kDecMaxClusters] = {0, 0, 0, 0, 0, 0, 0, 0};
  d.Wsh = 0;
  if (d.Fs > 0) {
    if (d.Fs < 64 || d.Fs % 64) return false;
    int hosts[kDecMaxClusters], nh = 0;
    for (int cc = NR; cc < NC; ++cc) hosts[nh++] = cc;
    if (nh == 0)
      for (int cc = 0; cc < NR; ++cc)
        if (n_routed[cc] < kDecMaxGroups) hosts[nh++] = cc;
    if (nh == 0) return false;
    // parts of at most 512 outputs (and of the routed width when there is one); at most
    // one run per host
    int w = d.K > 0 ? (d.F < d.Fs ? d.F : d.Fs) : (d.Fs < 512 ? d.Fs : 512);
    if (w > 512) w = 512;
    while (w > 64 && (d.Fs % w || (w / dc::kCS) % 4)) w -= 64;   // a divisor of Fs, n % 4 == 0
    if (d.Fs % w || (w / dc::kCS) % 4) return false;
    d.Wsh = w;
    const int S = d.Fs / d.Wsh;
    const int used = S < nh ? S : nh;
    for (int i = 0; i < used; ++i) sh_np[hosts[i]] = S / used + (i < S % used ? 1 : 0);
  }
  if (d.K == 0 && d.Fs == 0) return false;
  const uint32_t routed_bytes = d.K > 0 ? dc::GroupOff::of(d.F / dc::kCS, d.F, 1, H).bytes : 0u;
  d.sh_off = (uint32_t)((dc::kRouterBytes > routed_bytes ? dc::kRouterBytes : routed_bytes) + 127) & ~127u;
  if (d.K > 0 && routed_bytes > (uint32_t)dc::kBigBytes) return false;
  int p = 0;
  for (int cc = 0; cc < NC; ++cc) {
    if (sh_np[cc] > 0) {
      const int n = d.Wsh / dc::kCS, W = sh_np[cc] * d.Wsh;
      if (n < 4 || n > dc::kMaxN || (n & 3) || W > dc::kMaxW) return false;
      const uint32_t base = n_routed[cc] > 0 ? d.sh_off : 0u;
      if (base + dc::GroupOff::of(n, W, sh_np[cc], H).bytes > (uint32_t)dc::kBigBytes) return false;
      const int g = d.n_grp[cc]++;
      d.rank[cc][g] = -1;
      d.np[cc][g] = (unsigned char)sh_np[cc];
      d.p0[cc][g] = (unsigned char)p;
      p += sh_np[cc];
    }
  }
  for (int s = 0; s < d.K; ++s) {
    const int cc = s % NR;
    if (d.n_grp[cc] >= kDecMaxGroups) return false;
    const int g = d.n_grp[cc]++;
    d.rank[cc][g] = (signed char)s;
    d.np[cc][g] = 1;
    d.routed[cc] = 1;
  }
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.sync, 0, decode_workspace_bytes(a.H), st);
  if (e != cudaSuccess) return e;
  const size_t smem = decode_smem_bytes(a.H, a.Emax);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.NC * dc::kCS);
  cfg.blockDim = dim3(dc::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = dc::kCS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (a.H > 1024) return cudaLaunchKernelEx(&cfg, dc::k_decode<2>, a);
  return cudaLaunchKernelEx(&cfg, dc::k_decode<1>, a);
}

}  // namespace flint
