// prefill.cu -- one Flint MoE layer over T prompt tokens ("Flint-40B-A2B: AI-Built MoE
// Coding Model Hits 125 tok/s on MacBook Pro", section "Custom Inference Kernels": prompt
// processing), as a token-permuted grouped GEMM on block-scaled FP4 tensor cores.
//
//   1 router      logits[T, E] = x Wr^T (+ bias): tcgen05 kind::f16 (bf16 in, fp32 acc),
//                 128 tokens x all E experts per CTA, split 4 ways along K
//   2 top-k       per token (one warp): the partial logits summed in order plus the
//                 bias, softmax top-k, renormalised weights; per-expert token bitmaps
//   3 scan        per expert (one warp): prefix counts of its bitmap words; then one CTA:
//                 counts, offsets (plain and padded to 128-row tiles) and the
//                 device-side item lists
//   4 scatter     per token: x quantised to NVFP4 once (unit tensor scale) and written
//                 to the shared expert's operand Xq and to the K expert-major rows of Xp
//                 (each expert's rows start on a 128-row tile); out[t] = x[t] (fp32)
//   5 gate/up     grouped GEMM, tcgen05 kind::mxf4nvf4 (E2M1 x E2M1, E4M3 scale per
//                 16): per 128-row tile of one expert, the gate and up tiles accumulate
//                 in TMEM; the epilogue applies the tensor scales, SwiGLU, and
//                 quantises h to NVFP4 (unit tensor scale)
//   6 down        grouped GEMM as 5 over the shared and the routed tiles; the epilogue
//                 adds y (shared rows) and w_pair * y (routed rows, at their token: the
//                 un-permuting combine) into out with fp32 reductions (red.global.add),
//                 so the routed rows never go to memory.  The adds into one element
//                 commute but their order is not fixed: out may differ from run to run
//                 in its last bits
//
// Every FP4 operand's block scales are kept in the MMA scale layout (512 bytes per
// 128-row tile and 64 columns, see flint.h), so one pipeline stage of a GEMM is four
// TMA transfers: A codes and B codes (2D tensor maps, 128-byte swizzle) and A and B
// scales (bulk copies).  GEMM CTAs are warp-specialised (12 warps): warp 0 issues the
// TMA loads, warp 1 allocates TMEM and issues tcgen05.cp / tcgen05.mma, warps 4-11 read
// the accumulator back (tcgen05.ld; two warps per TMEM lane quarter, one per column
// half) and hand it back to the MMA warp before their arithmetic.  Waits are bounded:
// on expiry the CTA records FLINT_ERR_TIMEOUT and unwinds.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace flint {
namespace pf {

constexpr int kBM = 128;          // rows per tile (TMEM lanes)
constexpr int kBN = 128;          // output columns per B tile
constexpr int kGThreads = 384;    // 12 warps
constexpr int kWarpTMA = 0, kWarpMMA = 1, kWarpEpi0 = 4, kEpiWarps = 8;

struct __align__(16) Item {
  int kx;       // kind << 16 | expert; kind 0 = shared expert, 1 = routed expert
  int row0;     // first A row of the tile (a multiple of 128)
  int rows;     // valid rows (<= kBM)
  int n0;       // first output column
  __device__ int kind() const { return kx >> 16; }
  __device__ int expert() const { return kx & 0xFFFF; }
};
__device__ __forceinline__ Item load_item(const Item* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return Item{v.x, v.y, v.z, v.w};
}

enum Mode { kGateUp = 1, kDown = 2 };

template <int MODE>
struct Cfg {
  static constexpr int kB = MODE == kGateUp ? 2 : 1;      // B tiles per stage (gate + up)
  static constexpr int kStages = MODE == kGateUp ? 4 : 6;
  static constexpr int a = 0;                             // A codes, 128 rows x 128 B
  static constexpr int b = 16384;                         // B codes, kB x 16 KB
  static constexpr int sfa = b + kB * 16384;              // A scales, 4 x 512 B
  static constexpr int sfb = sfa + 2048;                  // B scales, kB x 4 x 512 B
  static constexpr int bytes = sfb + kB * 2048;
  static constexpr int stride = (bytes + 1023) / 1024 * 1024;
  static constexpr int smem = kStages * stride + 1024;
  static constexpr int dcols = kB * kBN;                  // accumulator columns
  static constexpr int sf_step = 4 + 4 * kB;              // TMEM scale columns per K=64 step
  static constexpr uint32_t tmem_cols = 512;
  static_assert(dcols + kStages * 4 * sf_step <= (int)tmem_cols, "TMEM budget");
};

struct GemmArgs {
  CUtensorMap mapA[2];          // A codes: [0] shared-expert rows, [1] expert-major rows
  CUtensorMap mapB[4];          // gate/up: sh_gate, sh_up, gate, up; down: sh_down, -, down, -
  const uint8_t* sfA[2];        // A scales, MMA scale layout
  const uint8_t* sfB[4];        // B scales, MMA scale layout
  int Kel[2];                   // K in elements: shared / routed
  int rowsB[2];                 // rows of one weight matrix: shared / routed
  const Item* items;
  const int* n_items;           // device count
  // epilogues
  const float* tscA[2];         // gate / sh_gate (down: down / sh_down) tensor scales
  const float* tscB[2];         // up / sh_up tensor scales
  uint8_t* hcodes[2];           // gate/up output codes: [0] shared h [Tp][Fs/2], [1] routed h
  uint8_t* hsf[2];              // gate/up output scales, MMA scale layout
  int Fout[2];
  float* out;                   // [T][H]: x (from the scatter), the down tiles add into it
  const int32_t* order;         // padded routed row -> pair id
  const float* wpair;           // [T*K]
  int H, K;
  unsigned long long wait_ns;   // bound of every wait
  int hold;                     // test aid: CTA 0's copy issuer withholds its first stage
};

// ---------------------------------------------------------------- primitives
__device__ __forceinline__ uint32_t sh(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)(16 >> 4) << 16;           // leading byte offset (unused with 128B swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;         // 8-row groups 1024 bytes apart
  d |= 1ull << 46;                          // tcgen05 descriptor version
  d |= 2ull << 61;                          // 128-byte swizzle
  return d;
}
__device__ __forceinline__ uint64_t sf_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;          // 8 rows x 16 bytes per core matrix
  d |= 1ull << 46;
  return d;
}

__device__ __forceinline__ void mb_init(uint64_t* b, unsigned n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(sh(b)), "r"(n));
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(sh(b)) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(sh(b)), "r"(bytes) : "memory");
}
// Bounded parity wait (limit in ns of %globaltimer); false on expiry (FLINT_ERR_TIMEOUT
// recorded, *abort set) or once *abort is set.
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t parity, volatile int* abort,
                                        unsigned long long limit) {
  unsigned long long t0 = 0;
  for (unsigned i = 0;; ++i) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
                 "selp.u32 %0, 1, 0, p; }" : "=r"(ok) : "r"(sh(b)), "r"(parity) : "memory");
    if (ok) return true;
    if ((i & 63u) == 63u) {
      if (*abort) return false;
      const unsigned long long now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit) {
        raise_status(FLINT_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
               "[%0], [%1, {%2, %3}], [%4];"
               :: "r"(sh(dst)), "l"(m), "r"(x), "r"(y), "r"(sh(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(sh(dst)), "l"(src), "r"(bytes), "r"(sh(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(sh(b)) : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc,
                                        uint32_t sfa, uint32_t sfb) {
  asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; "
               "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%5], [%6], p; }"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; "
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// 32 lanes x 16 consecutive fp32 columns; thread (lane) gets its row.  No wait.
__device__ __forceinline__ void tmem_ld16(uint32_t t, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(t));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Byte offset of (row, 64-column step k) in an MMA scale layout with K/64 steps per row tile.
__device__ __forceinline__ size_t sf_word_offset(int row, int k, int ksteps) {
  return ((size_t)(row >> 7) * ksteps + k) * 512 + 16 * (row & 31) + 4 * ((row & 127) >> 5);
}

// 16 fp32 values -> one NVFP4 block with unit tensor scale (the quantiser's recipe).
__device__ __forceinline__ void quant_block_unit(const float* v, uint2& codes, uint32_t& scale) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t s = to_e4m3(__fdiv_rn(__fdiv_rn(amax, 6.0f), 1.0f));
  const float eff = e4m3_value(s);
  uint32_t packed[2] = {0u, 0u};
  if (eff != 0.f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = to_e2m1x2(__fdiv_rn(v[2 * j], eff), __fdiv_rn(v[2 * j + 1], eff));
      packed[j >> 2] |= byte << (8 * (j & 3));
    }
  }
  codes = make_uint2(packed[0], packed[1]);
  scale = s;
}

// The same recipe for the GEMM epilogue: the block's effective scale is applied as a
// product with its reciprocal, and SwiGLU uses the fast exponential and division.
// (h comes from fp32 accumulators, so its codes are compared within tolerance, never
// bit for bit.)
__device__ __forceinline__ void quant_block_unit_fast(const float* v, uint2& codes, uint32_t& scale) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t s = to_e4m3(__fdiv_rn(amax, 6.0f));
  const float eff = e4m3_value(s);
  uint32_t packed[2] = {0u, 0u};
  if (eff != 0.f) {
    const float inv = __frcp_rn(eff);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = to_e2m1x2(v[2 * j] * inv, v[2 * j + 1] * inv);
      packed[j >> 2] |= byte << (8 * (j & 3));
    }
  }
  codes = make_uint2(packed[0], packed[1]);
  scale = s;
}
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ---------------------------------------------------------------- grouped FP4 GEMM
template <int MODE>
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_fp4(const __grid_constant__ GemmArgs g) {
  using C = Cfg<MODE>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[S], empty[S], accf, acce;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mb_init(&full[s], 1); mb_init(&empty[s], 1); }
    mb_init(&accf, 1);
    mb_init(&acce, kEpiWarps);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(sh(&tmem_base)), "r"(C::tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int n_items = __ldcg(g.n_items);
  const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

  if (warp == kWarpTMA && lane == 0) {
    uint32_t it = 0;
    int last[S];                                  // per stage slot: the last issued iteration
#pragma unroll
    for (int s = 0; s < S; ++s) last[s] = -1;
    Item nxt = blockIdx.x < n_items ? load_item(g.items + blockIdx.x) : Item{0, 0, 0, 0};
    for (int i = blockIdx.x; i < n_items && !abort_flag; i += gridDim.x) {
      const Item item = nxt;
      if (i + (int)gridDim.x < n_items) nxt = load_item(g.items + i + gridDim.x);
      const int K = g.Kel[item.kind()], ksteps = K / 64;
      const int brow = item.expert() * g.rowsB[item.kind()] + item.n0;
      const uint8_t* sfa = g.sfA[item.kind()] + (size_t)(item.row0 >> 7) * ksteps * 512;
      for (int kt = 0; kt < K / 256; ++kt, ++it) {
        const int s = it % S;
        if (it >= S && !mb_wait(&empty[s], ((it / S) - 1) & 1, &abort_flag, g.wait_ns)) break;
        if (g.hold && blockIdx.x == 0 && it == 0) continue;   // withheld: its phase never completes
        last[s] = (int)it;
        uint8_t* st = smem + s * C::stride;
        mb_expect(&full[s], C::bytes);
        tma2d(st + C::a, &g.mapA[item.kind()], kt * 128, item.row0, &full[s]);
        bulk_g2s(st + C::sfa, sfa + (size_t)kt * 2048, 2048, &full[s]);
#pragma unroll
        for (int b = 0; b < C::kB; ++b) {
          tma2d(st + C::b + b * 16384, &g.mapB[2 * item.kind() + b], kt * 128, brow, &full[s]);
          bulk_g2s(st + C::sfb + b * 2048,
                   g.sfB[2 * item.kind() + b] + ((size_t)(brow >> 7) * ksteps + 4 * kt) * 512, 2048, &full[s]);
        }
      }
    }
    // after an expired wait: the stages issued but not consumed land before the CTA exits
    if (abort_flag) {
      volatile int no_abort = 0;
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (last[s] >= 0) mb_wait(&full[s], (last[s] / S) & 1, &no_abort, g.wait_ns);
    }
  } else if (warp == kWarpMMA && lane == 0) {
    const uint64_t dA0 = umma_desc_sw128(sh(smem + C::a)), dB0 = umma_desc_sw128(sh(smem + C::b));
    const uint64_t dSA0 = sf_desc(sh(smem + C::sfa)), dSB0 = sf_desc(sh(smem + C::sfb));
    uint32_t it = 0, done = 0;
    Item nxt = blockIdx.x < n_items ? load_item(g.items + blockIdx.x) : Item{0, 0, 0, 0};
    for (int i = blockIdx.x; i < n_items && !abort_flag; i += gridDim.x, ++done) {
      const Item item = nxt;
      if (i + (int)gridDim.x < n_items) nxt = load_item(g.items + i + gridDim.x);
      const int kt_n = g.Kel[item.kind()] / 256;
      if (done > 0 && !mb_wait(&acce, (done - 1) & 1, &abort_flag, g.wait_ns)) break;
      tc_fence_after();
      bool ok = true;
      for (int kt = 0; kt < kt_n; ++kt, ++it) {
        const int s = it % S;
        if (!mb_wait(&full[s], (it / S) & 1, &abort_flag, g.wait_ns)) { ok = false; break; }
        tc_fence_after();
        // descriptors of stage s: the stage-0 ones plus the stage offset (address field)
        const uint64_t so = (uint64_t)(s * (C::stride >> 4));
        const uint32_t sf0 = tmem + C::dcols + (uint32_t)(s * 4 * C::sf_step);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t sfs = sf0 + kk * C::sf_step;
          tc_cp_sf(sfs, dSA0 + so + kk * (512 >> 4));
#pragma unroll
          for (int b = 0; b < C::kB; ++b) tc_cp_sf(sfs + 4 + 4 * b, dSB0 + so + ((b * 2048 + kk * 512) >> 4));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t sfs = sf0 + kk * C::sf_step;
          const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
          for (int b = 0; b < C::kB; ++b)
            mma_fp4(tmem + b * kBN, dA0 + so + kk * 2, dB0 + so + ((b * 16384) >> 4) + kk * 2, idesc, acc, sfs,
                    sfs + 4 + 4 * b);
        }
        tc_commit(&empty[s]);
      }
      if (!ok) break;
      tc_commit(&accf);
    }
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;                                 // TMEM lane quarter
    const int hf = (warp - kWarpEpi0) >> 2;                 // column half: [64 hf, 64 hf + 64)
    const int r = q * 32 + lane;                            // tile row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t done = 0;
    // What an item's epilogue reads from global memory (its tensor scales; for a routed
    // down tile this row's token and pair weight, two dependent loads) is loaded one item
    // ahead, so that its latency passes while the tensor cores work.
    auto item_vals = [&](const Item& it, float& v0, float& v1, int& tok) {
      const int kd = it.kind(), ex = kd ? it.expert() : 0;
      v0 = g.tscA[kd][ex];
      tok = it.row0 + r;
      if (MODE == kGateUp) {
        v1 = g.tscB[kd][ex];
      } else {
        v1 = 1.0f;
        if (kd != 0 && r < it.rows) {
          const int pair = g.order[it.row0 + r];
          tok = pair / g.K;
          v1 = g.wpair[pair];
        }
      }
    };
    Item nxt = blockIdx.x < n_items ? load_item(g.items + blockIdx.x) : Item{0, 0, 0, 0};
    float nv0 = 0.f, nv1 = 0.f;
    int ntok = 0;
    if (blockIdx.x < n_items) item_vals(nxt, nv0, nv1, ntok);
    for (int i = blockIdx.x; i < n_items && !abort_flag; i += gridDim.x, ++done) {
      const Item item = nxt;
      const float v0 = nv0, v1 = nv1;
      const int vtok = ntok;
      if (i + (int)gridDim.x < n_items) {
        nxt = load_item(g.items + i + gridDim.x);
        item_vals(nxt, nv0, nv1, ntok);
      }
      if (!mb_wait(&accf, done & 1, &abort_flag, g.wait_ns)) break;
      tc_fence_after();
      const bool valid = r < item.rows;
      const int arow = item.row0 + r;
      if (MODE == kGateUp) {
        const float tg = v0;
        const float tu = v1;
        float h[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t gv[16], uv[16];
          tmem_ld16(lane_base + 64 * hf + c0, gv);
          tmem_ld16(lane_base + kBN + 64 * hf + c0, uv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            h[c0 + j] = silu_fast(__uint_as_float(gv[j]) * tg) * (__uint_as_float(uv[j]) * tu);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mb_arrive(&acce);                  // accumulator free for the next item
        if (valid) {
          const int F = g.Fout[item.kind()];
          const int col = item.n0 + 64 * hf;
          uint8_t* hc = g.hcodes[item.kind()] + (size_t)arow * (F / 2) + col / 2;
          uint32_t sw = 0;
          uint2 cw[4];
#pragma unroll
          for (int b4 = 0; b4 < 4; ++b4) {
            uint32_t sc;
            quant_block_unit_fast(h + 16 * b4, cw[b4], sc);
            sw |= sc << (8 * b4);
          }
          *reinterpret_cast<uint4*>(hc) = make_uint4(cw[0].x, cw[0].y, cw[1].x, cw[1].y);
          *reinterpret_cast<uint4*>(hc + 16) = make_uint4(cw[2].x, cw[2].y, cw[3].x, cw[3].y);
          *reinterpret_cast<uint32_t*>(g.hsf[item.kind()] + sf_word_offset(arow, col / 64, F / 64)) = sw;
        }
      } else {  // down
        float y[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(lane_base + 64 * hf + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) y[c0 + j] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mb_arrive(&acce);
        if (valid) {
          const int col = item.n0 + 64 * hf;
          // shared rows: token arow, weight 1; routed rows: the pair's token and weight
          const int tok = vtok;
          const float scale = v0 * v1;
          float* o = g.out + (size_t)tok * g.H + col;
#pragma unroll
          for (int j = 0; j < 64; j += 4)
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "l"(o + j), "f"(y[j] * scale), "f"(y[j + 1] * scale), "f"(y[j + 2] * scale),
                            "f"(y[j + 3] * scale) : "memory");
        }
      }
    }
  }
  // unwind: every role is done (or gave up); no MMA may be in flight at dealloc
  __syncthreads();
  if (warp == kWarpMMA) {
    if (lane == 0 && abort_flag) {
      __shared__ __align__(8) uint64_t drain;
      mb_init(&drain, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      tc_commit(&drain);
      volatile int no_abort = 0;
      mb_wait(&drain, 0, &no_abort, g.wait_ns);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(C::tmem_cols));
  }
}

// ---------------------------------------------------------------- warp top-k (k_topk)
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

// ---------------------------------------------------------------- router GEMM (bf16)
// Partial logits over one K split: part[ks][t][e] = x[t, K_ks] . Wr[e, K_ks] for 128 tokens
// and all E (<= 256) experts per CTA; A = x rows (TMA, 64 bf16 = 128 B per K-tile), B =
// the router rows, tcgen05 kind::f16 (K = 16 per instruction), one N = E instruction per
// K = 16.  The top-k kernel sums the kRSplit partials in order and adds the bias.
constexpr int kRStages = 4;
constexpr int kRSplit = 4;
constexpr int kRThreads = 256;

struct RouterArgs {
  CUtensorMap mapX;
  CUtensorMap mapW;
  float* part;             // [kRSplit][T][E]
  int T, E, H;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(kRThreads, 1) k_router_gemm(const __grid_constant__ RouterArgs g) {
  constexpr int kStageBytes = 16384 + 256 * 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], accf;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) { mb_init(&full[s], 1); mb_init(&empty[s], 1); }
    mb_init(&accf, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(sh(&tmem_base)), "r"(256));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int row0 = blockIdx.x * kBM, ks = blockIdx.y;
  const int kt_n = g.H / 64 / kRSplit, kt0 = ks * kt_n;
  const uint32_t stage_bytes = 16384 + (uint32_t)g.E * 128;
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(g.E >> 3) << 17) |
                         ((uint32_t)(kBM >> 4) << 24);
  if (warp == kWarpTMA && lane == 0) {
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % kRStages;
      if (kt >= kRStages && !mb_wait(&empty[s], ((kt / kRStages) - 1) & 1, &abort_flag, g.wait_ns)) break;
      uint8_t* st = smem + s * kStageBytes;
      mb_expect(&full[s], stage_bytes);
      tma2d(st, &g.mapX, (kt0 + kt) * 128, row0, &full[s]);
      tma2d(st + 16384, &g.mapW, (kt0 + kt) * 128, 0, &full[s]);
    }
  } else if (warp == kWarpMMA && lane == 0) {
    const uint64_t dA0 = umma_desc_sw128(sh(smem)), dB0 = umma_desc_sw128(sh(smem + 16384));
    bool ok = true;
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % kRStages;
      if (!mb_wait(&full[s], (kt / kRStages) & 1, &abort_flag, g.wait_ns)) { ok = false; break; }
      tc_fence_after();
      const uint64_t so = (uint64_t)(s * (kStageBytes >> 4));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem, dA0 + so + kk * 2, dB0 + so + kk * 2, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    if (ok) tc_commit(&accf);
  } else if (warp >= 4) {
    const int q = warp & 3;
    const int t = row0 + q * 32 + lane;
    if (mb_wait(&accf, 0, &abort_flag, g.wait_ns)) {
      tc_fence_after();
      float* dst = g.part + ((size_t)ks * g.T + t) * g.E;
      for (int c0 = 0; c0 < g.E; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        tmem_wait_ld();
        if (t < g.T)
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                   __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      }
      tc_fence_before();
    }
  }
  __syncthreads();
  if (warp == kWarpMMA) {
    if (lane == 0 && abort_flag) {
      __shared__ __align__(8) uint64_t drain;
      mb_init(&drain, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      tc_commit(&drain);
      volatile int no_abort = 0;
      mb_wait(&drain, 0, &no_abort, g.wait_ns);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(256));
  }
}

// ---------------------------------------------------------------- routing bookkeeping
struct RouteArgs {
  int T, E, K, W;          // W = words per expert bitmap = ceil(T/32)
  const float* part;       // [kRSplit][T][E] partial logits
  const float* bias;       // [E] or null
  int sigmoid;             // weights from sigmoid scores instead of the softmax
  int32_t* idx;            // [T][K]
  float* w;                // [T][K]
  int32_t* idx_out;
  float* w_out;
  unsigned* bits;          // [E][W]
  int* wordpre;            // [E][W]
  int* counts;             // [E]
  int* offsets;            // [E] expert-major offsets
  int* offp;               // [E] the same, each expert padded to 128-row tiles
  int32_t* counts_out;
};

// One warp per token: the logits (partials summed in order, plus the bias), top-k (the
// exact warp top-k of topk_dispatch) and the expert bitmaps.
__global__ void __launch_bounds__(256) k_topk(RouteArgs a) {
  __shared__ int s_sel[8][FLINT_MAX_TOP_K];
  __shared__ float s_w[8][FLINT_MAX_TOP_K];
  __shared__ float s_lg[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  for (int e = lane; e < a.E; e += 32) {
    float v = a.part[(size_t)t * a.E + e];
#pragma unroll
    for (int ks = 1; ks < kRSplit; ++ks) v += a.part[((size_t)ks * a.T + t) * a.E + e];
    s_lg[warp][e] = v + (a.bias ? a.bias[e] : 0.f);
  }
  __syncwarp();
  topk_dispatch(s_lg[warp], a.E, a.K, s_sel[warp], s_w[warp]);
  if (a.sigmoid) {
    // the same experts; weights = their sigmoid scores over the selected sum
    float p = 0.f;
    if (lane < a.K) {
      float l = s_lg[warp][s_sel[warp][lane]];
      l = (l == l) ? l : -INFINITY;
      p = 1.0f / (1.0f + expf(-l));
    }
    float z = p;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < a.K) s_w[warp][lane] = p / z;
    __syncwarp();
  }
  if (lane < a.K) {
    const int e = s_sel[warp][lane];
    const float wv = s_w[warp][lane];
    a.idx[t * a.K + lane] = e;
    a.w[t * a.K + lane] = wv;
    if (a.idx_out) a.idx_out[t * a.K + lane] = e;
    if (a.w_out) a.w_out[t * a.K + lane] = wv;
    atomicOr(&a.bits[(size_t)e * a.W + (t >> 5)], 1u << (t & 31));
  }
}

// One warp per expert: prefix counts of its token-bitmap words (the rank of a token
// among the expert's tokens is wordpre + popc of the lower bits of its word) and the
// expert's token count.
__global__ void __launch_bounds__(256) k_expert_prefix(RouteArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= a.E) return;
  const unsigned* bits = a.bits + (size_t)e * a.W;
  int* pre = a.wordpre + (size_t)e * a.W;
  int run = 0;
  for (int base = 0; base < a.W; base += 128) {
    int v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int w = base + 32 * k + lane;
      v[k] = w < a.W ? __popc(__ldcg(bits + w)) : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int w = base + 32 * k + lane;
      int incl = v[k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (w < a.W) pre[w] = run + incl - v[k];
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) a.counts[e] = run;
}

// One CTA: expert offsets (plain and tile-padded) and the item lists of both GEMMs.
struct ScanArgs {
  RouteArgs r;
  Item* items_gu;          // gate/up items: shared first, then routed
  int* n_items_gu;
  Item* items_dn;          // down items: shared first, then routed
  int* n_items_dn;
  int H, F, Fs;
};

__global__ void __launch_bounds__(1024) k_scan(ScanArgs s) {
  const RouteArgs& a = s.r;
  __shared__ int s_cnt[FLINT_MAX_EXPERTS], s_toff[FLINT_MAX_EXPERTS];
  __shared__ int s_wsum[2][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = __ldcg(a.counts + e);
  __syncthreads();
  // exclusive scans over experts of the counts and of the 128-row tile counts
  const int e = threadIdx.x;
  const int cnt = e < a.E ? s_cnt[e] : 0;
  const int til = (cnt + kBM - 1) / kBM;
  int ic = cnt, it = til;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nc = __shfl_up_sync(0xffffffffu, ic, o), nt = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) { ic += nc; it += nt; }
  }
  if (lane == 31) { s_wsum[0][warp] = ic; s_wsum[1][warp] = it; }
  __syncthreads();
  int pc = 0, pt = 0;
  for (int w = 0; w < warp; ++w) { pc += s_wsum[0][w]; pt += s_wsum[1][w]; }
  const int off = pc + ic - cnt, toff = pt + it - til;
  if (e < a.E) {
    s_toff[e] = toff;
    a.offsets[e] = off;
    a.offp[e] = toff * kBM;
    if (a.counts_out) a.counts_out[e] = cnt;
  }
  int tot_tiles = 0;
  for (int w = 0; w < 32; ++w) tot_tiles += s_wsum[1][w];
  const int mt_sh = (a.T + kBM - 1) / kBM;
  if (threadIdx.x == 0) {
    *s.n_items_gu = mt_sh * (s.Fs / kBN) + tot_tiles * (s.F / kBN);
    *s.n_items_dn = mt_sh * (s.H / kBN) + tot_tiles * (s.H / kBN);
  }
  __syncthreads();
  const int nt_gu = s.Fs / kBN, nt_dn = s.H / kBN;
  for (int i = threadIdx.x; i < mt_sh * nt_gu; i += blockDim.x) {
    const int mt = i / nt_gu, nt = i % nt_gu;
    s.items_gu[i] = Item{0, mt * kBM, min(kBM, a.T - mt * kBM), nt * kBN};
  }
  for (int i = threadIdx.x; i < mt_sh * nt_dn; i += blockDim.x) {
    const int mt = i / nt_dn, nt = i % nt_dn;
    s.items_dn[i] = Item{0, mt * kBM, min(kBM, a.T - mt * kBM), nt * kBN};
  }
  // routed items: tile (expert-major, padded) x N tile; the expert of a tile by binary
  // search over the tile offsets
  const int rt_gu = s.F / kBN;
  const int n_rt_tiles = tot_tiles;
  for (int i = threadIdx.x; i < n_rt_tiles * (rt_gu + nt_dn); i += blockDim.x) {
    const bool gu = i < n_rt_tiles * rt_gu;
    const int ii = gu ? i : i - n_rt_tiles * rt_gu;
    const int nt_n = gu ? rt_gu : nt_dn;
    const int tile = ii / nt_n, nt = ii % nt_n;
    int lo = 0, hi = a.E - 1;                        // last e with s_toff[e] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_toff[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    while (lo < a.E - 1 && s_cnt[lo] == 0) ++lo;     // empty experts share the offset
    const int mt = tile - s_toff[lo];
    const Item it = Item{(1 << 16) | lo, tile * kBM, min(kBM, s_cnt[lo] - mt * kBM), nt * kBN};
    if (gu) s.items_gu[mt_sh * nt_gu + ii] = it;
    else s.items_dn[mt_sh * nt_dn + ii] = it;
  }
}

// One warp per token: x[t] quantised to NVFP4 once (unit tensor scale), written to the
// shared expert's operand row t and to the token's K expert-major rows; out[t] = x[t];
// the pair order (plain and padded positions).
struct ScatterArgs {
  RouteArgs r;
  const uint16_t* x;
  int H;
  int32_t* pos_of_pair;    // pair -> padded row
  int32_t* order_pad;      // padded row -> pair
  int32_t* order_out;      // plain position -> pair (optional)
  float* out;              // [T][H]: x, to which the down GEMM adds
  uint8_t* xq_codes;  uint8_t* xq_sf;   // [Tp][H/2], MMA scale layout
  uint8_t* xp_codes;  uint8_t* xp_sf;   // [Pp][H/2], MMA scale layout
};

__global__ void __launch_bounds__(256) k_scatter_quant(ScatterArgs s) {
  const RouteArgs& a = s.r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  // rows of this token's K pairs (lanes < K), shared through the warp
  int mypos = 0;
  if (lane < a.K) {
    const int pair = t * a.K + lane;
    const int e = a.idx[pair];
    const unsigned word = a.bits[(size_t)e * a.W + (t >> 5)];
    const int rank = a.wordpre[(size_t)e * a.W + (t >> 5)] + __popc(word & ((1u << (t & 31)) - 1u));
    mypos = a.offp[e] + rank;
    s.order_pad[mypos] = pair;
    s.pos_of_pair[pair] = mypos;
    if (s.order_out) s.order_out[a.offsets[e] + rank] = pair;
  }
  // lane l takes elements [256 i + 8 l, + 8): loads, the fp32 copy and the codes of a
  // warp are contiguous; a 16-element block is a lane pair (its amax by one shuffle), the
  // four block scales of a 64-element group meet in the group's first lane.  Each block
  // is quantised by the same recipe as quant_block_unit.
  const int H = s.H, ks = H / 64;
  const uint16_t* xr = s.x + (size_t)t * H;
  int pos[FLINT_MAX_TOP_K];
#pragma unroll 1
  for (int j = 0; j < a.K; ++j) pos[j] = __shfl_sync(0xffffffffu, mypos, j);
#pragma unroll 1
  for (int e0 = 8 * lane; e0 < H; e0 += 256) {
    float f[8];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + e0));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = bf16_bits_to_f32(u[q] & 0xFFFFu);
      f[2 * q + 1] = bf16_bits_to_f32(u[q] >> 16);
    }
    float4* o = reinterpret_cast<float4*>(s.out + (size_t)t * H + e0);
    o[0] = make_float4(f[0], f[1], f[2], f[3]);
    o[1] = make_float4(f[4], f[5], f[6], f[7]);
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(f[q]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t sc = to_e4m3(__fdiv_rn(__fdiv_rn(amax, 6.0f), 1.0f));
    const float eff = e4m3_value(sc);
    uint32_t cw = 0u;
    if (eff != 0.f) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        cw |= to_e2m1x2(__fdiv_rn(f[2 * q], eff), __fdiv_rn(f[2 * q + 1], eff)) << (8 * q);
    }
    // the group's scale word: blocks 0..3 from lanes 8m, 8m + 2, 8m + 4, 8m + 6
    uint32_t sw = 0u;
#pragma unroll
    for (int b4 = 0; b4 < 4; ++b4) sw |= __shfl_sync(0xffffffffu, sc, (lane & ~7) + 2 * b4) << (8 * b4);
    const int gk = e0 >> 6;
    *reinterpret_cast<uint32_t*>(s.xq_codes + (size_t)t * (H / 2) + (e0 >> 1)) = cw;
    if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(s.xq_sf + sf_word_offset(t, gk, ks)) = sw;
#pragma unroll 1
    for (int j = 0; j < a.K; ++j) {
      *reinterpret_cast<uint32_t*>(s.xp_codes + (size_t)pos[j] * (H / 2) + (e0 >> 1)) = cw;
      if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(s.xp_sf + sf_word_offset(pos[j], gk, ks)) = sw;
    }
  }
}

// ---------------------------------------------------------------- MMA scale copies
// scales [m][rows][cols/16] -> [m][rows/128][cols/64][512] (see flint.h)
__global__ void k_mma_scales(const uint8_t* __restrict__ scales, int rows, int cols,
                             uint8_t* __restrict__ out) {
  const int m = blockIdx.y;
  const int ks = cols / 64;
  const int64_t n = (int64_t)rows * ks;
  const uint8_t* sm = scales + (size_t)m * rows * (cols / 16);
  uint8_t* om = out + (size_t)m * rows * (cols / 16);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / ks), k = (int)(i % ks);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(sm + (size_t)r * (cols / 16) + 4 * k);
    *reinterpret_cast<uint32_t*>(om + sf_word_offset(r, k, ks)) = v;
  }
}

// ---------------------------------------------------------------- host side
struct WsLayout {
  size_t logits, idx, w, bits, wordpre, counts, offsets, offp, order, pos, xq_c, xq_s, xp_c, xp_s, hs_c,
      hs_s, hq_c, hq_s, items_gu, items_dn, nitems, total;
};

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// Rows of the padded expert-major operands: every expert's rows start on a 128-row tile.
static size_t padded_rows(int T, int K, int E) {
  const size_t P = (size_t)T * K;
  const size_t touched = P < (size_t)E ? P : (size_t)E;
  return (P + touched * (kBM - 1) + kBM - 1) / kBM * kBM;
}

static WsLayout ws_layout(int H, int E, int K, int F, int Fs, int T) {
  WsLayout L;
  const size_t P = (size_t)T * K, Pp = padded_rows(T, K, E), W = (T + 31) / 32;
  const size_t Tp = (T + kBM - 1) / kBM * kBM;
  const size_t mt_sh = Tp / kBM, mt_rt = Pp / kBM;
  size_t o = 0;
  L.logits = o;   o += a256(sizeof(float) * kRSplit * T * E);
  L.idx = o;      o += a256(sizeof(int) * P);
  L.w = o;        o += a256(sizeof(float) * P);
  L.bits = o;     o += a256(sizeof(unsigned) * E * W);
  L.wordpre = o;  o += a256(sizeof(int) * E * W);
  L.counts = o;   o += a256(sizeof(int) * E);
  L.offsets = o;  o += a256(sizeof(int) * E);
  L.offp = o;     o += a256(sizeof(int) * E);
  L.order = o;    o += a256(sizeof(int) * Pp);
  L.pos = o;      o += a256(sizeof(int) * P);
  L.xq_c = o;     o += a256(Tp * H / 2);
  L.xq_s = o;     o += a256(Tp * H / 16);
  L.xp_c = o;     o += a256(Pp * H / 2);
  L.xp_s = o;     o += a256(Pp * H / 16);
  L.hs_c = o;     o += a256(Tp * Fs / 2);
  L.hs_s = o;     o += a256(Tp * Fs / 16);
  L.hq_c = o;     o += a256(Pp * F / 2);
  L.hq_s = o;     o += a256(Pp * F / 16);
  L.items_gu = o; o += a256(sizeof(Item) * (mt_sh * (Fs / kBN) + mt_rt * (F / kBN)));
  L.items_dn = o; o += a256(sizeof(Item) * (mt_sh + mt_rt) * (H / kBN));
  L.nitems = o;   o += 256;
  L.total = o;
  return L;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool encode_init() {
  if (g_encode) return true;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2D byte tensor [rows][row_bytes], box {128 bytes, box_rows}, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pf

size_t prefill_workspace_bytes(int H, int E, int K, int F, int Fs, int T) {
  return pf::ws_layout(H, E, K, F, Fs, T).total;
}

bool prefill_shape_ok(int H, int E, int K, int F, int Fs) {
  return H % 256 == 0 && F % 256 == 0 && Fs % 256 == 0 && E % 16 == 0 && E <= 256 && K <= FLINT_MAX_TOP_K &&
         H <= 8192 && F <= 8192 && Fs <= 8192;
}

cudaError_t launch_mma_scales(const uint8_t* scales, int n_mat, int rows, int cols, uint8_t* out,
                              cudaStream_t st) {
  const int64_t n = (int64_t)rows * (cols / 64);
  int g = (int)((n + 255) / 256);
  if (g > 4096) g = 4096;
  pf::k_mma_scales<<<dim3(g, n_mat), 256, 0, st>>>(scales, rows, cols, out);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, void* ws, cudaStream_t st) {
  using namespace pf;
  if (!encode_init()) return cudaErrorNotSupported;
  const int H = a.H, E = a.E, K = a.K, F = a.F, Fs = a.Fs, T = a.T;
  const size_t Pp = padded_rows(T, K, E), Tp = (T + kBM - 1) / kBM * kBM;
  const WsLayout L = ws_layout(H, E, K, F, Fs, T);
  char* b = static_cast<char*>(ws);
  auto at = [&](size_t off) { return b + off; };
  RouteArgs r;
  r.T = T; r.E = E; r.K = K; r.W = (T + 31) / 32;
  r.part = reinterpret_cast<float*>(at(L.logits));
  r.bias = a.router_bias;
  r.sigmoid = a.router_score == FLINT_ROUTER_SIGMOID;
  r.idx = reinterpret_cast<int32_t*>(at(L.idx));
  r.w = reinterpret_cast<float*>(at(L.w));
  r.idx_out = a.idx_out; r.w_out = a.w_out;
  r.bits = reinterpret_cast<unsigned*>(at(L.bits));
  r.wordpre = reinterpret_cast<int*>(at(L.wordpre));
  r.counts = reinterpret_cast<int*>(at(L.counts));
  r.offsets = reinterpret_cast<int*>(at(L.offsets));
  r.offp = reinterpret_cast<int*>(at(L.offp));
  r.counts_out = a.counts_out;
  cudaError_t e = cudaMemsetAsync(r.bits, 0, sizeof(unsigned) * E * r.W, st);
  if (e != cudaSuccess) return e;

  // 1 router GEMM (partial logits over kRSplit K ranges)
  RouterArgs ra;
  memset(&ra, 0, sizeof(ra));
  ra.part = reinterpret_cast<float*>(at(L.logits)); ra.T = T; ra.E = E; ra.H = H;
  ra.wait_ns = a.wait_ns;
  if (!make_map(&ra.mapX, a.x, T, (uint64_t)H * 2, kBM) || !make_map(&ra.mapW, a.router_w, E, (uint64_t)H * 2, E))
    return cudaErrorInvalidValue;
  const int smem_r = kRStages * (16384 + 256 * 128) + 1024;
  e = cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_r);
  if (e != cudaSuccess) return e;
  k_router_gemm<<<dim3((T + kBM - 1) / kBM, kRSplit), kRThreads, smem_r, st>>>(ra);

  // 2 top-k + bitmaps, 3 scan + item lists, 4 scatter + quantise (+ out = x)
  k_topk<<<(T + 7) / 8, 256, 0, st>>>(r);
  ScanArgs sc;
  sc.r = r;
  sc.items_gu = reinterpret_cast<Item*>(at(L.items_gu));
  sc.items_dn = reinterpret_cast<Item*>(at(L.items_dn));
  sc.n_items_gu = reinterpret_cast<int*>(at(L.nitems));
  sc.n_items_dn = reinterpret_cast<int*>(at(L.nitems)) + 1;
  sc.H = H; sc.F = F; sc.Fs = Fs;
  k_expert_prefix<<<(E + 7) / 8, 256, 0, st>>>(r);
  k_scan<<<1, 1024, 0, st>>>(sc);
  ScatterArgs sa;
  sa.r = r; sa.x = a.x; sa.H = H; sa.out = a.out;
  sa.order_pad = reinterpret_cast<int32_t*>(at(L.order));
  sa.pos_of_pair = reinterpret_cast<int32_t*>(at(L.pos));
  sa.order_out = a.order_out;
  sa.xq_codes = reinterpret_cast<uint8_t*>(at(L.xq_c)); sa.xq_sf = reinterpret_cast<uint8_t*>(at(L.xq_s));
  sa.xp_codes = reinterpret_cast<uint8_t*>(at(L.xp_c)); sa.xp_sf = reinterpret_cast<uint8_t*>(at(L.xp_s));
  k_scatter_quant<<<(T + 7) / 8, 256, 0, st>>>(sa);

  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  // 5 gate/up grouped GEMM
  GemmArgs gu;
  memset(&gu, 0, sizeof(gu));
  bool ok = make_map(&gu.mapA[0], sa.xq_codes, Tp, H / 2, kBM) && make_map(&gu.mapA[1], sa.xp_codes, Pp, H / 2, kBM) &&
            make_map(&gu.mapB[0], a.sh_gate.codes, Fs, H / 2, kBN) && make_map(&gu.mapB[1], a.sh_up.codes, Fs, H / 2, kBN) &&
            make_map(&gu.mapB[2], a.gate.codes, (uint64_t)E * F, H / 2, kBN) &&
            make_map(&gu.mapB[3], a.up.codes, (uint64_t)E * F, H / 2, kBN);
  if (!ok) return cudaErrorInvalidValue;
  gu.sfA[0] = sa.xq_sf; gu.sfA[1] = sa.xp_sf;
  gu.sfB[0] = a.sf[3]; gu.sfB[1] = a.sf[4]; gu.sfB[2] = a.sf[0]; gu.sfB[3] = a.sf[1];
  gu.Kel[0] = H; gu.Kel[1] = H;
  gu.rowsB[0] = Fs; gu.rowsB[1] = F;
  gu.items = sc.items_gu; gu.n_items = sc.n_items_gu;
  gu.tscA[0] = a.sh_gate.tsc; gu.tscA[1] = a.gate.tsc; gu.tscB[0] = a.sh_up.tsc; gu.tscB[1] = a.up.tsc;
  gu.hcodes[0] = reinterpret_cast<uint8_t*>(at(L.hs_c)); gu.hsf[0] = reinterpret_cast<uint8_t*>(at(L.hs_s));
  gu.hcodes[1] = reinterpret_cast<uint8_t*>(at(L.hq_c)); gu.hsf[1] = reinterpret_cast<uint8_t*>(at(L.hq_s));
  gu.Fout[0] = Fs; gu.Fout[1] = F;
  gu.H = H; gu.K = K;
  gu.wait_ns = a.wait_ns;
  gu.hold = a.hold;
  e = cudaFuncSetAttribute(k_gemm_fp4<kGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kGateUp>::smem);
  if (e != cudaSuccess) return e;
  k_gemm_fp4<kGateUp><<<sms, kGThreads, Cfg<kGateUp>::smem, st>>>(gu);

  // 6 down grouped GEMM over the shared and routed tiles: out += rows (bulk reduce-add)
  GemmArgs dn;
  memset(&dn, 0, sizeof(dn));
  ok = make_map(&dn.mapA[0], gu.hcodes[0], Tp, Fs / 2, kBM) && make_map(&dn.mapA[1], gu.hcodes[1], Pp, F / 2, kBM) &&
       make_map(&dn.mapB[0], a.sh_down.codes, H, Fs / 2, kBN) &&
       make_map(&dn.mapB[2], a.down.codes, (uint64_t)E * H, F / 2, kBN);
  if (!ok) return cudaErrorInvalidValue;
  dn.sfA[0] = gu.hsf[0]; dn.sfA[1] = gu.hsf[1];
  dn.sfB[0] = a.sf[5]; dn.sfB[2] = a.sf[2];
  dn.Kel[0] = Fs; dn.Kel[1] = F;
  dn.rowsB[0] = H; dn.rowsB[1] = H;
  dn.items = sc.items_dn; dn.n_items = sc.n_items_dn;
  dn.tscA[0] = a.sh_down.tsc; dn.tscA[1] = a.down.tsc;
  dn.out = a.out;
  dn.order = sa.order_pad; dn.wpair = r.w;
  dn.H = H; dn.K = K;
  dn.wait_ns = a.wait_ns;
  e = cudaFuncSetAttribute(k_gemm_fp4<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kDown>::smem);
  if (e != cudaSuccess) return e;
  k_gemm_fp4<kDown><<<sms, kGThreads, Cfg<kDown>::smem, st>>>(dn);

  return cudaGetLastError();
}

}  // namespace flint
