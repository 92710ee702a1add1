// prefill.cu -- one Flint MoE layer over T prompt tokens ("Flint-40B-A2B: AI-Built MoE
// Coding Model Hits 125 tok/s on MacBook Pro", section "Custom Inference Kernels": prompt
// processing), as a token-permuted grouped GEMM on block-scaled FP4 tensor cores.
//
//   1 router      logits[T, E] = x Wr^T (+ bias): tcgen05 kind::f16 (bf16 in, fp32 acc)
//   2 top-k       per token (one warp): softmax top-k, renormalised weights; per-expert
//                 token bitmaps
//   3 scan        per-expert counts and exclusive offsets (expert-major order, tokens
//                 ascending within an expert), and the device-side tile lists
//   4 scatter     every (token, slot) pair gets its position; its x row is quantised
//                 to NVFP4 (unit tensor scale) into the permuted operand Xp; slot 0
//                 also writes the unpermuted Xq used by the shared expert
//   5 gate/up     grouped GEMM, tcgen05 kind::mxf4nvf4 (E2M1 x E2M1, E4M3 scale per
//                 16): per 128-row tile of one expert, the gate and up tiles accumulate
//                 in TMEM; the epilogue applies the tensor scales, SwiGLU, and
//                 quantises h to NVFP4 (unit tensor scale)
//   6 down        grouped GEMM as 5; the shared expert writes out = x + y, then the
//                 routed tiles add w_pair * y into out (red.global.add.v4.f32): the
//                 un-permuting combine
//
// GEMM CTAs are warp-specialised (8 warps): warp 0 issues TMA loads of the operand
// tiles (128-byte swizzle), warp 1 gathers the block scales into the layout the MMA
// expects, warp 2 allocates TMEM and issues tcgen05.cp / tcgen05.mma, warps 4-7 read the
// accumulator back (tcgen05.ld) for the epilogue.  Stages are handed over with mbarriers
// whose waits are bounded: on expiry the CTA records FLINT_ERR_TIMEOUT and unwinds.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace flint {
namespace pf {

constexpr int kBM = 128;          // tokens per tile (TMEM lanes)
constexpr int kBN = 128;          // output columns per tile
constexpr int kStages = 3;
constexpr int kGThreads = 256;    // 8 warps
constexpr int kWarpTMA = 0, kWarpScale = 1, kWarpMMA = 2, kWarpEpi0 = 4;

struct Item {
  int kind;     // 0 shared expert, 1 routed expert
  int expert;
  int row0;     // first A row of the tile
  int rows;     // valid rows (<= kBM)
  int n0;       // first output column
};

enum Mode { kGateUp = 1, kDown = 2, kRouter = 3 };

struct GemmArgs {
  CUtensorMap mapA[2];          // A operand: [0] shared-expert rows, [1] expert-major rows
  CUtensorMap mapB[4];          // gate/up: sh_gate, sh_up, gate, up; down: sh_down, -, down, -
  const uint8_t* sclA[2];       // A block scales, row-major [rows][K/16]
  int rowsA[2];
  const uint8_t* sclB[4];       // weight block scales, row-major
  int Kel[2];                   // K in elements: shared / routed
  int rowsB[2];                 // rows of one weight matrix: shared / routed
  const Item* items;
  const int* n_items;           // device count (total items)
  int item_begin;               // first item this launch processes
  int item_end_host;            // upper bound from the host (-1: use *n_items)
  // epilogues
  const float* tscA[2];         // gate / sh_gate (or down / sh_down) tensor scales
  const float* tscB[2];         // up / sh_up tensor scales
  uint8_t* hcodes[2];           // gate/up output: [0] shared h, [1] routed h
  uint8_t* hscales[2];
  int Fout[2];
  const uint16_t* x;            // [T][H] bf16
  float* out;                   // [T][H]
  const int32_t* order;         // position -> pair id
  const float* wpair;           // [T*K]
  int H, K, T, E;
  const float* bias;            // router
  float* logits;                // router output [T][E]
  int nE;                       // router N (E rounded up to 16)
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
// Bounded parity wait; false on expiry (FLINT_ERR_TIMEOUT recorded, *abort set).
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t parity, volatile int* abort) {
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
      else if (now - t0 > kWaitLimitNs) {
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
// 32 lanes x N consecutive fp32 columns; thread (lane) gets its row.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t t, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(t));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void red_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// 16 fp32 values -> one NVFP4 block with unit tensor scale (the quantiser's recipe).
__device__ __forceinline__ void quant_block_unit(const float (&v)[16], uint2& codes, uint8_t& scale) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const float t = __fdiv_rn(__fdiv_rn(amax, 6.0f), 1.0f);
  const uint32_t s = to_e4m3(t);
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
  scale = (uint8_t)s;
}

// ---------------------------------------------------------------- grouped FP4 GEMM
// Shared-memory stage: A tile (16 KB), B tiles (16 KB each), scale chunks.
template <int MODE>
struct StageLayout {
  static constexpr int kB = MODE == kGateUp ? 2 : 1;
  static constexpr int a = 0;
  static constexpr int b = 16384;
  static constexpr int sfa = b + kB * 16384;            // 4 chunks of 512 B
  static constexpr int sfb = sfa + 2048;                // kB x 4 chunks of 512 B
  static constexpr int bytes = sfb + kB * 2048;
  static constexpr int stride = (bytes + 1023) / 1024 * 1024;
};

template <int MODE>
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_fp4(const __grid_constant__ GemmArgs g) {
  using SL = StageLayout<MODE>;
  constexpr int kB = SL::kB;
  constexpr uint32_t kTmemCols = MODE == kGateUp ? 512 : 256;
  constexpr int kDCols = kB * kBN;                        // accumulator columns
  constexpr int kSfPerStep = 4 + 4 * kB;                  // TMEM columns of scales per K=64 step
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], accf, acce;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mb_init(&full[s], 1 + 32); mb_init(&empty[s], 1); }
    mb_init(&accf, 1);
    mb_init(&acce, 4);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(sh(&tmem_base)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int n_items = g.item_end_host >= 0 ? g.item_end_host : __ldcg(g.n_items);
  const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

  if (warp == kWarpTMA && lane == 0) {
    uint32_t it = 0;
    for (int i = g.item_begin + blockIdx.x; i < n_items && !abort_flag; i += gridDim.x) {
      const Item item = g.items[i];
      const int kt_n = g.Kel[item.kind] / 256;
      for (int kt = 0; kt < kt_n; ++kt, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mb_wait(&empty[s], ((it / kStages) - 1) & 1, &abort_flag)) break;
        uint8_t* st = smem + s * SL::stride;
        mb_expect(&full[s], 16384 * (1 + kB));
        tma2d(st + SL::a, &g.mapA[item.kind], kt * 128, item.row0, &full[s]);
        const int brow = item.expert * g.rowsB[item.kind] + item.n0;
        tma2d(st + SL::b, &g.mapB[2 * item.kind], kt * 128, brow, &full[s]);
        if (kB == 2) tma2d(st + SL::b + 16384, &g.mapB[2 * item.kind + 1], kt * 128, brow, &full[s]);
      }
    }
  } else if (warp == kWarpScale) {
    uint32_t it = 0;
    for (int i = g.item_begin + blockIdx.x; i < n_items && !abort_flag; i += gridDim.x) {
      const Item item = g.items[i];
      const int K = g.Kel[item.kind];
      const int kt_n = K / 256;
      const int ldk = K / 16;
      for (int kt = 0; kt < kt_n; ++kt, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mb_wait(&empty[s], ((it / kStages) - 1) & 1, &abort_flag)) break;
        uint8_t* st = smem + s * SL::stride;
        // A scales: 128 rows, 16 bytes (blocks 16 kt .. 16 kt + 15) per row
        for (int r = lane; r < kBM; r += 32) {
          const int row = item.row0 + r;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < g.rowsA[item.kind])
            v = __ldg(reinterpret_cast<const uint4*>(g.sclA[item.kind] + (size_t)row * ldk + kt * 16));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
          uint8_t* base = st + SL::sfa + 16 * (r & 31) + 4 * (r >> 5);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) *reinterpret_cast<uint32_t*>(base + kk * 512) = w4[kk];
        }
        // B scales: kB matrices x 128 rows
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const uint8_t* src = g.sclB[2 * item.kind + b];
          const size_t row0 = (size_t)item.expert * g.rowsB[item.kind] + item.n0;
          for (int r = lane; r < kBN; r += 32) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + (row0 + r) * ldk + kt * 16));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            uint8_t* base = st + SL::sfb + b * 2048 + 16 * (r & 31) + 4 * (r >> 5);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) *reinterpret_cast<uint32_t*>(base + kk * 512) = w4[kk];
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mb_arrive(&full[s]);
      }
    }
  } else if (warp == kWarpMMA && lane == 0) {
    uint32_t it = 0, done = 0;
    for (int i = g.item_begin + blockIdx.x; i < n_items && !abort_flag; i += gridDim.x, ++done) {
      const Item item = g.items[i];
      const int kt_n = g.Kel[item.kind] / 256;
      if (done > 0 && !mb_wait(&acce, (done - 1) & 1, &abort_flag)) break;
      tc_fence_after();
      bool ok = true;
      for (int kt = 0; kt < kt_n; ++kt, ++it) {
        const int s = it % kStages;
        if (!mb_wait(&full[s], (it / kStages) & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint8_t* st = smem + s * SL::stride;
        const uint32_t sf0 = tmem + kDCols + (uint32_t)(s * 4 * kSfPerStep);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t sfs = sf0 + kk * kSfPerStep;
          tc_cp_sf(sfs, sf_desc(sh(st + SL::sfa + kk * 512)));
#pragma unroll
          for (int b = 0; b < kB; ++b) tc_cp_sf(sfs + 4 + 4 * b, sf_desc(sh(st + SL::sfb + b * 2048 + kk * 512)));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t sfs = sf0 + kk * kSfPerStep;
          const uint64_t ad = umma_desc_sw128(sh(st + SL::a) + kk * 32);
          const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
          for (int b = 0; b < kB; ++b) {
            const uint64_t bd = umma_desc_sw128(sh(st + SL::b + b * 16384) + kk * 32);
            mma_fp4(tmem + b * kBN, ad, bd, idesc, acc, sfs, sfs + 4 + 4 * b);
          }
        }
        tc_commit(&empty[s]);
      }
      if (!ok) break;
      tc_commit(&accf);
    }
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;                                 // TMEM lane quarter
    const int r = q * 32 + lane;                            // tile row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t done = 0;
    for (int i = g.item_begin + blockIdx.x; i < n_items && !abort_flag; i += gridDim.x, ++done) {
      const Item item = g.items[i];
      if (!mb_wait(&accf, done & 1, &abort_flag)) break;
      tc_fence_after();
      const bool valid = r < item.rows;
      const int arow = item.row0 + r;
      if (MODE == kGateUp) {
        const float tg = g.tscA[item.kind][item.kind ? item.expert : 0];
        const float tu = g.tscB[item.kind][item.kind ? item.expert : 0];
        const int F = g.Fout[item.kind];
        uint8_t* hc = g.hcodes[item.kind] + (size_t)arow * (F / 2);
        uint8_t* hs = g.hscales[item.kind] + (size_t)arow * (F / 16);
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 16) {
          float gv[16], uv[16], hv[16];
          tmem_ld<16>(lane_base + c0, gv);
          tmem_ld<16>(lane_base + kBN + c0, uv);
#pragma unroll
          for (int j = 0; j < 16; ++j) hv[j] = silu(gv[j] * tg) * (uv[j] * tu);
          uint2 cw;
          uint8_t sc;
          quant_block_unit(hv, cw, sc);
          if (valid) {
            *reinterpret_cast<uint2*>(hc + (item.n0 + c0) / 2) = cw;
            hs[(item.n0 + c0) / 16] = sc;
          }
        }
      } else {  // down
        const float td = g.tscA[item.kind][item.kind ? item.expert : 0];
        const int H = g.H;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 16) {
          float yv[16];
          tmem_ld<16>(lane_base + c0, yv);
          if (!valid) continue;
          if (item.kind == 0) {
            const int t = arow;
            const uint16_t* xr = g.x + (size_t)t * H + item.n0 + c0;
            float* o = g.out + (size_t)t * H + item.n0 + c0;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const uint2 xb = *reinterpret_cast<const uint2*>(xr + j);
              float4 v;
              v.x = bf16_bits_to_f32(xb.x & 0xFFFFu) + yv[j] * td;
              v.y = bf16_bits_to_f32(xb.x >> 16) + yv[j + 1] * td;
              v.z = bf16_bits_to_f32(xb.y & 0xFFFFu) + yv[j + 2] * td;
              v.w = bf16_bits_to_f32(xb.y >> 16) + yv[j + 3] * td;
              *reinterpret_cast<float4*>(o + j) = v;
            }
          } else {
            const int pair = g.order[arow];
            const int t = pair / g.K;
            const float w = g.wpair[pair] * td;
            float* o = g.out + (size_t)t * H + item.n0 + c0;
#pragma unroll
            for (int j = 0; j < 16; j += 4) red_v4(o + j, yv[j] * w, yv[j + 1] * w, yv[j + 2] * w, yv[j + 3] * w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mb_arrive(&acce);
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
      mb_wait(&drain, 0, &no_abort);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols));
  }
}

// ---------------------------------------------------------------- router GEMM (bf16)
// logits[t][e] = x[t] . Wr[e] (+ bias[e]); A = x rows (TMA, 64 bf16 = 128 B per K-tile),
// B = Wr rows (N = nE <= 256), tcgen05 kind::f16 with K = 16 per instruction.
constexpr int kRStages = 4;

__global__ void __launch_bounds__(kGThreads, 1) k_router_gemm(const __grid_constant__ GemmArgs g) {
  constexpr int kStageBytes = 16384 + 32768;
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
  const int row0 = blockIdx.x * kBM;
  const int kt_n = g.H / 64;
  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(g.nE >> 3) << 17) |
                         ((uint32_t)(kBM >> 4) << 24);
  if (warp == kWarpTMA && lane == 0) {
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % kRStages;
      if (kt >= kRStages && !mb_wait(&empty[s], ((kt / kRStages) - 1) & 1, &abort_flag)) break;
      uint8_t* st = smem + s * kStageBytes;
      mb_expect(&full[s], 16384 + 128 * g.nE);
      tma2d(st, &g.mapA[0], kt * 128, row0, &full[s]);
      tma2d(st + 16384, &g.mapB[0], kt * 128, 0, &full[s]);
    }
  } else if (warp == kWarpMMA && lane == 0) {
    bool ok = true;
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % kRStages;
      if (!mb_wait(&full[s], (kt / kRStages) & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint8_t* st = smem + s * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem, umma_desc_sw128(sh(st) + kk * 32), umma_desc_sw128(sh(st + 16384) + kk * 32), idesc,
                 (kt > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    if (ok) tc_commit(&accf);
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int t = row0 + r;
    if (mb_wait(&accf, 0, &abort_flag)) {
      tc_fence_after();
      for (int c0 = 0; c0 < g.nE; c0 += 16) {
        float v[16];
        tmem_ld<16>(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        if (t < g.T)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < g.E) g.logits[(size_t)t * g.E + c0 + j] = v[j] + (g.bias ? g.bias[c0 + j] : 0.f);
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
      mb_wait(&drain, 0, &no_abort);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(256));
  }
}

// ---------------------------------------------------------------- routing bookkeeping
struct RouteArgs {
  int T, E, K, W;          // W = words per expert bitmap = ceil(T/32)
  const float* logits;     // [T][E]
  int32_t* idx;            // [T][K]
  float* w;                // [T][K]
  int32_t* idx_out;
  float* w_out;
  unsigned* bits;          // [E][W]
  int* wordpre;            // [E][W]
  int* counts;             // [E]
  int* offsets;            // [E]
  int32_t* counts_out;
};

// One warp per token: top-k (the decode path's warp top-k) and the expert bitmaps.
__global__ void __launch_bounds__(256) k_topk(RouteArgs a) {
  __shared__ int s_sel[8][FLINT_MAX_TOP_K];
  __shared__ float s_w[8][FLINT_MAX_TOP_K];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  const float* lg = a.logits + (size_t)t * a.E;
  topk_dispatch(lg, a.E, a.K, s_sel[warp], s_w[warp]);
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

// One CTA: per-expert word prefix counts, expert offsets, and the tile lists.
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
  __shared__ int s_tiles[FLINT_MAX_EXPERTS];
  __shared__ int s_tile_off[FLINT_MAX_EXPERTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = warp; e < a.E; e += 32) {
    int run = 0;
    for (int base = 0; base < a.W; base += 32) {
      const int w = base + lane;
      const int v = w < a.W ? __popc(a.bits[(size_t)e * a.W + w]) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (w < a.W) a.wordpre[(size_t)e * a.W + w] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      a.counts[e] = run;
      if (a.counts_out) a.counts_out[e] = run;
      s_tiles[e] = (run + kBM - 1) / kBM;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, toff = 0;
    for (int e = 0; e < a.E; ++e) {
      a.offsets[e] = off;
      off += a.counts[e];
      s_tile_off[e] = toff;
      toff += s_tiles[e];
    }
    const int mt_sh = (a.T + kBM - 1) / kBM;
    *s.n_items_gu = mt_sh * (s.Fs / kBN) + toff * (s.F / kBN);
    *s.n_items_dn = mt_sh * (s.H / kBN) + toff * (s.H / kBN);
  }
  __syncthreads();
  const int mt_sh = (a.T + kBM - 1) / kBM;
  // shared-expert items
  for (int i = threadIdx.x; i < mt_sh * (s.Fs / kBN); i += blockDim.x) {
    const int mt = i / (s.Fs / kBN), nt = i % (s.Fs / kBN);
    s.items_gu[i] = Item{0, 0, mt * kBM, min(kBM, a.T - mt * kBM), nt * kBN};
  }
  for (int i = threadIdx.x; i < mt_sh * (s.H / kBN); i += blockDim.x) {
    const int mt = i / (s.H / kBN), nt = i % (s.H / kBN);
    s.items_dn[i] = Item{0, 0, mt * kBM, min(kBM, a.T - mt * kBM), nt * kBN};
  }
  // routed items, expert by expert
  const int base_gu = mt_sh * (s.Fs / kBN), base_dn = mt_sh * (s.H / kBN);
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const int cnt = a.counts[e], off = a.offsets[e];
    for (int mt = 0; mt < s_tiles[e]; ++mt) {
      const int rows = min(kBM, cnt - mt * kBM);
      for (int nt = 0; nt < s.F / kBN; ++nt)
        s.items_gu[base_gu + (s_tile_off[e] + mt) * (s.F / kBN) + nt] = Item{1, e, off + mt * kBM, rows, nt * kBN};
      for (int nt = 0; nt < s.H / kBN; ++nt)
        s.items_dn[base_dn + (s_tile_off[e] + mt) * (s.H / kBN) + nt] = Item{1, e, off + mt * kBM, rows, nt * kBN};
    }
  }
}

// One warp per (token, slot) pair: its expert-major position, and its x row quantised to
// NVFP4 with unit tensor scale (slot 0 also writes the unpermuted copy).
struct ScatterArgs {
  RouteArgs r;
  const uint16_t* x;
  int H;
  int32_t* pos_of_pair;   // [T*K]
  int32_t* order;         // [P]
  int32_t* order_out;
  uint8_t* xq_codes;  uint8_t* xq_scales;   // [T][H/2], [T][H/16]
  uint8_t* xp_codes;  uint8_t* xp_scales;   // [P+128][H/2], [P+128][H/16]
};

__global__ void __launch_bounds__(256) k_scatter_quant(ScatterArgs s) {
  const RouteArgs& a = s.r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + warp;
  if (pair >= a.T * a.K) return;
  const int t = pair / a.K, j = pair % a.K;
  const int e = a.idx[pair];
  const unsigned word = a.bits[(size_t)e * a.W + (t >> 5)];
  const int pos = a.offsets[e] + a.wordpre[(size_t)e * a.W + (t >> 5)] + __popc(word & ((1u << (t & 31)) - 1u));
  if (lane == 0) {
    s.pos_of_pair[pair] = pos;
    s.order[pos] = pair;
    if (s.order_out) s.order_out[pos] = pair;
  }
  const int H = s.H;
  const uint16_t* xr = s.x + (size_t)t * H;
  for (int b = lane; b < H / 16; b += 32) {
    const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(xr + 16 * b + 8));
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) { f[2 * q] = bf16_bits_to_f32(u[q] & 0xFFFFu); f[2 * q + 1] = bf16_bits_to_f32(u[q] >> 16); }
    uint2 cw;
    uint8_t sc;
    quant_block_unit(f, cw, sc);
    *reinterpret_cast<uint2*>(s.xp_codes + (size_t)pos * (H / 2) + 8 * b) = cw;
    s.xp_scales[(size_t)pos * (H / 16) + b] = sc;
    if (j == 0) {
      *reinterpret_cast<uint2*>(s.xq_codes + (size_t)t * (H / 2) + 8 * b) = cw;
      s.xq_scales[(size_t)t * (H / 16) + b] = sc;
    }
  }
}

// ---------------------------------------------------------------- host side
struct WsLayout {
  size_t logits, idx, w, bits, wordpre, counts, offsets, pos, order, xq_c, xq_s, xp_c, xp_s, hs_c,
      hs_s, hq_c, hq_s, items_gu, items_dn, nitems, total;
};

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

static WsLayout ws_layout(int H, int E, int K, int F, int Fs, int T) {
  WsLayout L;
  const size_t P = (size_t)T * K, PP = P + kBM, W = (T + 31) / 32;
  const size_t mt_sh = (T + kBM - 1) / kBM, mt_rt = P / kBM + E;
  size_t o = 0;
  L.logits = o;   o += a256(sizeof(float) * T * E);
  L.idx = o;      o += a256(sizeof(int) * P);
  L.w = o;        o += a256(sizeof(float) * P);
  L.bits = o;     o += a256(sizeof(unsigned) * E * W);
  L.wordpre = o;  o += a256(sizeof(int) * E * W);
  L.counts = o;   o += a256(sizeof(int) * E);
  L.offsets = o;  o += a256(sizeof(int) * E);
  L.pos = o;      o += a256(sizeof(int) * P);
  L.order = o;    o += a256(sizeof(int) * PP);
  L.xq_c = o;     o += a256((size_t)T * H / 2);
  L.xq_s = o;     o += a256((size_t)T * H / 16);
  L.xp_c = o;     o += a256(PP * H / 2);
  L.xp_s = o;     o += a256(PP * H / 16);
  L.hs_c = o;     o += a256((size_t)T * Fs / 2);
  L.hs_s = o;     o += a256((size_t)T * Fs / 16);
  L.hq_c = o;     o += a256(PP * F / 2);
  L.hq_s = o;     o += a256(PP * F / 16);
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

cudaError_t launch_prefill(const PrefillArgs& a, void* ws, cudaStream_t st) {
  using namespace pf;
  if (!encode_init()) return cudaErrorNotSupported;
  const int H = a.H, E = a.E, K = a.K, F = a.F, Fs = a.Fs, T = a.T;
  const size_t P = (size_t)T * K, PP = P + kBM;
  const WsLayout L = ws_layout(H, E, K, F, Fs, T);
  char* b = static_cast<char*>(ws);
  auto at = [&](size_t off) { return b + off; };
  RouteArgs r;
  r.T = T; r.E = E; r.K = K; r.W = (T + 31) / 32;
  r.logits = reinterpret_cast<float*>(at(L.logits));
  r.idx = reinterpret_cast<int32_t*>(at(L.idx));
  r.w = reinterpret_cast<float*>(at(L.w));
  r.idx_out = a.idx_out; r.w_out = a.w_out;
  r.bits = reinterpret_cast<unsigned*>(at(L.bits));
  r.wordpre = reinterpret_cast<int*>(at(L.wordpre));
  r.counts = reinterpret_cast<int*>(at(L.counts));
  r.offsets = reinterpret_cast<int*>(at(L.offsets));
  r.counts_out = a.counts_out;
  cudaError_t e = cudaMemsetAsync(r.bits, 0, sizeof(unsigned) * E * r.W, st);
  if (e != cudaSuccess) return e;

  // 1 router GEMM
  GemmArgs gr;
  memset(&gr, 0, sizeof(gr));
  gr.H = H; gr.T = T; gr.E = E; gr.nE = E; gr.bias = a.router_bias; gr.logits = const_cast<float*>(r.logits);
  if (!make_map(&gr.mapA[0], a.x, T, (uint64_t)H * 2, 128) || !make_map(&gr.mapB[0], a.router_w, E, (uint64_t)H * 2, E))
    return cudaErrorInvalidValue;
  const int smem_r = kRStages * (16384 + 32768) + 1024;
  e = cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_r);
  if (e != cudaSuccess) return e;
  k_router_gemm<<<(T + kBM - 1) / kBM, kGThreads, smem_r, st>>>(gr);

  // 2 top-k + bitmaps, 3 scan + tile lists, 4 scatter + quantise
  k_topk<<<(T + 7) / 8, 256, 0, st>>>(r);
  ScanArgs sc;
  sc.r = r;
  sc.items_gu = reinterpret_cast<Item*>(at(L.items_gu));
  sc.items_dn = reinterpret_cast<Item*>(at(L.items_dn));
  sc.n_items_gu = reinterpret_cast<int*>(at(L.nitems));
  sc.n_items_dn = reinterpret_cast<int*>(at(L.nitems)) + 1;
  sc.H = H; sc.F = F; sc.Fs = Fs;
  k_scan<<<1, 1024, 0, st>>>(sc);
  ScatterArgs sa;
  sa.r = r; sa.x = a.x; sa.H = H;
  sa.pos_of_pair = reinterpret_cast<int32_t*>(at(L.pos));
  sa.order = reinterpret_cast<int32_t*>(at(L.order));
  sa.order_out = a.order_out;
  sa.xq_codes = reinterpret_cast<uint8_t*>(at(L.xq_c)); sa.xq_scales = reinterpret_cast<uint8_t*>(at(L.xq_s));
  sa.xp_codes = reinterpret_cast<uint8_t*>(at(L.xp_c)); sa.xp_scales = reinterpret_cast<uint8_t*>(at(L.xp_s));
  k_scatter_quant<<<(int)((P + 7) / 8), 256, 0, st>>>(sa);

  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  // 5 gate/up grouped GEMM
  GemmArgs gu;
  memset(&gu, 0, sizeof(gu));
  bool ok = make_map(&gu.mapA[0], sa.xq_codes, T, H / 2, 128) && make_map(&gu.mapA[1], sa.xp_codes, PP, H / 2, 128) &&
            make_map(&gu.mapB[0], a.sh_gate.codes, Fs, H / 2, 128) && make_map(&gu.mapB[1], a.sh_up.codes, Fs, H / 2, 128) &&
            make_map(&gu.mapB[2], a.gate.codes, (uint64_t)E * F, H / 2, 128) &&
            make_map(&gu.mapB[3], a.up.codes, (uint64_t)E * F, H / 2, 128);
  if (!ok) return cudaErrorInvalidValue;
  gu.sclA[0] = sa.xq_scales; gu.sclA[1] = sa.xp_scales;
  gu.rowsA[0] = T; gu.rowsA[1] = (int)PP;
  gu.sclB[0] = a.sh_gate.scales; gu.sclB[1] = a.sh_up.scales; gu.sclB[2] = a.gate.scales; gu.sclB[3] = a.up.scales;
  gu.Kel[0] = H; gu.Kel[1] = H;
  gu.rowsB[0] = Fs; gu.rowsB[1] = F;
  gu.items = sc.items_gu; gu.n_items = sc.n_items_gu; gu.item_begin = 0; gu.item_end_host = -1;
  gu.tscA[0] = a.sh_gate.tsc; gu.tscA[1] = a.gate.tsc; gu.tscB[0] = a.sh_up.tsc; gu.tscB[1] = a.up.tsc;
  gu.hcodes[0] = reinterpret_cast<uint8_t*>(at(L.hs_c)); gu.hscales[0] = reinterpret_cast<uint8_t*>(at(L.hs_s));
  gu.hcodes[1] = reinterpret_cast<uint8_t*>(at(L.hq_c)); gu.hscales[1] = reinterpret_cast<uint8_t*>(at(L.hq_s));
  gu.Fout[0] = Fs; gu.Fout[1] = F;
  gu.H = H; gu.K = K; gu.T = T; gu.E = E;
  const int smem_gu = kStages * StageLayout<kGateUp>::stride + 1024;
  e = cudaFuncSetAttribute(k_gemm_fp4<kGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_gu);
  if (e != cudaSuccess) return e;
  k_gemm_fp4<kGateUp><<<sms, kGThreads, smem_gu, st>>>(gu);

  // 6 down grouped GEMM: shared items (write out = x + y), then routed (red.add)
  GemmArgs dn;
  memset(&dn, 0, sizeof(dn));
  ok = make_map(&dn.mapA[0], gu.hcodes[0], T, Fs / 2, 128) && make_map(&dn.mapA[1], gu.hcodes[1], PP, F / 2, 128) &&
       make_map(&dn.mapB[0], a.sh_down.codes, H, Fs / 2, 128) &&
       make_map(&dn.mapB[2], a.down.codes, (uint64_t)E * H, F / 2, 128);
  if (!ok) return cudaErrorInvalidValue;
  dn.sclA[0] = gu.hscales[0]; dn.sclA[1] = gu.hscales[1];
  dn.rowsA[0] = T; dn.rowsA[1] = (int)PP;
  dn.sclB[0] = a.sh_down.scales; dn.sclB[2] = a.down.scales;
  dn.Kel[0] = Fs; dn.Kel[1] = F;
  dn.rowsB[0] = H; dn.rowsB[1] = H;
  dn.items = sc.items_dn; dn.n_items = sc.n_items_dn;
  dn.tscA[0] = a.sh_down.tsc; dn.tscA[1] = a.down.tsc;
  dn.x = a.x; dn.out = a.out; dn.order = sa.order; dn.wpair = r.w;
  dn.H = H; dn.K = K; dn.T = T; dn.E = E;
  const int smem_dn = kStages * StageLayout<kDown>::stride + 1024;
  e = cudaFuncSetAttribute(k_gemm_fp4<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_dn);
  if (e != cudaSuccess) return e;
  const int n_sh_dn = (T + kBM - 1) / kBM * (H / kBN);
  dn.item_begin = 0; dn.item_end_host = n_sh_dn;
  k_gemm_fp4<kDown><<<sms, kGThreads, smem_dn, st>>>(dn);
  dn.item_begin = n_sh_dn; dn.item_end_host = -1;
  k_gemm_fp4<kDown><<<sms, kGThreads, smem_dn, st>>>(dn);
  return cudaGetLastError();
}

}  // namespace flint
