// mma_bench.cu -- block-scaled FP4 tensor-core microbenchmark (tcgen05.mma
// kind::mxf4nvf4, E2M1 x E2M1 with an E4M3 scale per 16 elements), the measured FP4
// peak that prefill's GEMM is compared with, and the latency of the small MMA chains
// the decode kernel issues.  Operands live in shared memory and TMEM only: no global
// traffic inside the timed loop.
//
//   mode 0 (throughput): per iteration, four K = 64 steps x two 128 x 128 accumulators
//          (eight MMAs of M = 128, N = 128, K = 64, 2 * 128 * 128 * 64 FLOP each), all
//          issued back to back by one thread; one commit at the end.
//   mode 1 (latency): per iteration, the decode gate/up shape -- 16 K = 64 steps of
//          M = 128, N = 32, each with its two scale copies (tcgen05.cp), then a commit,
//          the wait for it and a tcgen05.ld of the accumulator.
//   modes 2-4 split that cost: 2 the same chain with the scales copied once before the
//          loop, 3 the scale copies alone (no MMA), 4 as 2 with the K steps alternating
//          between two accumulators (two independent chains of 8); 5 and 6 are modes 1
//          and 2 with the 16 steps unrolled.
// cycles[b] receives CTA b's clock64 cycles over the loop.
#include "common.cuh"

namespace flint {
namespace mb {

constexpr int kThreads = 128;
constexpr int kSmem = 64 * 1024 + 32 * 1024 + 2 * 8192 + 1024;   // A, B, scale chunks, alignment

__global__ void __launch_bounds__(kThreads, 1) k_fp4_mma_bench(int mode, int iters, unsigned long long* cycles) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* A = smem;                          // 128 rows x 512 B codes (4 swizzle atoms of 16 KB)
  uint8_t* B = smem + 64 * 1024;              // mode 0: 2 x 128 rows x 128 B; mode 1: 32 rows x 512 B
  uint8_t* SFA = B + 32 * 1024;               // 16 chunks of 512 B
  uint8_t* SFB = SFA + 8192;                  // 16 chunks of 512 B
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ volatile uint32_t sink;
  const int warp = threadIdx.x >> 5;

  // operands: any byte is a valid E2M1 pair; scales 0x38 = 1.0 in E4M3
  for (int i = threadIdx.x; i < 96 * 1024 / 4; i += kThreads)
    reinterpret_cast<uint32_t*>(A)[i] = (uint32_t)i * 2654435761u;
  for (int i = threadIdx.x; i < 16384 / 4; i += kThreads) reinterpret_cast<uint32_t*>(SFA)[i] = 0x38383838u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    pf::mb_init(&done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(pf::sh(&tmem_base)), "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pf::tc_fence_before();
  __syncthreads();
  pf::tc_fence_after();
  const uint32_t tmem = tmem_base;
  long long t0 = clock64();
  uint32_t phase = 0;
  if (mode == 0) {
    // D0 = columns [0, 128), D1 = [128, 256); scales: A at 256, B tiles at 260 / 264
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    if (threadIdx.x == 0) {
      const uint64_t dA = pf::umma_desc_sw128(pf::sh(A)), dB = pf::umma_desc_sw128(pf::sh(B));
      pf::tc_cp_sf(tmem + 256, pf::sf_desc(pf::sh(SFA)));
      pf::tc_cp_sf(tmem + 260, pf::sf_desc(pf::sh(SFB)));
      pf::tc_cp_sf(tmem + 264, pf::sf_desc(pf::sh(SFB + 512)));
      t0 = clock64();
#pragma unroll 1
      for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int b = 0; b < 2; ++b)
            pf::mma_fp4(tmem + 128 * b, dA + kk * 2, dB + ((b * 16384) >> 4) + kk * 2, idesc,
                        (it > 0 || kk > 0) ? 1u : 0u, tmem + 256, tmem + 260 + 4 * b);
      pf::tc_commit(&done);
    }
    __syncwarp();
    int abort_flag = 0;
    pf::mb_wait(&done, 0, &abort_flag, kWaitLimitNs);
  } else {
    // D = columns [0, 32) (mode 4: [32 c, 32 c + 32) for chain c); A scales at 64 + 4 s,
    // B scales at 128 + 4 s (s = K step)
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(32 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint64_t dA = pf::umma_desc_sw128(pf::sh(A)), dB = pf::umma_desc_sw128(pf::sh(B));
    if (mode != 1 && mode != 5 && threadIdx.x == 0)
#pragma unroll 1
      for (int s = 0; s < 16; ++s) {
        pf::tc_cp_sf(tmem + 64 + 4 * s, pf::sf_desc(pf::sh(SFA + 512 * s)));
        pf::tc_cp_sf(tmem + 128 + 4 * s, pf::sf_desc(pf::sh(SFB + 512 * s)));
      }
    t0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
      if (threadIdx.x == 0 && mode >= 5) {
        // modes 5 / 6: mode 1 / mode 2 with the 16 steps unrolled (descriptors fold to constants)
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (mode == 5) {
            pf::tc_cp_sf(tmem + 64 + 4 * s, pf::sf_desc(pf::sh(SFA + 512 * s)));
            pf::tc_cp_sf(tmem + 128 + 4 * s, pf::sf_desc(pf::sh(SFB + 512 * s)));
          }
          pf::mma_fp4(tmem, dA + ((s >> 2) * 16384 >> 4) + (s & 3) * 2, dB + ((s >> 2) * 4096 >> 4) + (s & 3) * 2,
                      idesc, s > 0 ? 1u : 0u, tmem + 64 + 4 * s, tmem + 128 + 4 * s);
        }
        pf::tc_commit(&done);
      } else if (threadIdx.x == 0) {
#pragma unroll 1
        for (int s = 0; s < 16; ++s) {
          if (mode == 1 || mode == 3) {
            pf::tc_cp_sf(tmem + 64 + 4 * s, pf::sf_desc(pf::sh(SFA + 512 * s)));
            pf::tc_cp_sf(tmem + 128 + 4 * s, pf::sf_desc(pf::sh(SFB + 512 * s)));
          }
          if (mode != 3) {
            const uint32_t d = mode == 4 ? tmem + 32 * (s & 1) : tmem;
            const uint32_t acc = mode == 4 ? (s > 1 ? 1u : 0u) : (s > 0 ? 1u : 0u);
            pf::mma_fp4(d, dA + ((s >> 2) * 16384 >> 4) + (s & 3) * 2, dB + ((s >> 2) * 4096 >> 4) + (s & 3) * 2,
                        idesc, acc, tmem + 64 + 4 * s, tmem + 128 + 4 * s);
          }
        }
        pf::tc_commit(&done);
      }
      __syncwarp();
      int abort_flag = 0;
      pf::mb_wait(&done, phase, &abort_flag, kWaitLimitNs);
      phase ^= 1u;
      pf::tc_fence_after();
      uint32_t r[16];
      pf::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16), r);
      pf::tmem_wait_ld();
      if (threadIdx.x == 0) sink = r[0] ^ r[15];      // keeps the load
      pf::tc_fence_before();
      __syncthreads();
    }
  }
  const long long t1 = clock64();
  if (threadIdx.x == 0) cycles[blockIdx.x] = (unsigned long long)(t1 - t0);
  pf::tc_fence_before();
  __syncthreads();
  pf::tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(512));
}

}  // namespace mb

cudaError_t launch_fp4_mma_bench(int mode, int iters, int ctas, unsigned long long* cycles, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(mb::k_fp4_mma_bench, cudaFuncAttributeMaxDynamicSharedMemorySize, mb::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  mb::k_fp4_mma_bench<<<ctas, mb::kThreads, mb::kSmem, st>>>(mode, iters, cycles);
  return cudaGetLastError();
}

}  // namespace flint
