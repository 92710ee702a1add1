// common.cuh -- device helpers shared by the Flint kernels (sm_103a).
//
// NVFP4 element decode uses the hardware conversion cvt.rn.f16x2.e2m1x2 (one byte,
// two E2M1 codes -> two f16 values, exact) and the products with activations use the
// mixed-precision fma.rn.f32.f16 (f16 x f16 products are exact in fp32, accumulation
// is fp32).  Both were measured on B300: the mixed FMA issues at the full FP32 rate,
// the conversion at a quarter of it, which together cover more than the ~40 weights
// per SM clock that HBM can deliver.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/flint.h"

namespace flint {

// ------------------------------------------------------------------ device status
// One status word per device, holding the first condition raised since the last
// read (FLINT_OK = nothing).  Kernels never trap; they record and return.  The library
// is one translation unit, so this definition is the only one.
__device__ unsigned int g_status = 0;

__device__ __forceinline__ void raise_status(unsigned int code) {
  atomicCAS(&g_status, 0u, code);
}

// Default bound of any spin on a flag/counter/mbarrier: 2 s of %globaltimer (the library's
// decode and prompt kernels take the runtime bound of flint_set_wait_limit_ns instead).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ memory
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ conversions
// Four bytes of E2M1 code pairs -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                  uint32_t& h2, uint32_t& h3) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}
// Two E4M3 bytes (low byte first) -> f16x2 (exact: every E4M3 value is an f16 normal).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t in = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}
// f16x2 -> two fp32 through the full-rate mixed FMA (x * 1 + (-0): exact, keeps -0).
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h, float& lo, float& hi) {
  asm("{ .reg .b16 l, u, one;\n"
      "  mov.b32 {l, u}, %2;\n"
      "  mov.b16 one, 0x3C00;\n"
      "  fma.rn.f32.f16 %0, l, one, 0f80000000;\n"
      "  fma.rn.f32.f16 %1, u, one, 0f80000000; }"
      : "=f"(lo), "=f"(hi) : "r"(h));
}
// acc_lo += w.lo * x.lo ; acc_hi += w.hi * x.hi   (f16 inputs, fp32 accumulate)
__device__ __forceinline__ void fma2_f16(float& acc_lo, float& acc_hi, uint32_t w, uint32_t x) {
  asm("{ .reg .b16 wl, wh, xl, xh;\n"
      "  mov.b32 {wl, wh}, %2;\n"
      "  mov.b32 {xl, xh}, %3;\n"
      "  fma.rn.f32.f16 %0, wl, xl, %0;\n"
      "  fma.rn.f32.f16 %1, wh, xh, %1; }"
      : "+f"(acc_lo), "+f"(acc_hi) : "r"(w), "r"(x));
}
// Same with bf16 inputs (router: bf16 weights x bf16 activations).
__device__ __forceinline__ void fma2_bf16(float& acc_lo, float& acc_hi, uint32_t w, uint32_t x) {
  asm("{ .reg .b16 wl, wh, xl, xh;\n"
      "  mov.b32 {wl, wh}, %2;\n"
      "  mov.b32 {xl, xh}, %3;\n"
      "  fma.rn.f32.bf16 %0, wl, xl, %0;\n"
      "  fma.rn.f32.bf16 %1, wh, xh, %1; }"
      : "+f"(acc_lo), "+f"(acc_hi) : "r"(w), "r"(x));
}
__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}
// 2^k as fp32, k in [-126, 127]
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }

// Power-of-two exponent k such that amax * 2^k lies in [2^14, 2^15): f16 then holds
// every activation at full precision down to amax * 2^-29.  0 when amax == 0.
__device__ __forceinline__ int f16_stage_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  int e = (int)(b >> 23) - 126;  // amax in [2^(e-1), 2^e) for a normal amax
  if ((b >> 23) == 0) frexpf(amax, &e);
  int k = 15 - e;
  return k > 126 ? 126 : (k < -126 ? -126 : k);
}

// ------------------------------------------------------------------ warp helpers
template <int W>
__device__ __forceinline__ float sum_lanes(float v) {
#pragma unroll
  for (int o = W / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float sum_lanes_rt(float v, int width) {
  for (int o = width / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float max_lanes_rt(float v, int width) {
  for (int o = width / 2; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

}  // namespace flint
