// quantize.cu -- bf16 -> NVFP4 (E2M1 codes, E4M3 scale per 16, fp32 tensor scale) and
// the reverse.  The format is the 4.5-bit NVFP4 of "Flint: 125 tokens a second is what
// 2.5B active parameters buy at 273 GB/s", section "Checking 125 tokens a second"; the
// recipe (two-level scales, fp32 with IEEE division, round-to-nearest-even with
// saturation) is the one documented in flint.h.
//
// Pass 1: per-matrix amax (and a non-finite check), 128-bit loads, one atomicMax per
//         block on the fp32 bit pattern (valid for non-negative floats).
// Pass 2: one thread per 16-element block: block amax, E4M3 block scale through
//         cvt.rn.satfinite.e4m3x2.f32, codes through cvt.rn.satfinite.e2m1x2.f32.
#include "common.cuh"
#include "launch.h"

namespace flint {

__global__ void __launch_bounds__(256) k_amax(const uint16_t* __restrict__ w, int64_t per_mat,
                                              int64_t n_vec /* 8-element vectors per matrix */,
                                              unsigned int* __restrict__ amax_bits) {
  const int m = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)m * per_mat);
  float amax = 0.f;
  bool finite = true;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = src[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = fabsf(bf16_bits_to_f32(u[j] & 0xFFFFu));
      const float b = fabsf(bf16_bits_to_f32(u[j] >> 16));
      finite &= (a <= 3.4e38f) & (b <= 3.4e38f);   // false for NaN and Inf
      amax = fmaxf(amax, fmaxf(a, b));
    }
  }
  // block reduction
  __shared__ float red[8];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  if (!finite) bad = 1;
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) a = fmaxf(a, red[i]);
    if (bad) {
      raise_status(FLINT_ERR_NONFINITE);
      atomicExch(&amax_bits[m], 0xFFFFFFFFu);  // marks the matrix
    } else {
      atomicMax(&amax_bits[m], __float_as_uint(a));
    }
  }
}

// E4M3 (satfinite, RNE) of a non-negative fp32 -> byte
__device__ __forceinline__ uint32_t to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}
// two fp32 -> E2M1 pair byte: lo in bits 0-3, hi in bits 4-7
__device__ __forceinline__ uint32_t to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.rn.satfinite.e2m1x2.f32 b, %1, %2; cvt.u32.u8 %0, b; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float e4m3_value(uint32_t byte) {
  float lo, hi;
  f16x2_to_f32x2(e4m3x2_to_f16x2(byte & 0xFFu), lo, hi);
  return lo;
}

__global__ void __launch_bounds__(256) k_quantize(const uint16_t* __restrict__ w, int n_mat,
                                                  int rows, int cols,
                                                  const unsigned int* __restrict__ amax_bits,
                                                  uint8_t* __restrict__ codes,
                                                  uint8_t* __restrict__ scales,
                                                  float* __restrict__ tsc_out) {
  const int m = blockIdx.y;
  const unsigned int ab = amax_bits[m];
  if (ab == 0xFFFFFFFFu) return;                       // non-finite matrix
  const float amax = __uint_as_float(ab);
  const float tsc = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) tsc_out[m] = tsc;
  const int64_t nblk = (int64_t)rows * (cols / 16);
  const uint16_t* wm = w + (size_t)m * rows * cols;
  uint8_t* cm = codes + (size_t)m * rows * (cols / 2);
  uint8_t* sm = scales + (size_t)m * rows * (cols / 16);
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(wm + b * 16);
    const uint4 v0 = src[0], v1 = src[1];
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = bf16_bits_to_f32(u[j] & 0xFFFFu);
      f[2 * j + 1] = bf16_bits_to_f32(u[j] >> 16);
    }
    float amax_b = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax_b = fmaxf(amax_b, fabsf(f[j]));
    const float t = __fdiv_rn(__fdiv_rn(amax_b, 6.0f), tsc);
    const uint32_t s = to_e4m3(t);
    const float eff = __fmul_rn(e4m3_value(s), tsc);
    uint32_t packed[2] = {0u, 0u};
    if (eff != 0.f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t byte = to_e2m1x2(__fdiv_rn(f[2 * j], eff), __fdiv_rn(f[2 * j + 1], eff));
        packed[j >> 2] |= byte << (8 * (j & 3));
      }
    }
    *reinterpret_cast<uint2*>(cm + b * 8) = make_uint2(packed[0], packed[1]);
    sm[b] = (uint8_t)s;
  }
}

__global__ void __launch_bounds__(256) k_dequantize(const uint8_t* __restrict__ codes,
                                                    const uint8_t* __restrict__ scales,
                                                    const float* __restrict__ tsc, int rows,
                                                    int cols, float* __restrict__ out) {
  const int m = blockIdx.y;
  const int64_t npair = (int64_t)rows * cols / 2;
  const uint8_t* cm = codes + (size_t)m * npair;
  const uint8_t* sm = scales + (size_t)m * rows * (cols / 16);
  float* om = out + (size_t)m * rows * cols;
  const float t = tsc[m];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < npair;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_f16x2x4(cm[i], h0, h1, h2, h3);
    float lo, hi;
    f16x2_to_f32x2(h0, lo, hi);
    const float s = e4m3_value(sm[(2 * i) / 16]);
    om[2 * i] = __fmul_rn(__fmul_rn(lo, s), t);
    om[2 * i + 1] = __fmul_rn(__fmul_rn(hi, s), t);
  }
}

cudaError_t launch_quantize(const uint16_t* w, int n_mat, int rows, int cols, uint8_t* codes,
                            uint8_t* scales, float* tsc, void* ws, cudaStream_t st) {
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(ws);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned int) * n_mat, st);
  if (e != cudaSuccess) return e;
  const int64_t per_mat = (int64_t)rows * cols;
  const int64_t n_vec = per_mat / 8;
  int gx = (int)((n_vec + 255) / 256);
  if (gx > 1184) gx = 1184;
  k_amax<<<dim3(gx, n_mat), 256, 0, st>>>(w, per_mat, n_vec, amax_bits);
  const int64_t nblk = (int64_t)rows * (cols / 16);
  int gq = (int)((nblk + 255) / 256);
  if (gq > 2368) gq = 2368;
  k_quantize<<<dim3(gq, n_mat), 256, 0, st>>>(w, n_mat, rows, cols, amax_bits, codes, scales, tsc);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* tsc,
                              int n_mat, int rows, int cols, float* out, cudaStream_t st) {
  const int64_t npair = (int64_t)rows * cols / 2;
  int g = (int)((npair + 255) / 256);
  if (g > 4736) g = 4736;
  k_dequantize<<<dim3(g, n_mat), 256, 0, st>>>(codes, scales, tsc, rows, cols, out);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status(unsigned int* out, cudaStream_t st) {
  unsigned int zero = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace flint
