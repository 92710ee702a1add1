// gemv.cuh -- warp-level NVFP4 (and bf16) row-times-vector building blocks.
//
// Work layout.  A row of K elements is cut into 16-byte chunks of codes (32 elements,
// two 16-element scale blocks).  A "slice" of LPR = min(32, K/32) consecutive lanes
// owns one row at a time; lane sl of the slice reads chunks sl + LPR*i, i < CPL, so
// each warp-wide load instruction covers 32 consecutive 16-byte chunks (coalesced).
// 32/LPR slices in a warp work on different rows at once.  The activation vector is
// staged once per warp in registers, in the same chunk order, as f16 pairs scaled by
// a power of two (so every product with an E2M1 value is exact) -- one f16 term for
// bf16 inputs, a hi/lo pair of f16 terms for fp32 inputs.  Per chunk the lane decodes
// 16 code bytes with cvt.rn.f16x2.e2m1x2, multiplies into eight independent fp32
// accumulators with fma.rn.f32.f16, applies the two E4M3 block scales in fp32, and
// the slice reduces with shuffles.
#pragma once
#include "common.cuh"

namespace flint {

template <int CPL, int NX>
struct XStage {
  uint32_t p[NX][CPL * 16];  // f16x2 pairs (x[2q], x[2q+1]) * 2^k, chunk-major
  float unscale;             // 2^-k
};

template <int CPL>
struct XRawBF16 {
  uint32_t p[CPL * 16];      // bf16x2 pairs, unscaled
};

// Stage a bf16 vector (K = 32 * LPR * CPL elements) into f16 registers.
// Every lane of the warp must call this (shuffles over the whole warp).
template <int CPL>
__device__ __forceinline__ void stage_bf16(XStage<CPL, 1>& xs, XRawBF16<CPL>* raw,
                                           const uint16_t* __restrict__ x, int sl, int LPR) {
  uint32_t r[CPL * 16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(x + 32 * (sl + LPR * i));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 v = src[j];
      r[i * 16 + j * 4 + 0] = v.x; r[i * 16 + j * 4 + 1] = v.y;
      r[i * 16 + j * 4 + 2] = v.z; r[i * 16 + j * 4 + 3] = v.w;
    }
  }
#pragma unroll
  for (int q = 0; q < CPL * 16; ++q) {
    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(r[q] & 0xFFFFu)));
    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(r[q] >> 16)));
  }
  amax = max_lanes_rt(amax, LPR);
  const int k = f16_stage_exponent(amax);
  const float s = exp2i(k);
  xs.unscale = exp2i(-k);
#pragma unroll
  for (int q = 0; q < CPL * 16; ++q) {
    xs.p[0][q] = pack_f16x2_rn(bf16_bits_to_f32(r[q] & 0xFFFFu) * s, bf16_bits_to_f32(r[q] >> 16) * s);
    if (raw) raw->p[q] = r[q];
  }
}

template <int CPL>
struct RowRegs {
  uint4 q[CPL];
  uint32_t s[CPL];
};

template <int CPL>
__device__ __forceinline__ void load_row(RowRegs<CPL>& r, const uint8_t* __restrict__ codes_row,
                                         const uint8_t* __restrict__ scales_row, int sl, int LPR) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = sl + LPR * i;
    r.q[i] = ldg_stream(codes_row + 16 * c);
    r.s[i] = ldg_stream_u16(scales_row + 2 * c);
  }
}

// This lane's share of dot(row, x) (before the slice reduction, tensor scale and 2^-k).
template <int CPL, int NX>
__device__ __forceinline__ float dot_row(const RowRegs<CPL>& r, const XStage<CPL, NX>& xs) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const uint32_t w[4] = {r.q[i].x, r.q[i].y, r.q[i].z, r.q[i].w};
    float a[2][2][NX];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < NX; ++t) a[b][h][t] = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t h[4];
      e2m1x8_to_f16x2x4(w[wi], h[0], h[1], h[2], h[3]);
#pragma unroll
      for (int bi = 0; bi < 4; ++bi)
#pragma unroll
        for (int t = 0; t < NX; ++t)
          fma2_f16(a[wi >> 1][0][t], a[wi >> 1][1][t], h[bi], xs.p[t][i * 16 + wi * 4 + bi]);
    }
    float s0, s1;
    f16x2_to_f32x2(e4m3x2_to_f16x2(r.s[i]), s0, s1);
    float b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int t = 0; t < NX; ++t) {
      b0 += a[0][0][t] + a[0][1][t];
      b1 += a[1][0][t] + a[1][1][t];
    }
    acc = fmaf(b0, s0, acc);
    acc = fmaf(b1, s1, acc);
  }
  return acc;
}

}  // namespace flint
