// lm_head.cu -- NVFP4 output head: logits = W x, argmax (ties to the lower index).
//
// The head is 2,048 -> 150,144, untied and quantised to 4 bits ("Flint: 125 tokens a
// second is what 2.5B active parameters buy at 273 GB/s", sections "The shape, read
// from the headers" and "Why active parameters set the speed").  It is a GEMV per token,
// and its batch (B <= 8 tokens) maps onto the 8 columns of the B operand of mma.sync
// m16n8k16 (B = 1 takes a CUDA-core kernel, see k_lm_head_rows): a warp takes 16 rows
// at a time and reads them once from HBM with 128-bit
// streaming loads, decodes them to f16 (cvt.rn.f16x2.e2m1x2, times the E4M3 block scale:
// exact in f16) and multiplies them by all B tokens' f16 activations (each token scaled
// by its own power of two) with fp32 accumulation -- so B = 8 costs the weight stream
// and the decode once, not eight times.  Lane (g, t) of the mma fragments holds rows g
// and g + 8 and reads 32-column chunk 4 c + t of each; the B operand follows the same
// column order.  The vocabulary is split over a grid of 2 CTAs per SM; each warp keeps
// a running (max, index) per token, the CTA's best goes to the workspace, and the last
// CTA to finish reduces those to the argmax.
#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"

namespace flint {

constexpr int kHeadWarps = 8;
constexpr int kHeadThreads = 32 * kHeadWarps;
constexpr int kHeadCols = 8;          // tokens per launch (the mma's N)
constexpr int kHeadGroup = 4;         // chunk sets per loop iteration (loads in flight)

struct HeadArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tsc;
  int V, H, B;
  const uint16_t* x;      // [B][H] bf16
  float* logits;          // [B][V] or null
  int32_t* argmax;        // [B] or null
  float* best_v;          // ws [grid][FLINT_MAX_DECODE_TOKENS]
  int* best_i;            // ws [grid][FLINT_MAX_DECODE_TOKENS]
  unsigned int* counter;  // ws, zero between launches
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ uint32_t hmul2_h(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void mma16816_h(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One token (B = 1): CUDA cores.  A slice of LPR = H / (32 CPL) lanes takes a row with
// 128-bit streaming loads (kHeadNR rows in flight per slice), decodes it in registers and
// multiplies it by the token held in registers (f16, times 2^k) with fma.rn.f32.f16; the
// slice reduces with shuffles.  For a single token this beats the mma.sync path, whose
// decode and scale products are the same while its tensor-core work is 7/8 idle.
constexpr int kHeadNR = 4;   // rows in flight per slice

template <int CPL, int NT>
__global__ void __launch_bounds__(kHeadThreads, 2) k_lm_head_rows(HeadArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPR = a.H / (32 * CPL);
  const int RPP = 32 / LPR;
  const int slice = lane / LPR, sl = lane % LPR;
  const int gwarp = blockIdx.x * kHeadWarps + warp, nwarps = gridDim.x * kHeadWarps;
  const size_t cb = a.H / 2, sb = a.H / 16;
  const float tsc = a.tsc[0];
  XStage<CPL, 1> xs[NT];
  const int nt = min(NT, a.B);
#pragma unroll
  for (int t = 0; t < NT; ++t)
    stage_bf16<CPL>(xs[t], nullptr, a.x + (size_t)(t < nt ? t : 0) * a.H, sl, LPR);
  float bv[NT];
  int bi[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) { bv[t] = -INFINITY; bi[t] = 0x7FFFFFFF; }
  const int rows_per_task = RPP * kHeadNR;
  const int n_tasks = (a.V + rows_per_task - 1) / rows_per_task;
  for (int task = gwarp; task < n_tasks; task += nwarps) {
    RowRegs<CPL> r[kHeadNR];
#pragma unroll
    for (int p = 0; p < kHeadNR; ++p) {
      int row = task * rows_per_task + p * RPP + slice;
      row = row < a.V ? row : a.V - 1;
      load_row<CPL>(r[p], a.codes + row * cb, a.scales + row * sb, sl, LPR);
    }
#pragma unroll
    for (int p = 0; p < kHeadNR; ++p) {
      const int row = task * rows_per_task + p * RPP + slice;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = sum_lanes_rt(dot_row<CPL, 1>(r[p], xs[t]), LPR) * (tsc * xs[t].unscale);
        if (t < nt && row < a.V) {
          if (sl == 0 && a.logits) a.logits[(size_t)t * a.V + row] = v;
          const float vv = (v == v) ? v : -INFINITY;
          if (better(vv, row, bv[t], bi[t])) { bv[t] = vv; bi[t] = row; }
        }
      }
    }
  }
  // block reduction of the running best, per token
  __shared__ float sv[kHeadWarps][NT];
  __shared__ int si[kHeadWarps][NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float v = bv[t];
    int i = bi[t];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    if (lane == 0) { sv[warp][t] = v; si[warp][t] = i; }
  }
  __syncthreads();
  if (threadIdx.x < NT) {
    const int t = threadIdx.x;
    float v = sv[0][t];
    int i = si[0][t];
    for (int w = 1; w < kHeadWarps; ++w)
      if (better(sv[w][t], si[w][t], v, i)) { v = sv[w][t]; i = si[w][t]; }
    a.best_v[blockIdx.x * FLINT_MAX_DECODE_TOKENS + t] = v;
    a.best_i[blockIdx.x * FLINT_MAX_DECODE_TOKENS + t] = i;
  }
  // last CTA: argmax over the CTAs' bests
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < nt) {
    const int t = warp;
    float v = -INFINITY;
    int i = 0x7FFFFFFF;
    for (int c = lane; c < (int)gridDim.x; c += 32) {
      const float cv = __ldcg(a.best_v + c * FLINT_MAX_DECODE_TOKENS + t);
      const int ci = __ldcg(a.best_i + c * FLINT_MAX_DECODE_TOKENS + t);
      if (better(cv, ci, v, i)) { v = cv; i = ci; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
    if (lane == 0 && a.argmax) a.argmax[t] = (i < a.V) ? i : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.counter = 0;
}

// One group of kHeadGroup 128-column chunk sets of rows ra (pa, qa) and rb (pb, qb):
// loads (a short last group re-reads the last set; those are never used) ...
struct HeadGroup {
  uint4 wa[kHeadGroup], wb[kHeadGroup];
  uint32_t fa[kHeadGroup], fb[kHeadGroup];
};
__device__ __forceinline__ void head_load(HeadGroup& G, const uint8_t* pa, const uint8_t* pb, const uint8_t* qa,
                                          const uint8_t* qb, int c0, int csets, int t) {
#pragma unroll
  for (int u = 0; u < kHeadGroup; ++u) {
    const int q = 4 * min(c0 + u, csets - 1) + t;
    G.wa[u] = ldg_stream(pa + 16 * q);
    G.wb[u] = ldg_stream(pb + 16 * q);
    G.fa[u] = ldg_stream_u16(qa + 2 * q);
    G.fb[u] = ldg_stream_u16(qb + 2 * q);
  }
}
// ... and products: decode, block scale, mma with the B columns (xcol: this lane's token)
__device__ __forceinline__ void head_mma(const HeadGroup& G, const uint32_t* xcol, int c0, int csets, int t,
                                         float (&d)[kHeadGroup][4]) {
#pragma unroll
  for (int u = 0; u < kHeadGroup; ++u) {
    if (c0 + u >= csets) break;
    const int q = 4 * (c0 + u) + t;
    const uint32_t ea = e4m3x2_to_f16x2(G.fa[u]), eb = e4m3x2_to_f16x2(G.fb[u]);
    const uint32_t SA[2] = {__byte_perm(ea, 0, 0x1010), __byte_perm(ea, 0, 0x3232)};
    const uint32_t SB[2] = {__byte_perm(eb, 0, 0x1010), __byte_perm(eb, 0, 0x3232)};
    const uint4* xp = reinterpret_cast<const uint4*>(xcol + 16 * q);
    const uint4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
    const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                             x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
    const uint32_t av[4] = {G.wa[u].x, G.wa[u].y, G.wa[u].z, G.wa[u].w};
    const uint32_t bw[4] = {G.wb[u].x, G.wb[u].y, G.wb[u].z, G.wb[u].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {                      // word h: mmas 2h, 2h + 1
      uint32_t fa4[4], fb4[4];
      e2m1x8_to_f16x2x4(av[h], fa4[0], fa4[1], fa4[2], fa4[3]);
      e2m1x8_to_f16x2x4(bw[h], fb4[0], fb4[1], fb4[2], fb4[3]);
      const uint32_t S_a = SA[h >> 1], S_b = SB[h >> 1];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int j = 2 * h + m;
        mma16816_h(d[u], hmul2_h(fa4[2 * m], S_a), hmul2_h(fb4[2 * m], S_b), hmul2_h(fa4[2 * m + 1], S_a),
                   hmul2_h(fb4[2 * m + 1], S_b), xv[2 * j], xv[2 * j + 1]);
      }
    }
  }
}

__global__ void __launch_bounds__(kHeadThreads, 2) k_lm_head(HeadArgs a) {
  extern __shared__ __align__(16) uint32_t s_x[];            // [kHeadCols][H/2] f16 pairs
  __shared__ float s_unscale[kHeadCols];
  __shared__ float sv[kHeadWarps][kHeadCols];
  __shared__ int si[kHeadWarps][kHeadCols];
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H, V = a.V;
  // ---- stage: warp n converts token n to f16 pairs times 2^k (max |x| 2^k in [2^14, 2^15));
  // columns without a token are zero
  {
    const int n = warp;
    uint32_t* dst = s_x + (size_t)n * (H / 2);
    if (n < a.B) {
      const uint16_t* xr = a.x + (size_t)n * H;
      float am = 0.f;
      for (int e = 2 * lane; e < H; e += 64) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(xr + e);
        am = fmaxf(am, fmaxf(fabsf(bf16_bits_to_f32(w & 0xFFFFu)), fabsf(bf16_bits_to_f32(w >> 16))));
      }
      am = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(am)));
      const int k = f16_stage_exponent(am);
      const float sc = exp2i(k);
      for (int e = 2 * lane; e < H; e += 64) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(xr + e);
        dst[e / 2] = pack_f16x2_rn(bf16_bits_to_f32(w & 0xFFFFu) * sc, bf16_bits_to_f32(w >> 16) * sc);
      }
      if (lane == 0) s_unscale[n] = exp2i(-k) * a.tsc[0];
    } else {
      for (int e = lane; e < H / 2; e += 32) dst[e] = 0u;
      if (lane == 0) s_unscale[n] = 0.f;
    }
  }
  __syncthreads();
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* xcol = s_x + (size_t)g * (H / 2);          // this lane's B column: token g
  const size_t cb = H / 2, sb = H / 16;
  const int csets = H / 128;                                  // 128-column chunk sets (H % 128 == 0)
  const int gwarp = blockIdx.x * kHeadWarps + warp, nwarps = gridDim.x * kHeadWarps;
  const int n_tiles = (V + 15) / 16;
  const float us0 = s_unscale[2 * t], us1 = s_unscale[2 * t + 1];
  float bv0 = -INFINITY, bv1 = -INFINITY;                     // running best of tokens 2t, 2t + 1
  int bi0 = 0x7FFFFFFF, bi1 = 0x7FFFFFFF;
  for (int tile = gwarp; tile < n_tiles; tile += nwarps) {
    const int ra = min(16 * tile + g, V - 1), rb = min(16 * tile + g + 8, V - 1);
    const uint8_t* pa = a.codes + (size_t)ra * cb;
    const uint8_t* pb = a.codes + (size_t)rb * cb;
    const uint8_t* qa = a.scales + (size_t)ra * sb;
    const uint8_t* qb = a.scales + (size_t)rb * sb;
    float d[kHeadGroup][4];
#pragma unroll
    for (int u = 0; u < kHeadGroup; ++u) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
    // two groups in flight: the next group's loads are issued before this one's products
    HeadGroup G0, G1;
    head_load(G0, pa, pb, qa, qb, 0, csets, t);
    for (int c0 = 0; c0 < csets; c0 += 2 * kHeadGroup) {
      if (c0 + kHeadGroup < csets) head_load(G1, pa, pb, qa, qb, c0 + kHeadGroup, csets, t);
      head_mma(G0, xcol, c0, csets, t, d);
      if (c0 + kHeadGroup >= csets) break;
      if (c0 + 2 * kHeadGroup < csets) head_load(G0, pa, pb, qa, qb, c0 + 2 * kHeadGroup, csets, t);
      head_mma(G1, xcol, c0 + kHeadGroup, csets, t, d);
    }
#pragma unroll
    for (int u = 1; u < kHeadGroup; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) d[0][i] += d[u][i];
    // d[0]: (row g, token 2t), (row g, token 2t + 1), (row g + 8, token 2t), (row g + 8, token 2t + 1)
    const int r0 = 16 * tile + g, r1 = r0 + 8;
    const float v[4] = {d[0][0] * us0, d[0][1] * us1, d[0][2] * us0, d[0][3] * us1};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = i < 2 ? r0 : r1, tok = 2 * t + (i & 1);
      if (row < V && tok < a.B) {
        if (a.logits) a.logits[(size_t)tok * V + row] = v[i];
        const float vv = (v[i] == v[i]) ? v[i] : -INFINITY;
        if (i & 1) { if (better(vv, row, bv1, bi1)) { bv1 = vv; bi1 = row; } }
        else { if (better(vv, row, bv0, bi0)) { bv0 = vv; bi0 = row; } }
      }
    }
  }
  // ---- per-token best: over the 8 lanes of each t (lane bits 2-4), then the CTA
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, bv0, o);
    int oi = __shfl_xor_sync(0xffffffffu, bi0, o);
    if (better(ov, oi, bv0, bi0)) { bv0 = ov; bi0 = oi; }
    ov = __shfl_xor_sync(0xffffffffu, bv1, o);
    oi = __shfl_xor_sync(0xffffffffu, bi1, o);
    if (better(ov, oi, bv1, bi1)) { bv1 = ov; bi1 = oi; }
  }
  if (g == 0) {
    sv[warp][2 * t] = bv0; si[warp][2 * t] = bi0;
    sv[warp][2 * t + 1] = bv1; si[warp][2 * t + 1] = bi1;
  }
  __syncthreads();
  if (threadIdx.x < a.B) {
    const int n = threadIdx.x;
    float bv = sv[0][n];
    int bi = si[0][n];
    for (int w = 1; w < kHeadWarps; ++w)
      if (better(sv[w][n], si[w][n], bv, bi)) { bv = sv[w][n]; bi = si[w][n]; }
    a.best_v[blockIdx.x * FLINT_MAX_DECODE_TOKENS + n] = bv;
    a.best_i[blockIdx.x * FLINT_MAX_DECODE_TOKENS + n] = bi;
  }
  // last CTA: argmax over the CTAs' bests
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < a.B) {
    const int n = warp;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int cta = lane; cta < (int)gridDim.x; cta += 32) {
      const float cv = __ldcg(a.best_v + cta * FLINT_MAX_DECODE_TOKENS + n);
      const int ci = __ldcg(a.best_i + cta * FLINT_MAX_DECODE_TOKENS + n);
      if (better(cv, ci, bv, bi)) { bv = cv; bi = ci; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0 && a.argmax) a.argmax[n] = (bi < V) ? bi : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.counter = 0;
}

static int head_grid() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms * 2;
}

size_t lm_head_workspace_bytes(int H, int V, int B) {
  (void)H; (void)V; (void)B;
  const size_t grid = 2 * 1024;  // upper bound on CTAs (2 per SM)
  return grid * FLINT_MAX_DECODE_TOKENS * (sizeof(float) + sizeof(int)) + 256;
}

cudaError_t launch_lm_head(const uint8_t* codes, const uint8_t* scales, const float* tsc, int V,
                           int H, const uint16_t* x, int B, float* logits, int32_t* argmax,
                           void* ws, cudaStream_t st) {
  HeadArgs a;
  a.codes = codes; a.scales = scales; a.tsc = tsc; a.V = V; a.H = H; a.B = B;
  a.x = x; a.logits = logits; a.argmax = argmax;
  char* p = static_cast<char*>(ws);
  a.counter = reinterpret_cast<unsigned int*>(p);
  p += 256;
  a.best_v = reinterpret_cast<float*>(p);
  p += (size_t)2 * 1024 * FLINT_MAX_DECODE_TOKENS * sizeof(float);
  a.best_i = reinterpret_cast<int*>(p);
  const size_t smem = (size_t)kHeadCols * H * 2;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_lm_head, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kHeadCols * FLINT_MAX_HIDDEN * 2));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (B == 1 && (H & (H - 1)) == 0) {             // slices of a power-of-two width
    if (H <= 1024) k_lm_head_rows<1, 1><<<head_grid(), kHeadThreads, 0, st>>>(a);
    else if (H <= 2048) k_lm_head_rows<2, 1><<<head_grid(), kHeadThreads, 0, st>>>(a);
    else k_lm_head_rows<4, 1><<<head_grid(), kHeadThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  k_lm_head<<<head_grid(), kHeadThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace flint
