// fa_fp8.cu -- quantisation of Q, K, V to FP8 E4M3 for the FP8 forward pass,
// with the incoherent processing of the CMU 11-868 FlashAttention post (FA3
// section, slide page 24): the rows of Q and K are multiplied by the same
// Hadamard matrix, which leaves Q K^T unchanged up to the factor d and
// spreads outlier features over all columns before quantisation.
//
// Two HBM-bound passes over the bf16 inputs (d = 128): the first takes the
// per-head maximum |x| of the (rotated) tensors, the second writes the codes
// E4M3(x * 448 / amax), rounded to nearest-even and saturated.  V's codes are
// written transposed per head ([d][keys]) so that the attention kernel reads
// both operands of O += P V K-major.  One CTA handles a 128-row tile of one
// head of one tensor; each warp handles pairs of rows, lane l holding the
// eight consecutive elements 8l .. 8l+7 (l = lane mod 16) of one of the two
// (lanes 0-15 one row, lanes 16-31 the next).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 128;
constexpr int kQuantThreads = 256;

// Fast Walsh-Hadamard transform of a 128-element row held by 16 lanes,
// eight consecutive elements per lane (lane l of the half-warp holds
// elements 8l .. 8l+7): y_j = sum_i x_i (-1)^popcount(i & j) (Sylvester
// order).  Each stage replaces the pair (x_i, x_{i+s}) by (x_i + x_{i+s},
// x_i - x_{i+s}); strides 1, 2 and 4 stay inside the lane, strides 8 to 64
// pair lane l with lane l ^ (s / 8) of the same half-warp.
__device__ __forceinline__ void fwht128(float (&x)[8], int hl) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & s) == 0) {
        const float a = x[i], b = x[i + s];
        x[i] = a + b;
        x[i + s] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const bool upper = (hl & m) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? o - x[e] : x[e] + o;
    }
  }
}

// Work split of a 128-row tile: warp w, pass i (of kPasses) covers rows
// 2 * (w + 8 * i) + (lane >> 4); lane l & 15 holds elements 8l .. 8l+7.
constexpr int kPasses = kTile / (2 * (kQuantThreads / 32));  // 8
constexpr int kInFlight = 4;                                   // rows loaded ahead

__device__ __forceinline__ int tile_row(int warp, int i, int lane) {
  return 2 * (warp + 8 * i) + (lane >> 4);
}

// Eight elements of row `row` of head `bh` (0 past N), as fp32.
__device__ __forceinline__ uint4 load8(const __nv_bfloat16* base, int bh, int N, int row, int hl) {
  if (row >= N) return make_uint4(0u, 0u, 0u, 0u);
  return *reinterpret_cast<const uint4*>(base + ((size_t)bh * N + row) * kD + 8 * hl);
}

__device__ __forceinline__ void unpack8(uint4 raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

struct QuantArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* vt8;
  float* amax;                  // [3][BH]
  int BH, N, n_kv, hadamard;
};

// Visit the rows of this CTA's tile, kInFlight loads ahead of their use:
// f(i, row, x) receives pass i's row index and its (rotated) elements.
template <typename F>
__device__ __forceinline__ void for_rows(const QuantArgs& a, int which, int bh, int tile, F&& f) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, hl = lane & 15;
  const bool rotate = a.hadamard && which < 2;
  // (A select, not an index into the parameter block, which would copy it
  // to local memory.)
  const __nv_bfloat16* base = which == 0 ? a.q : (which == 1 ? a.k : a.v);
#pragma unroll
  for (int i0 = 0; i0 < kPasses; i0 += kInFlight) {
    uint4 raw[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u)
      raw[u] = load8(base, bh, a.N, tile * kTile + tile_row(warp, i0 + u, lane), hl);
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      float x[8];
      unpack8(raw[u], x);
      if (rotate) fwht128(x, hl);
      f(i0 + u, tile_row(warp, i0 + u, lane), x);
    }
  }
}

// Pass 1: amax[tensor][bh] = max |x| over the head (after the rotation for
// Q and K).  amax must be zero on entry; the maximum of non-negative floats
// is the maximum of their bit patterns as unsigned integers.
__global__ void __launch_bounds__(kQuantThreads) fa_fp8_amax_kernel(const QuantArgs a) {
  const int tile = blockIdx.x % a.n_kv, bh = blockIdx.x / a.n_kv, which = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = 0.f;
  for_rows(a, which, bh, tile, [&](int, int, const float(&x)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[e]));
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[kQuantThreads / 32];
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kQuantThreads / 32; ++w) t = fmaxf(t, wmax[w]);
    atomicMax(reinterpret_cast<unsigned int*>(a.amax + which * a.BH + bh), __float_as_uint(t));
  }
}

// Pass 2: the codes.  Q and K rows go to [BH][N][128]; V's tile is
// transposed through shared memory into [BH][128][n_kv * 128].
__global__ void __launch_bounds__(kQuantThreads) fa_fp8_quant_kernel(const QuantArgs a) {
  constexpr int kStride = kTile + 4;  // bytes per transposed row in shared memory
  __shared__ __align__(16) uint8_t vt[kD * kStride];
  const int tile = blockIdx.x % a.n_kv, bh = blockIdx.x / a.n_kv, which = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, hl = lane & 15;
  const float amax = a.amax[which * a.BH + bh];
  const float inv = amax == 0.f ? 1.f : 448.f / amax;
  uint8_t* qk = which == 0 ? a.q8 : a.k8;
  for_rows(a, which, bh, tile, [&](int, int r, const float(&x)[8]) {
    // Rows past N load as 0 and get code 0 (only V stores them).
    const uint32_t lo = pack_e4m3x2(x[0] * inv, x[1] * inv) |
                        (pack_e4m3x2(x[2] * inv, x[3] * inv) << 16);
    const uint32_t hi = pack_e4m3x2(x[4] * inv, x[5] * inv) |
                        (pack_e4m3x2(x[6] * inv, x[7] * inv) << 16);
    const int row = tile * kTile + r;
    if (which < 2) {
      if (row < a.N)
        *reinterpret_cast<uint2*>(qk + ((size_t)bh * a.N + row) * kD + 8 * hl) = make_uint2(lo, hi);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        vt[(8 * hl + e) * kStride + r] = (uint8_t)(lo >> (8 * e));
        vt[(8 * hl + 4 + e) * kStride + r] = (uint8_t)(hi >> (8 * e));
      }
    }
  });
  if (which < 2) return;
  __syncthreads();
  const size_t npad = (size_t)a.n_kv * kTile;
  for (int c = warp; c < kD; c += kQuantThreads / 32) {
    const uint32_t w4 = *reinterpret_cast<const uint32_t*>(&vt[c * kStride + 4 * lane]);
    *reinterpret_cast<uint32_t*>(a.vt8 + ((size_t)bh * kD + c) * npad + (size_t)tile * kTile +
                                 4 * lane) = w4;
  }
}

}  // namespace

int launch_fp8_quantize(const void* q, const void* k, const void* v, int BH, int N, int hadamard,
                        char* ws, const Fp8Workspace& layout, cudaStream_t stream) {
  QuantArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q8 = reinterpret_cast<uint8_t*>(ws + layout.q8);
  a.k8 = reinterpret_cast<uint8_t*>(ws + layout.k8);
  a.vt8 = reinterpret_cast<uint8_t*>(ws + layout.vt8);
  a.amax = reinterpret_cast<float*>(ws + layout.amax);
  a.BH = BH;
  a.N = N;
  a.n_kv = ceil_div(N, kTile);
  a.hadamard = hadamard;
  if (cudaMemsetAsync(a.amax, 0, (size_t)3 * BH * sizeof(float), stream) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const dim3 grid((unsigned)a.n_kv * (unsigned)BH, 3);  // n_kv * BH < 2^31 (checked)
  fa_fp8_amax_kernel<<<grid, kQuantThreads, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  fa_fp8_quant_kernel<<<grid, kQuantThreads, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

}  // namespace fa
