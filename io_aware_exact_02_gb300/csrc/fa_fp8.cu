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
// head of one tensor; each warp handles whole rows, lane l holding the four
// consecutive elements 4l .. 4l+3 of a row.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 128;
constexpr int kQuantThreads = 256;

// Fast Walsh-Hadamard transform of a 128-element row held four elements
// per lane: y_j = sum_i x_i (-1)^popcount(i & j) (Sylvester order).  Each
// stage replaces the pair (x_i, x_{i+s}) by (x_i + x_{i+s}, x_i - x_{i+s});
// strides 1 and 2 stay inside the lane, strides 4 to 64 pair lane l with
// lane l ^ (s / 4).
__device__ __forceinline__ void fwht128(float (&x)[4], int lane) {
  const float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
  x[0] = a0 + a2;
  x[1] = a1 + a3;
  x[2] = a0 - a2;
  x[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? o - x[e] : x[e] + o;
    }
  }
}

// Row `row` of head `bh` of a [BH][N][128] bf16 tensor, four elements per
// lane, rotated when `rotate`.
__device__ __forceinline__ void load_row(const __nv_bfloat16* base, int bh, int N, int row,
                                         bool rotate, int lane, float (&x)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(base + ((size_t)bh * N + row) * kD + 4 * lane);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
  if (rotate) fwht128(x, lane);
}

struct QuantArgs {
  const __nv_bfloat16* src[3];  // Q, K, V
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* vt8;
  float* amax;                  // [3][BH]
  int BH, N, n_kv, hadamard;
};

// Pass 1: amax[tensor][bh] = max |x| over the head (after the rotation for
// Q and K).  amax must be zero on entry; the maximum of non-negative floats
// is the maximum of their bit patterns as unsigned integers.
__global__ void __launch_bounds__(kQuantThreads) fa_fp8_amax_kernel(const QuantArgs a) {
  const int tile = blockIdx.x % a.n_kv, bh = blockIdx.x / a.n_kv, which = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool rotate = a.hadamard && which < 2;
  float m = 0.f;
  for (int r = warp; r < kTile; r += kQuantThreads / 32) {
    const int row = tile * kTile + r;
    if (row >= a.N) break;
    float x[4];
    load_row(a.src[which], bh, a.N, row, rotate, lane, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(x[e]));
  }
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool rotate = a.hadamard && which < 2;
  const float amax = a.amax[which * a.BH + bh];
  const float inv = amax == 0.f ? 1.f : 448.f / amax;
  for (int r = warp; r < kTile; r += kQuantThreads / 32) {
    const int row = tile * kTile + r;
    uint32_t codes = 0;  // rows past N: code 0 (only V stores them)
    if (row < a.N) {
      float x[4];
      load_row(a.src[which], bh, a.N, row, rotate, lane, x);
      codes = pack_e4m3x2(x[0] * inv, x[1] * inv) | (pack_e4m3x2(x[2] * inv, x[3] * inv) << 16);
    }
    if (which < 2) {
      if (row < a.N) {
        uint8_t* dst = (which == 0 ? a.q8 : a.k8) + ((size_t)bh * a.N + row) * kD + 4 * lane;
        *reinterpret_cast<uint32_t*>(dst) = codes;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) vt[(4 * lane + e) * kStride + r] = (uint8_t)(codes >> (8 * e));
    }
  }
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
  a.src[0] = static_cast<const __nv_bfloat16*>(q);
  a.src[1] = static_cast<const __nv_bfloat16*>(k);
  a.src[2] = static_cast<const __nv_bfloat16*>(v);
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
