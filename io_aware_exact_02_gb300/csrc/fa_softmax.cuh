// fa_softmax.cuh -- one step of the forward pass's online softmax over a
// 128 x 128 score tile in tensor memory, shared by the forward kernels.
//
// Thread r of a softmax warpgroup owns row r of the tile (TMEM lane r).  The
// step reads the row's 128 scores S from tensor memory, masks columns at and
// past `tlim` (the row's visible keys end there), takes the tile's extreme,
// moves the row's reference maximum only when the tile's exceeds it by more
// than kRescaleSlack (log2 units), writes P = 2^(c2 * S - m) over S as bf16
// pairs (or E4M3 quadruples), adds P's row sum to l, and rescales the row's O
// accumulator in tensor memory when the reference moved (cs2680 Lecture 9,
// sec. 9.4; "Reading CMU 11-868 LLM Systems: FlashAttention", slide pages
// 12 and 51-52).  O and l share the reference, so O / l and
// lse = (m + log2 l) ln 2 are exact whatever the reference is.
#pragma once

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

constexpr float kRescaleSlack = 8.0f;  // log2 units

// colS / colO: this thread's TMEM address of the tile's S and O columns.
// c2 = scale * log2(e) (nonzero).  may_rescale: O holds earlier tiles'
// products (false on the row's first key tile, whose O is overwritten).
// The caller waits for S and fences before the call, and fences and signals
// P's completion after it.  bf16 P is published in two halves: once the
// probabilities of keys 0-63 are in tensor memory, half_ready() is called,
// so that the first half of O += P V can run while keys 64-127 are
// exponentiated.  A warp that rescales O (rarely) calls it only after the
// rescale, at the end.  before_rescale() is called before O is read for a
// rescale: it must return once the previous P V product has written O (the
// caller's S having completed implies that, unless the tensor core computed
// S ahead of that product).  Warp-collective (TMEM loads and stores).
template <int D, bool kNeg, bool kFp8, class HalfReady, class BeforeRescale>
__device__ __forceinline__ void softmax_tile_w(uint32_t colS, uint32_t colO, float c2, int tlim,
                                               bool may_rescale, float& m_ref, float& l,
                                               HalfReady&& half_ready,
                                               BeforeRescale&& before_rescale) {
  // A masked score is replaced by the value that loses every max (min)
  // and whose exponent c2 * s is -inf, so its probability is exactly 0.
  const float neutral = kNeg ? __int_as_float(0x7f800000) : __int_as_float(0xff800000);
  const float ninf = __int_as_float(0xff800000);
  uint32_t sr[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(colS + c * 32, sr[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);

  if (tlim < kTile) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c * 32 + i >= tlim) sr[c][i] = __float_as_uint(neutral);
  }
  // Tile extreme of the raw scores: eight independent chains of
  // three-input max (min), joined by a tree (exact in any order).
  float mx8[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx8[u] = neutral;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const int u = (i >> 1) & 7;
      mx8[u] = kNeg ? fmin3(mx8[u], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]))
                    : fmax3(mx8[u], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
    }
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int u = 0; u < w; ++u)
      mx8[u] = kNeg ? fminf(mx8[u], mx8[u + w]) : fmaxf(mx8[u], mx8[u + w]);
  const float m_tile = mx8[0] * c2;
  float alpha = 1.f;
  if (m_tile > m_ref + kRescaleSlack) {
    alpha = ex2_approx(m_ref - m_tile);  // 0 on the first tile (m_ref = -inf)
    m_ref = m_tile;
  }
  l *= alpha;
  // O must be rescaled if this row's reference moved (warp-wide decision:
  // TMEM loads/stores are warp-collective).
  const bool rescale = may_rescale && __any_sync(0xffffffffu, alpha != 1.f);
  // p = 2^(c2 * s - m) for pairs of scores with packed f32x2 FMAs (a
  // row that has seen no key yet keeps m = -inf and all p = 0); four
  // packed partial row sums, joined by a tree below.
  const float neg_m = m_ref == ninf ? 0.f : -m_ref;
  const uint64_t c2x2 = f2_pack(c2, c2);
  const uint64_t negm2 = f2_pack(neg_m, neg_m);
  uint64_t ls4[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) ls4[u] = 0;
  uint32_t pk8[kFp8 ? 32 : 1];  // FP8: all 128 probabilities, four per column
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int c2i = 0; c2i < 2; ++c2i) {
      const int c = 2 * h + c2i;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])),
                         c2x2, negm2),
                  x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        ls4[(i >> 1) & 3] = f2_add(ls4[(i >> 1) & 3], f2_pack(p0, p1));
        if constexpr (kFp8) {
          const uint32_t two = pack_e4m3x2(p0, p1);
          if (((i >> 1) & 1) == 0)
            pk8[(c * 32 + i) >> 2] = two;
          else
            pk8[(c * 32 + i) >> 2] |= two << 16;
        } else {
          pk[c2i * 16 + i / 2] = pack_bf16x2(p0, p1);
        }
      }
    }
    if constexpr (!kFp8) {
      tmem_st32(colS + h * 32, pk);
      if (h == 0 && !rescale) {
        tmem_wait_st();
        tc_fence_before();
        half_ready();
      }
    }
  }
  if constexpr (kFp8) tmem_st32(colS, pk8);
  ls4[0] = f2_add(f2_add(ls4[0], ls4[1]), f2_add(ls4[2], ls4[3]));
  float lsa, lsb;
  f2_unpack(ls4[0], lsa, lsb);
  l += lsa + lsb;
  tmem_wait_st();
  // Correct the O accumulator once the previous P V product has written it
  // (before_rescale); no product of this tile's P reads O before the warp's
  // half_ready().
  if (rescale) {
    before_rescale();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t orow[32];
      tmem_ld32(colO + c * 32, orow);
      tmem_wait_ld(orow);
#pragma unroll
      for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
      tmem_st32(colO + c * 32, orow);
    }
    tmem_wait_st();
    if constexpr (!kFp8) {
      tc_fence_before();
      half_ready();
    }
  }
}

template <int D, bool kNeg, bool kFp8, class HalfReady>
__device__ __forceinline__ void softmax_tile(uint32_t colS, uint32_t colO, float c2, int tlim,
                                             bool may_rescale, float& m_ref, float& l,
                                             HalfReady&& half_ready) {
  softmax_tile_w<D, kNeg, kFp8>(colS, colO, c2, tlim, may_rescale, m_ref, l, half_ready, [] {});
}

}  // namespace fa
