// fa_fwd.cu -- forward pass of exact attention on sm_103a.
//
// A work item is 256 query rows (two 128-row Q tiles) of one head.  The grid
// is persistent (one CTA per SM; CMU 11-868 FlashAttention post, slide page
// 26), so the next item's Q and K/V loads overlap the end of the current
// one: without a mask each CTA walks a static share of the items; under a
// causal or block mask the CTAs claim the longest-first list greedily from a
// work counter (slide pages 27-46).  The producer decodes each item and
// hands the record to the other roles through a small ring in shared
// memory.  A CTA keeps both Q tiles in
// shared memory, streams the head's K and V tiles through a ring of
// shared-memory slots filled by TMA, and never writes a score to HBM: S
// lives in tensor memory, P replaces it there as bf16, and only O and the
// per-row logsumexp are stored (cs2680 Lecture 9, sec. 9.2 and 9.4; CMU post,
// slide pages 9-12).
//
// Warp roles (320 threads; 352 when O is staged; 384 at d = 64 and 512 with
// the epilogue warpgroup, see FwdCfg):
//   warps 0-3  softmax for Q tile 0 (thread r owns row r of the tile)
//   warps 4-7  softmax for Q tile 1
//   (kEpi)     warps 8-11 the epilogue warpgroup (O out of tensor memory)
//   then       the TMA producer (Q tiles once, then K_0, V_0, K_1, V_1, ...),
//              the MMA issuer (one thread, TMEM owner) and, when O is staged,
//              the O store warp (TMA stores of the staged O tiles)
// The two softmax warpgroups ping-pong: while one exponentiates its tile
// the tensor core computes the other tile's S and PV products (the overlap
// the CMU post motivates on slide pages 20-22 and 51-52).
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [0,128)  S for tile 0, overwritten in place by P (bf16 pairs, 64 cols)
//   [128,256) S / P for tile 1
//   [256,256+d) O accumulator of tile 0, [256+d, 256+2d) O of tile 1
//
// Online softmax per row (cs2680 Lecture 9 sec. 9.4, CMU post slide page 12):
// scores are used in log2 units t = scale*log2(e)*s.  The reference maximum
// m only moves when a tile's maximum exceeds it by more than kRescaleSlack,
// in which case the running denominator l and the O accumulator are
// multiplied by 2^(m_old - m_new); otherwise the stale m is kept and the
// exponentials stay below 2^kRescaleSlack.  O and l always share the same
// reference, so O / l and lse = (m + log2 l) * ln 2 are exact.
#include "fa_internal.h"
#include "fa_softmax.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kItemRing = 4;  // claimed item indices in flight between the roles

template <int D, bool kFp8 = false>
struct FwdCfg {
  static constexpr int kTileBytes = kTile * D * (kFp8 ? 1 : 2);  // one 128 x d tile
  static constexpr int kStages = kFp8 ? 10 : ((D == 128) ? 5 : 8);  // K/V ring slots
  // 2 softmax warpgroups, producer, MMA (and the O store warp when staging).
  // Ten or eleven warps put three on some SM sub-partitions, which caps a
  // thread at 168 registers.  At d = 64 (bf16) the kernel launches a twelfth
  // warp instead, so that the producer / MMA / store warps form a full
  // warpgroup that gives registers up (setmaxnreg) to the two softmax
  // warpgroups; the split uses the launch's 384 x 168 registers exactly.
  static constexpr bool kRealloc = D == 64 && !kFp8;
  // kEpi (d = 128, O staged): a third warpgroup takes each finished O tile
  // out of tensor memory, normalises it and stages it for the store, so
  // that the softmax warpgroups go straight on to the next item's first key
  // tile instead of spending the epilogue at every item boundary.  Sixteen
  // warps: softmax 0-7, epilogue 8-11, producer, MMA, store and one idle
  // warp 12-15; the registers of the launch (512 x 128) are split
  // 184 / 80 / 56.  (At d = 64 it measured no faster than the twelve-warp
  // split: 1097 against 1093 TFLOP/s at N = 8K, 693 against 712 for
  // B16 H12 N1K.)
  static constexpr bool epi(bool stage) { return stage && D == 128 && !kFp8; }
  static constexpr bool realloc(bool stage) { return kRealloc && !epi(stage); }
  static constexpr int threads(bool stage) {
    return epi(stage) ? 512 : (kRealloc ? 384 : (stage ? 352 : 320));
  }
  static constexpr int kRegsLaunch = 168;
  static constexpr int kRegsCtl = 72;
  static constexpr int kRegsSoftmax = 216;
  static_assert(!kRealloc || 2 * 128 * kRegsSoftmax + 128 * kRegsCtl <= 384 * kRegsLaunch,
                "register split above the launch's total");
  static constexpr int kEpiRegsLaunch = 128, kEpiRegsSoftmax = 184, kEpiRegsEpi = 80,
                       kEpiRegsCtl = 56;
  static_assert(2 * 128 * kEpiRegsSoftmax + 128 * kEpiRegsEpi + 128 * kEpiRegsCtl <=
                    512 * kEpiRegsLaunch,
                "register split above the launch's total");
  static constexpr uint32_t kTmemCols = 512;
  // TMEM column of S/P and of O for Q tile t.
  static __device__ __forceinline__ uint32_t col_s(int t) { return (uint32_t)t * 128u; }
  static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + (uint32_t)t * D; }
  // kSRing (d = 64, bf16): the 128 columns past the two 64-column O
  // accumulators are a third S buffer.  An item's S products (t, j), taken in
  // the order k = 2j + t, use buffer k % 3, so the tensor core computes
  // S(t, j+1) while softmax t still works on S(t, j): the product that last
  // used S(t, j+1)'s buffer is P(t, j) V's predecessor, product k - 1,
  // whose P V has been issued by then.  Buffer b's columns:
  static constexpr bool kSRing = D == 64 && !kFp8;
  static __device__ __forceinline__ uint32_t col_buf(int b) {
    return b < 2 ? (uint32_t)b * 128u : 256u + 2u * D;
  }
  static_assert(!kSRing || 256 + 2 * D + 128 <= (int)kTmemCols, "third S buffer past tensor memory");
  // MMA K-steps (32 bytes of each operand row per step) of S = Q K^T and
  // of O += P V.
  static constexpr int kKSteps = kFp8 ? D / 32 : D / 16;
  static constexpr int kPvSteps = kFp8 ? kTile / 32 : kTile / 16;
  // 128-byte TMA boxes per tile row (64 bf16 or 128 8-bit elements each).
  static constexpr int kBoxes = kFp8 ? D / 128 : D / 64;
};

// A work item: K/V head bh, pair `pair` of its packed query rows, key
// split; idx is its index in the list (the list's length: no item).  Q
// tile t's rows see key tiles [j0, j0 + n_t[t]) of the split.  Block-
// sparse: Q tile t has n_t[t] active key tiles and the item takes
// nmax = max(n_t[0], n_t[1]) steps.
struct FwdItem {
  int idx, bh, pair, split, row0, j0, n_t[2], nmax, hi[2];
};

template <int D, bool kFp8 = false>
struct alignas(1024) FwdSmem {
  uint8_t q[2][FwdCfg<D, kFp8>::kTileBytes];
  uint8_t kv[FwdCfg<D, kFp8>::kStages][FwdCfg<D, kFp8>::kTileBytes];
  uint64_t q_full;
  uint64_t q_empty;  // both Q tiles consumed by the item's last S product
  uint64_t kv_full[FwdCfg<D, kFp8>::kStages];
  uint64_t kv_empty[FwdCfg<D, kFp8>::kStages];
  uint64_t s_full[2];
  uint64_t p_half[2];   // bf16: P of keys 0-63 of the tile in tensor memory
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t pv_done[2];  // kSRing: O_t += P_t V complete (one phase per product)
  uint64_t o_empty[2];  // softmax t has read O_t of the item (epilogue done)
  uint64_t staged[2];   // softmax t has written O_t into its ring slot for the store
  uint64_t stored[2];   // the store warp has read softmax t's staged O_t
  uint64_t stage_ready[2];  // softmax t's staging slot of the item is free
  uint64_t ml_full[2];      // kEpi: softmax t has published its rows' 1 / l
  uint64_t ml_empty[2];     // kEpi: the epilogue has read them
  float inv_l[2][kTile];    // kEpi: 1 / l per row of each Q tile (0: no key seen)
  // The item ring: the producer writes the CTA's m-th item, decoded, into
  // slot m % kItemRing (item_full); every other role reads it and arrives
  // on item_empty.
  uint64_t item_full[kItemRing];
  uint64_t item_empty[kItemRing];
  FwdItem item_rec[kItemRing];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Wait sites reported through the status word.
enum : int {
  kSiteQFull = 101, kSiteKvEmpty, kSiteKvFull, kSitePFull, kSiteSFull, kSiteOFull, kSiteDrain,
  kSiteQEmpty, kSiteOEmpty, kSiteStageSlot, kSiteStaged, kSiteStored, kSitePHalf, kSiteMlFull,
  kSiteMlEmpty, kSiteItemFull, kSiteItemEmpty, kSitePvDone
};
// Bounds checks of the checked build (FA_CHECKS).
enum : int {
  kChkItem = 1101,  // a work item's head, pair, split or key-tile range
  kChkKvTile,       // a key tile loaded or scored
  kChkMask,         // an entry of the block mask
  kChkRow,          // an output row (O, lse, or a split's O and lse)
  kChkCombine       // a row or split of the combine kernel
};

// Descriptor of the K-major, 128B-swizzled tile at `base` for MMA K-step kk:
// 64-column blocks are 16 KB apart; a 16-element step is 32 bytes.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}

// Descriptor of a row-major [keys][d] tile used as the MN-major B operand of
// O += P V for K-step kk (16 keys = two 8-row groups = 2048 bytes).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, 16384, 1024);
}

// Wait without the abort shortcut: used while winding down after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > 100000000ull) return;  // 100 ms
  }
}

// kNeg: the scale is negative, so the tile's extreme is a minimum of the raw
// scores (the exponent scale * s is largest where s is smallest).
// kGeneral: grouped heads, N_q != N_kv or key splits; without it the kernel
// is the square case (rows = N_q = N_kv, one split) in its simplest form.
// kSparse (square case only): a block mask over (128-query tile, 128-key
// tile) pairs; each query tile of a pair walks its own active key tiles, and
// step j of the item loads the j-th active tile of each, so that the two
// tiles keep alternating on the tensor core as in the dense case.
// kFp8 (square case, d = 128): Q, K and V^T are E4M3 codes with one scale
// per head (the FP8 forward pass of the CMU 11-868 FlashAttention post,
// slide pages 18 and 24); S and O += P V run as kind::f8f6f4 products, P is
// rounded to E4M3 in tensor memory, and V arrives transposed ([d][keys]) so
// that both operands of O += P V are K-major.
// kDyn: persistent CTAs claim their items from the work counter p.sched
// (under a causal or block mask); otherwise the list is split statically.
template <int D, bool kNeg, bool kGeneral, bool kSparse, bool kFp8, bool kStage, bool kDyn>
__global__ void __launch_bounds__(FwdCfg<D, kFp8>::threads(kStage), 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  const FwdParams p) {
  using Cfg = FwdCfg<D, kFp8>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D, kFp8>& sm = *reinterpret_cast<FwdSmem<D, kFp8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abortf = &sm.abort_flag;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  constexpr bool kEpi = Cfg::epi(kStage);
  constexpr bool kRe = Cfg::realloc(kStage);
  // Warp roles: softmax 0-7, then (kEpi) the epilogue warpgroup 8-11, then
  // the producer, the MMA issuer and the O store warp.
  constexpr int kWarpLoad = kEpi ? 12 : 8, kWarpMma = kWarpLoad + 1, kWarpStore = kWarpLoad + 2;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_half[t], 128);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_full[t], 1);
      mbar_init(&sm.pv_done[t], 1);
      mbar_init(&sm.o_empty[t], 128);
      mbar_init(&sm.staged[t], 128);
      mbar_init(&sm.stored[t], 1);
      mbar_init(&sm.stage_ready[t], 1);
      mbar_init(&sm.ml_full[t], 128);
      mbar_init(&sm.ml_empty[t], 128);
    }
    // Readers of an item record: the MMA thread, the eight softmax warps,
    // the four epilogue warps and the store thread (when the kernel has them).
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&sm.item_full[i], 1);
      mbar_init(&sm.item_empty[i], 1 + 8 + (kEpi ? 4 : 0) + (kStage ? 1 : 0));
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // The setup above may overlap the end of the previous kernel on the stream
  // (programmatic dependent launch); its outputs are read only after this.
  wait_prior_grid();

  // Persistent CTAs without a work counter: CTA c takes the work items of
  // the longest-first list in "snake" order -- items c, 2G-1-c, 2G+c,
  // 4G-1-c, ... for G CTAs -- so that every CTA gets a similar mix of long
  // and short items.  With one CTA per item (G = items) each CTA takes
  // exactly item c.  With a work counter (p.sched) the producer claims the
  // next item of the list whenever it is ready to load one.  Either way the
  // producer decodes the item and hands the record to the other roles
  // through the item ring, so that they spend no time on it at an item
  // boundary.
  constexpr bool dyn = kDyn;
  const int splits = kGeneral ? p.splits : 1;
  const int num_items = p.BH * p.n_pairs * splits;
  const int G = gridDim.x;
  // kStage (square bf16 kernels on persistent CTAs): O leaves through the
  // K/V ring.  After an item's last K/V tiles the ring takes two more uses,
  // one per Q tile, in which the producer loads nothing; softmax warpgroup
  // t writes its O tile into that slot (128B-swizzled, as the TMA boxes)
  // and the store warp sends it out with TMA stores and then releases the
  // slot, so the softmax warps go on to the next item without waiting for
  // the stores.
  constexpr bool stage_epi = kStage;
  constexpr int ring_per_item_extra = stage_epi ? 2 : 0;
  auto item_of_round = [&](int k) -> int {
    const int base = k * G;
    return (k & 1) ? base + (G - 1 - (int)blockIdx.x) : base + (int)blockIdx.x;
  };
  // The list index of the CTA's m-th item (num_items: none left), for the
  // producer: claimed from the work counter, or the static split's.
  auto next_index = [&](int m) -> int {
    if (dyn) return min(atomicAdd(p.sched, 1), num_items);
    return m * G < num_items ? item_of_round(m) : num_items;
  };
  using Item = FwdItem;
  // The CTA's m-th item as the producer published it (idx == num_items:
  // none left).  The caller then releases the ring slot with
  // release_item(m), once per warp (or by the single thread of a
  // one-thread role) after all of its lanes have read the record.
  auto take_item = [&](int m, bool& ok) -> Item {
    const int slot = m % kItemRing;
    ok = mbar_wait(&sm.item_full[slot], (m / kItemRing) & 1, p.status, abortf, kSiteItemFull);
    Item it;
    if (ok) {
      it = sm.item_rec[slot];
    } else {
      it.idx = num_items;
    }
    return it;
  };
  auto release_item = [&](int m) { mbar_arrive(&sm.item_empty[m % kItemRing]); };
  // Block-sparse: is key tile jj active for query tile t of the item?
  auto active = [&](const Item& it, int t, int jj) -> bool {
    if (jj >= it.hi[t]) return false;
    const int qt = it.row0 / kTile + t;
    if (!bound_ok(qt < p.n_kv && jj >= 0 && jj < p.n_kv, p.status, abortf, kChkMask)) return false;
    return p.block_mask[(size_t)qt * p.n_kv + jj] != 0;
  };
  // The next key tile at or after c that query tile t uses; callers ask only
  // for tiles that exist, and the scan stops at the tile's last visible key
  // tile anyway.
  auto next_tile_t = [&](const Item& it, int t, int c) -> int {
    if constexpr (kSparse) {
      while (c < it.hi[t] && !active(it, t, c)) ++c;
    }
    return c;
  };
  auto decode = [&](int idx) -> Item {
    Item it;
    it.idx = idx;
    it.split = idx % splits;
    fwd_item(idx / splits, p.BH, p.n_pairs, &it.bh, &it.pair);
    it.row0 = it.pair * kPairRows;
    it.j0 = it.split * p.tiles_per_split;
    const int j1 = min(it.j0 + p.tiles_per_split, p.n_kv);
    it.nmax = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = it.row0 + t * kTile;
      int hi;
      if (kGeneral) {
        hi = fwd_tile_key_tiles(r0, p);
      } else {  // rows = N_kv: the causal tile r0/128 ends on the diagonal
        hi = r0 >= p.rows ? 0 : (p.causal ? min(r0 / kTile + 1, p.n_kv) : p.n_kv);
      }
      it.hi[t] = hi;
      const int n = min(hi, j1) - it.j0;
      it.n_t[t] = n > 0 ? n : 0;
      it.nmax = max(it.nmax, it.n_t[t]);
    }
    if (kSparse) {
      const int top = max(it.hi[0], it.hi[1]);
      it.n_t[0] = it.n_t[1] = 0;
      for (int jj = 0; jj < top; ++jj) {
        it.n_t[0] += active(it, 0, jj) ? 1 : 0;
        it.n_t[1] += active(it, 1, jj) ? 1 : 0;
      }
      it.nmax = max(it.n_t[0], it.n_t[1]);
    }
    return it;
  };
  // The S ring (FwdCfg::kSRing) serves the dense square kernels' items whose
  // Q tile 1 takes all the item's key tiles and Q tile 0 the same or all but
  // the last (every item without a mask, and under the causal mask, whose
  // tile 0 ends one key tile earlier); the others keep one S buffer per Q
  // tile.
  constexpr bool kRing = Cfg::kSRing && !kGeneral && !kSparse;
  auto ring_item = [&](const Item& it) -> bool {
    return kRing && it.nmax > 0 && it.n_t[1] == it.nmax && it.n_t[0] >= 1 &&
           it.n_t[0] >= it.nmax - 1;
  };
  // Checked build: the item's head, pair and split exist and its key tiles
  // [j0, j0 + n_t) lie inside the head's.
  auto item_ok = [&](const Item& it) -> bool {
    bool in = it.bh >= 0 && it.bh < p.BH && it.pair >= 0 && it.pair < p.n_pairs &&
              it.split >= 0 && it.split < splits && it.j0 >= 0;
    for (int t = 0; t < 2; ++t) in = in && it.n_t[t] >= 0 && it.j0 + it.n_t[t] <= p.n_kv;
    return bound_ok(in, p.status, abortf, kChkItem);
  };

  // kEpi: warps 8-11 (thread r of the warpgroup owns row r of both Q tiles'
  // O accumulators) take each O tile once the MMA thread has committed its
  // last product and the softmax warpgroup has published the rows' 1 / l:
  // O / l as bf16 into the tile's staging slot of the ring (or, for an item
  // without keys, zeros straight to memory), o_empty as soon as the tensor
  // memory reads are done, staged for the store warp.
  auto epilogue_role = [&] {
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int n_done = 0, cb = 0, n_staged = 0;
    bool ok = true;
    for (int m = 0; ok; ++m) {
      const Item item = take_item(m, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();  // every lane has read the record
      if (lane_id() == 0) release_item(m);
      if (item.idx >= num_items) break;
      if (!warp_bound_ok(item_ok(item), p.status, abortf, kChkItem)) {
        ok = false;
        break;
      }
      const bool staged = item.nmax > 0;
      const int cb_item = cb;
      if (item.nmax > 0) cb += 2 * item.nmax + ring_per_item_extra;
      for (int t = 0; t < 2 && ok; ++t) {
        const uint32_t colO = tmem + lane_base + Cfg::col_o(t);
        const int R = item.row0 + t * kTile + r;
        const bool valid = R < p.rows;
        const size_t row_g = (size_t)item.bh * p.rows + R;
        ok = mbar_wait(&sm.o_full[t], n_done & 1, p.status, abortf, kSiteOFull);
        if (ok) ok = mbar_wait(&sm.ml_full[t], n_done & 1, p.status, abortf, kSiteMlFull);
        if (ok) ok = warp_bound_ok(!valid || (R >= 0 && row_g < (size_t)p.BH * p.rows), p.status,
                                   abortf, kChkRow);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float inv_l = sm.inv_l[t][r];
        mbar_arrive(&sm.ml_empty[t]);
        const bool any = inv_l != 0.f;  // 1 / l of a row that saw a key is positive
        if (staged) {
          const int slot = (cb_item + 2 * item.nmax + t) % S;
          ok = mbar_wait(&sm.stage_ready[t], n_staged & 1, p.status, abortf, kSiteStageSlot);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orow[32];
            tmem_ld32(colO + c * 32, orow);
            tmem_wait_ld(orow);
            if (c == D / 32 - 1) {
              // O_t may now be overwritten by the next item's first product.
              tc_fence_before();
              mbar_arrive(&sm.o_empty[t]);
            }
            uint8_t* rowp = sm.kv[slot] + (c / 2) * 16384 + r * 128;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = any ? pack_bf16x2(__uint_as_float(orow[2 * i]) * inv_l,
                                       __uint_as_float(orow[2 * i + 1]) * inv_l)
                         : 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4*>(rowp + ((((c % 2) * 4 + e) ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(&sm.staged[t]);
        } else {
          // No key for any row of the item: O = 0.
          tc_fence_before();
          mbar_arrive(&sm.o_empty[t]);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + row_g * D);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (staged) ++n_staged;
      ++n_done;
    }
  };

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if constexpr (kRe) setmaxnreg_dec<Cfg::kRegsCtl>();
    if constexpr (kEpi) setmaxnreg_dec<Cfg::kEpiRegsCtl>();
    if (lane_id() == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int c = 0;         // K/V loads issued, over all items
      int q_issued = 0;  // Q pairs issued
      int n_staged = 0;  // items whose O staging uses were handed over
      bool ok = true;
      for (int m = 0; ok; ++m) {
        // Publish the next item once every role has read the record that
        // last used this ring slot.
        const int slot = m % kItemRing;
        if (m >= kItemRing && !mbar_wait(&sm.item_empty[slot], (m / kItemRing - 1) & 1,
                                         p.status, abortf, kSiteItemEmpty)) {
          ok = false;
          break;
        }
        const int idx = next_index(m);
        Item it;
        if (idx < num_items) {
          it = decode(idx);
        } else {
          it.idx = num_items;
        }
        sm.item_rec[slot] = it;
        mbar_arrive(&sm.item_full[slot]);
        if (idx >= num_items) break;
        if (!item_ok(it)) {
          ok = false;
          break;
        }
        if (it.nmax == 0) continue;  // no key visible to any row of the item
        if (q_issued > 0 &&
            !mbar_wait(&sm.q_empty, (q_issued - 1) & 1, p.status, abortf, kSiteQEmpty)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.q_full, 2 * Cfg::kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < Cfg::kBoxes; ++h)
            tma_load_3d(sm.q[t] + h * 16384, &tq, &sm.q_full, h * 64, it.row0 + t * kTile, it.bh);
        ++q_issued;
        if constexpr (kSparse) {
          // K (w = 0) or V (w = 1) of key tile jj into the next ring slot.
          auto load_kv = [&](int w, int jj) -> bool {
            if (!bound_ok(jj >= 0 && jj < p.n_kv, p.status, abortf, kChkKvTile)) return false;
            const int slot = c % S, use = c / S;
            if (use > 0 &&
                !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, p.status, abortf, kSiteKvEmpty))
              return false;
            ++c;
            mbar_arrive_expect_tx(&sm.kv_full[slot], Cfg::kTileBytes);
            if (kFp8 && w == 1) {  // V^T tile: d rows of 128 keys
              tma_load_3d(sm.kv[slot], &tv, &sm.kv_full[slot], jj * kTile, 0, it.bh);
            } else {
              for (int h = 0; h < Cfg::kBoxes; ++h)
                tma_load_3d(sm.kv[slot] + h * 16384, w == 0 ? &tk : &tv, &sm.kv_full[slot], h * 64,
                            jj * kTile, it.bh);
            }
            return true;
          };
          // Step j: K, V of query tile 0's j-th active tile, then of tile 1's.
          int cur_t[2] = {it.j0, it.j0};
          for (int j = 0; j < it.nmax && ok; ++j)
            for (int t = 0; t < 2 && ok; ++t) {
              if (j >= it.n_t[t]) continue;
              const int jj = next_tile_t(it, t, cur_t[t]);
              cur_t[t] = jj + 1;
              ok = load_kv(0, jj) && load_kv(1, jj);
            }
        } else {
          for (int j = 0; j < it.nmax && ok; ++j) {
            const int jj = it.j0 + j;
            if (!bound_ok(jj < p.n_kv, p.status, abortf, kChkKvTile)) {
              ok = false;
              break;
            }
            for (int w = 0; w < 2 && ok; ++w, ++c) {
              const int slot = c % S, use = c / S;
              if (use > 0 &&
                  !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, p.status, abortf, kSiteKvEmpty)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&sm.kv_full[slot], Cfg::kTileBytes);
              if (kFp8 && w == 1) {  // V^T tile: d rows of 128 keys
                tma_load_3d(sm.kv[slot], &tv, &sm.kv_full[slot], jj * kTile, 0, it.bh);
              } else {
                for (int h = 0; h < Cfg::kBoxes; ++h)
                  tma_load_3d(sm.kv[slot] + h * 16384, w == 0 ? &tk : &tv, &sm.kv_full[slot],
                              h * 64, jj * kTile, it.bh);
              }
            }
          }
          // The item's two O staging uses: hand the slots over empty, each
          // once the store warp has read the warpgroup's previous staged tile
          // (so that a warpgroup is never two staged tiles ahead of it).
          for (int t = 0; t < ring_per_item_extra && ok; ++t, ++c) {
            const int slot = c % S, use = c / S;
            if (use > 0 &&
                !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, p.status, abortf, kSiteKvEmpty)) {
              ok = false;
              break;
            }
            if (n_staged > 0 &&
                !mbar_wait(&sm.stored[t], (n_staged - 1) & 1, p.status, abortf, kSiteStored)) {
              ok = false;
              break;
            }
            mbar_arrive(&sm.kv_full[slot]);
            mbar_arrive(&sm.stage_ready[t]);
          }
          if (stage_epi) ++n_staged;
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        if (q_issued > 0) drain_wait(&sm.q_full, (q_issued - 1) & 1);
        for (int cc = c - 1; cc >= 0 && cc >= c - S; --cc) drain_wait(&sm.kv_full[cc % S], (cc / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (kRe) setmaxnreg_dec<Cfg::kRegsCtl>();
    if constexpr (kEpi) setmaxnreg_dec<Cfg::kEpiRegsCtl>();
    if (lane_id() == 0) {
      const uint32_t id_s = kFp8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, false, false);
      const uint32_t id_pv = kFp8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, false, true);
      const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
      uint32_t p_par[2] = {0, 0};
      int cb = 0;       // K/V loads consumed before the current item
      int n_done = 0;   // items finished by this CTA (o_full / o_empty phases)
      int q_used = 0;   // items that loaded Q (q_full / q_empty phases)
      bool ok = true;

      // S_t = Q_t K into the S buffer at column `col` (Q tile t's own, or
      // the S ring's).
      auto issue_s_at = [&](int t, int kslot, uint32_t col) {
        const uint64_t qd = desc_here(kmajor_desc(q_addr[t], 0)), kd = desc_here(kmajor_desc(smem_u32(sm.kv[kslot]), 0));
#pragma unroll
        for (int kk = 0; kk < Cfg::kKSteps; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if constexpr (kFp8)
            mma_ss_f8(tmem + col, desc_plus(qd, off), desc_plus(kd, off), id_s, kk > 0);
          else
            mma_ss(tmem + col, desc_plus(qd, off), desc_plus(kd, off), id_s, kk > 0);
        }
        tc_commit(&sm.s_full[t]);
      };
      auto issue_s = [&](int t, int kslot) { issue_s_at(t, kslot, Cfg::col_s(t)); };
      // O_t += P_t V with P_t in the S buffer at column `pcol`; the item's
      // first product overwrites O_t, so it waits until softmax t has stored
      // the previous item's O_t.
      auto issue_pv_at = [&](int t, int vslot, bool accumulate, uint32_t pcol) -> bool {
        if (!accumulate && n_done > 0) {
          if (!mbar_wait(&sm.o_empty[t], (n_done - 1) & 1, p.status, abortf, kSiteOEmpty))
            return false;
          tc_fence_after();
        }
        const uint32_t vb = smem_u32(sm.kv[vslot]);
        const uint64_t vd = desc_here(kFp8 ? kmajor_desc(vb, 0) : mnmajor_desc(vb, 0));
#pragma unroll
        for (int kk = 0; kk < Cfg::kPvSteps; ++kk) {
          if (!kFp8 && kk == Cfg::kPvSteps / 2) {
            // bf16: the second half of P (keys 64-127).
            const bool r = mbar_wait(&sm.p_full[t], p_par[t], p.status, abortf, kSitePFull);
            p_par[t] ^= 1;
            if (!r) return false;
            tc_fence_after();
          }
          // P occupies 8 TMEM columns per K-step: 16 bf16 or 32 E4M3 keys.
          if constexpr (kFp8)
            mma_ts_f8(tmem + Cfg::col_o(t), tmem + pcol + kk * 8,
                      desc_plus(vd, (kk >> 2) * 16384 + (kk & 3) * 32), id_pv,
                      (accumulate || kk > 0) ? 1u : 0u);
          else
            mma_ts(tmem + Cfg::col_o(t), tmem + pcol + kk * 8, desc_plus(vd, kk * 2048),
                   id_pv, (accumulate || kk > 0) ? 1u : 0u);
        }
        if constexpr (kRing) tc_commit(&sm.pv_done[t]);
        return true;
      };
      auto issue_pv = [&](int t, int vslot, bool accumulate) -> bool {
        return issue_pv_at(t, vslot, accumulate, Cfg::col_s(t));
      };
      auto wait_full = [&](int cnt) -> bool {
        return mbar_wait(&sm.kv_full[cnt % S], (cnt / S) & 1, p.status, abortf, kSiteKvFull);
      };
      // A Q tile without keys in this item: its O is final at once.  Softmax
      // t must first have seen the previous item's o_full[t] phase (its
      // epilogue's o_empty arrival says so): a commit right after that
      // phase could otherwise complete the next one before the softmax
      // looked, and its parity wait would then miss both.
      auto finish_empty = [&](int t) -> bool {
        if (n_done > 0 &&
            !mbar_wait(&sm.o_empty[t], (n_done - 1) & 1, p.status, abortf, kSiteOEmpty))
          return false;
        tc_commit(&sm.o_full[t]);
        return true;
      };
      // P_t ready for the next O += P V: all of it (FP8), or its first half
      // (bf16; issue_pv waits for the second half itself).
      auto wait_p = [&](int t) -> bool {
        if constexpr (kFp8) {
          const bool r = mbar_wait(&sm.p_full[t], p_par[t], p.status, abortf, kSitePFull);
          p_par[t] ^= 1;
          return r;
        } else {
          return mbar_wait(&sm.p_half[t], p_par[t], p.status, abortf, kSitePHalf);
        }
      };

      for (int m = 0; ok; ++m) {
        const Item it = take_item(m, ok);
        if (!ok) break;
        release_item(m);
        if (it.idx >= num_items) break;
        if (!item_ok(it)) {
          ok = false;
          break;
        }
        const int nmax = it.nmax;
        if constexpr (!kSparse) {
          // A Q tile without keys is final at once (its rows get O = 0).
          for (int t = 0; t < 2 && ok; ++t)
            if (it.n_t[t] == 0) ok = finish_empty(t);
          if (!ok) break;
          if (nmax == 0) {
            ++n_done;
            continue;
          }
          ok = mbar_wait(&sm.q_full, q_used & 1, p.status, abortf, kSiteQFull);
          if (ok) ok = wait_full(cb);
          if (ok && ring_item(it)) {
            // S ring: S(0,0), S(1,0) into buffers 0 and 1; at step j, as soon
            // as softmax t has the first half of P(t, j) in tensor memory
            // (so it is past its wait for S(t, j)), S(t, j+1) goes into the
            // buffer of product 2j + t - 1, whose P V is already issued, and
            // then O_t += P(t, j) V_j.  K_{j+1}'s last reader is S(1, j+1),
            // V_j's is PV(1, j).
            tc_fence_after();
            issue_s_at(0, cb % S, Cfg::col_buf(0));
            issue_s_at(1, cb % S, Cfg::col_buf(1));
            tc_commit(&sm.kv_empty[cb % S]);
            if (nmax == 1) tc_commit(&sm.q_empty);
            for (int j = 0; j < nmax && ok; ++j) {
              const int vc = cb + 2 * j + 1, kc = cb + 2 * j + 2;
              ok = wait_full(vc) && (j + 1 >= nmax || wait_full(kc));
              for (int t = 0; t < 2 && ok; ++t) {
                if (j >= it.n_t[t]) continue;  // Q tile 0 of a causal item: no last step
                ok = wait_p(t);
                if (!ok) break;
                tc_fence_after();
                if (j + 1 < it.n_t[t]) {
                  issue_s_at(t, kc % S, Cfg::col_buf((2 * j + t + 2) % 3));
                  if (t == 1) {
                    tc_commit(&sm.kv_empty[kc % S]);
                    if (j + 1 == nmax - 1) tc_commit(&sm.q_empty);  // last product reading Q
                  }
                }
                ok = issue_pv_at(t, vc % S, j > 0, Cfg::col_buf((2 * j + t) % 3));
                if (!ok) break;
                if (j == it.n_t[t] - 1) tc_commit(&sm.o_full[t]);
              }
              if (ok) tc_commit(&sm.kv_empty[vc % S]);
            }
            cb += 2 * nmax + ring_per_item_extra;
            ++q_used;
            ++n_done;
            continue;
          }
          if (ok) {
            tc_fence_after();
            for (int t = 0; t < 2; ++t)
              if (it.n_t[t] > 0) issue_s(t, cb % S);
            tc_commit(&sm.kv_empty[cb % S]);
            if (nmax == 1) tc_commit(&sm.q_empty);
          }
          // Key tile j: PV_t(j-1) then S_t(j) for each Q tile that has them.
          for (int j = 1; j < nmax && ok; ++j) {
            const int kc = cb + 2 * j, vc = cb + 2 * j - 1;
            ok = wait_full(kc) && wait_full(vc);
            if (!ok) break;
            for (int t = 0; t < 2 && ok; ++t) {
              if (j - 1 >= it.n_t[t]) continue;
              ok = wait_p(t);
              if (!ok) break;
              tc_fence_after();
              ok = issue_pv(t, vc % S, j - 1 > 0);
              if (!ok) break;
              if (j < it.n_t[t]) {
                issue_s(t, kc % S);
              } else {
                tc_commit(&sm.o_full[t]);  // tile t has no more keys
              }
            }
            if (!ok) break;
            tc_commit(&sm.kv_empty[vc % S]);
            tc_commit(&sm.kv_empty[kc % S]);
            if (j == nmax - 1) tc_commit(&sm.q_empty);  // last product reading Q
          }
          if (ok) {
            const int vc = cb + 2 * nmax - 1;
            ok = wait_full(vc);
            for (int t = 0; t < 2 && ok; ++t) {
              if (it.n_t[t] != nmax) continue;
              ok = wait_p(t);
              if (!ok) break;
              tc_fence_after();
              ok = issue_pv(t, vc % S, nmax - 1 > 0);
              if (ok) tc_commit(&sm.o_full[t]);
            }
            if (ok) tc_commit(&sm.kv_empty[vc % S]);
          }
          cb += 2 * nmax + ring_per_item_extra;
        } else {
          // Block-sparse: Q tile t walks its own n_t[t] active key tiles.
          // Step j's loads are K and V of tile 0's j-th tile, then of tile
          // 1's (for the tiles that have one), so the load index of each
          // product follows from the counts alone.
          for (int t = 0; t < 2 && ok; ++t)
            if (it.n_t[t] == 0) ok = finish_empty(t);
          if (!ok) break;
          if (nmax == 0) {
            ++n_done;
            continue;
          }
          int base = cb;                    // first load of the next step
          int ks[2] = {0, 0}, vs[2] = {0, 0};  // this step's K and V loads per tile
          int vp[2] = {0, 0};               // the previous step's V loads
          auto step_loads = [&](int j) {
            for (int t = 0; t < 2; ++t)
              if (j < it.n_t[t]) {
                ks[t] = base;
                vs[t] = base + 1;
                base += 2;
              }
          };
          ok = mbar_wait(&sm.q_full, q_used & 1, p.status, abortf, kSiteQFull);
          step_loads(0);
          for (int t = 0; t < 2 && ok; ++t) {
            if (it.n_t[t] == 0) continue;
            ok = wait_full(ks[t]);
            if (!ok) break;
            tc_fence_after();
            issue_s(t, ks[t] % S);
            tc_commit(&sm.kv_empty[ks[t] % S]);
          }
          if (ok && nmax == 1) tc_commit(&sm.q_empty);
          for (int j = 1; j < nmax && ok; ++j) {
            vp[0] = vs[0];
            vp[1] = vs[1];
            step_loads(j);
            for (int t = 0; t < 2 && ok; ++t) {
              if (j - 1 < it.n_t[t]) {  // P V of tile t's (j-1)-th key tile
                ok = wait_p(t) && wait_full(vp[t]);
                if (!ok) break;
                tc_fence_after();
                ok = issue_pv(t, vp[t] % S, j - 1 > 0);
                if (!ok) break;
                tc_commit(&sm.kv_empty[vp[t] % S]);
                if (j - 1 == it.n_t[t] - 1) tc_commit(&sm.o_full[t]);  // no more keys
              }
              if (j < it.n_t[t]) {  // S of tile t's j-th key tile
                ok = wait_full(ks[t]);
                if (!ok) break;
                tc_fence_after();
                issue_s(t, ks[t] % S);
                tc_commit(&sm.kv_empty[ks[t] % S]);
              }
            }
            if (ok && j == nmax - 1) tc_commit(&sm.q_empty);  // last product reading Q
          }
          for (int t = 0; t < 2 && ok; ++t) {
            if (nmax - 1 >= it.n_t[t]) continue;
            ok = wait_p(t) && wait_full(vs[t]);
            if (!ok) break;
            tc_fence_after();
            ok = issue_pv(t, vs[t] % S, nmax - 1 > 0);
            if (!ok) break;
            tc_commit(&sm.kv_empty[vs[t] % S]);
            tc_commit(&sm.o_full[t]);
          }
          cb = base;
        }
        ++q_used;
        ++n_done;
      }
      // Every MMA issued so far must finish before TMEM is released.
      tc_commit(&sm.drain);
      drain_wait(&sm.drain, 0);
    }
    __syncwarp();
  } else if (warp == kWarpStore) {
    // ------------------------------------------------------------ O store warp
    if constexpr (kRe) setmaxnreg_dec<Cfg::kRegsCtl>();
    if constexpr (kEpi) setmaxnreg_dec<Cfg::kEpiRegsCtl>();
    // Sends each staged O tile out with TMA stores (rows past the tensor's
    // end are not written) and releases its ring slot once the stores have
    // read it.
    if (lane_id() == 0 && stage_epi) {
      int cb = 0, n_staged = 0;
      bool ok = true;
      for (int m = 0; ok; ++m) {
        const Item it = take_item(m, ok);
        if (!ok) break;
        release_item(m);
        if (it.idx >= num_items) break;
        if (!item_ok(it)) {
          ok = false;
          break;
        }
        if (it.nmax == 0) continue;
        for (int t = 0; t < 2 && ok; ++t) {
          const int use = cb + 2 * it.nmax + t;
          const int slot = use % S;
          if (!mbar_wait_sleep(&sm.staged[t], n_staged & 1, p.status, abortf, kSiteStaged)) {
            ok = false;
            break;
          }
          for (int h = 0; h < Cfg::kBoxes; ++h)
            tma_store_3d(&to, sm.kv[slot] + h * 16384, h * 64, it.row0 + t * kTile, it.bh);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&sm.stored[t]);
          mbar_arrive(&sm.kv_empty[slot]);
        }
        ++n_staged;
        cb += 2 * it.nmax + ring_per_item_extra;
      }
      // The stores must be complete before the CTA exits.
      bulk_wait_group0();
    }
    __syncwarp();
  } else if ((kRe && warp == 11) || (kEpi && warp == 15)) {
    // Idle: its registers go to the softmax warpgroups.
    if constexpr (kRe) setmaxnreg_dec<Cfg::kRegsCtl>();
    if constexpr (kEpi) setmaxnreg_dec<Cfg::kEpiRegsCtl>();
  } else if (kEpi && warp >= 8) {
    // ------------------------------------------------------------ epilogue
    if constexpr (kEpi) {
      setmaxnreg_dec<Cfg::kEpiRegsEpi>();
      epilogue_role();
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    if constexpr (kRe) setmaxnreg_inc<Cfg::kRegsSoftmax>();
    if constexpr (kEpi) setmaxnreg_inc<Cfg::kEpiRegsSoftmax>();
    const int t = warp >> 2;             // which Q tile
    const int r = tid & 127;             // row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float c2 = p.scale_log2;  // nonzero: a zero scale arrives as a tiny positive one
    const float ninf = __int_as_float(0xff800000);
    const uint32_t colS = tmem + lane_base + Cfg::col_s(t);
    const uint32_t colO = tmem + lane_base + Cfg::col_o(t);
    uint32_t s_par = 0;
    int n_done = 0;
    int cb = 0;        // ring uses before the current item (as the MMA thread counts them)
    int n_staged = 0;  // this warpgroup's O tiles handed to the store warp
    int n_pv = 0;      // kRing: O_t += P_t V products before this step, over all items
    bool ok = true;

    for (int m = 0; ok; ++m) {
      const Item item = take_item(m, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();  // every lane has read the record
      if (lane_id() == 0) release_item(m);
      if (item.idx >= num_items) break;
      if (!warp_bound_ok(item_ok(item), p.status, abortf, kChkItem)) {
        ok = false;
        break;
      }
      const int bh = item.bh;
      const int n_t = item.n_t[t];
      const bool ring = ring_item(item);
      // This tile's O staging use of the ring, when the item has one.
      const bool staged = stage_epi && item.nmax > 0;
      const int stage_use = cb + 2 * item.nmax + t;
      if (item.nmax > 0) cb += 2 * item.nmax + ring_per_item_extra;
      float o_mul = 1.f;  // FP8: the V scale, applied with 1 / l
      if constexpr (kFp8) {
        // Scores of codes carry the Q and K scales (and d, the squared norm
        // of the Hadamard rotation's rows); fold them into the exponent.
        auto descale = [&](int which) {
          const float a = p.fp8_amax[which * p.BH + bh];
          return a == 0.f ? 1.f : a / 448.f;
        };
        c2 = p.scale_log2 * descale(0) * descale(1);
        if (p.fp8_hadamard) c2 *= 1.f / (float)D;
        if (c2 == 0.f) c2 = kNeg ? -1.17549435e-38f : 1.17549435e-38f;
        o_mul = descale(2);
      }
      const int R = item.row0 + t * kTile + r;  // packed query row of this K/V head
      // Keys visible to this row: [0, lim) (bottom-right causal alignment).
      int lim = p.Nkv;
      if (p.causal)
        lim = kGeneral ? min(max(R % p.Nq + p.causal_off + 1, 0), p.Nkv) : min(R + 1, p.Nkv);
      float m_ref = ninf;
      float l = 0.f;
      int cur = item.j0;
      for (int j = 0; j < n_t; ++j) {
        const int jj = next_tile_t(item, t, cur);  // key tile
        cur = jj + 1;
        if (!warp_bound_ok(jj >= 0 && jj < p.n_kv, p.status, abortf, kChkKvTile)) {
          ok = false;
          break;
        }
        // Columns >= tlim of this key tile are masked for this row.
        const int tlim = lim - jj * kTile;
        ok = mbar_wait(&sm.s_full[t], s_par, p.status, abortf, kSiteSFull);
        ok = __all_sync(0xffffffffu, ok);  // keep the warp's collective TMEM ops converged
        s_par ^= 1;
        if (!ok) break;
        tc_fence_after();
        // S ring: step j's S is product 2j + t of the item, in buffer (2j + t) % 3;
        // it may have completed before the previous P V, which a rescale of O
        // must wait for.
        const uint32_t colSj =
            ring ? tmem + lane_base + Cfg::col_buf((2 * j + t) % 3) : colS;
        softmax_tile_w<D, kNeg, kFp8>(colSj, colO, c2, tlim, j > 0, m_ref, l,
                                      [&] { mbar_arrive(&sm.p_half[t]); },
                                      [&] {
                                        if constexpr (kRing)
                                          (void)mbar_wait(&sm.pv_done[t], (n_pv - 1) & 1, p.status,
                                                          abortf, kSitePvDone);
                                      });
        if constexpr (kRing) ++n_pv;
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
      }
      if constexpr (kEpi) {
        // The epilogue warpgroup takes O; this warpgroup writes lse and
        // hands over 1 / l (0 for a row that saw no key).
        const bool any = l > 0.f;
        const bool valid = R < p.rows;
        const size_t row_g = (size_t)bh * p.rows + R;
        if (ok && n_done > 0)
          ok = mbar_wait(&sm.ml_empty[t], (n_done - 1) & 1, p.status, abortf, kSiteMlEmpty);
        if (ok) ok = warp_bound_ok(!valid || (R >= 0 && row_g < (size_t)p.BH * p.rows), p.status,
                                   abortf, kChkRow);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (valid) p.lse[row_g] = any ? (m_ref + __log2f(l)) * kLn2 : ninf;
        sm.inv_l[t][r] = any ? o_mul / l : 0.f;
        mbar_arrive(&sm.ml_full[t]);
        ++n_done;
        continue;
      }
      if (ok) ok = mbar_wait(&sm.o_full[t], n_done & 1, p.status, abortf, kSiteOFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // Epilogue: O / l (0 for a row that saw no key) and lse; with several
      // key splits, the split's normalised fp32 O and its lse, for the combine.
      const bool any = l > 0.f;
      const float inv_l = any ? o_mul / l : 0.f;
      const bool valid = R < p.rows;
      const size_t row_g = (size_t)bh * p.rows + R;
      if (!warp_bound_ok(!valid || (R >= 0 && row_g < (size_t)p.BH * p.rows), p.status, abortf,
                         kChkRow)) {
        ok = false;
        break;
      }
      if (staged) {
        const int slot = stage_use % S;
        ok = mbar_wait(&sm.stage_ready[t], n_staged & 1, p.status, abortf, kSiteStageSlot);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // Row r of the tile in the 128B-swizzled layout of the TMA boxes
        // (64 columns each): 16-byte chunk ch of the row at ch ^ (r % 8).
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orow[32];
          tmem_ld32(colO + c * 32, orow);
          tmem_wait_ld(orow);
          uint8_t* rowp = sm.kv[slot] + (c / 2) * 16384 + r * 128;
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = any ? pack_bf16x2(__uint_as_float(orow[2 * i]) * inv_l,
                                     __uint_as_float(orow[2 * i + 1]) * inv_l)
                       : 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(rowp + ((((c % 2) * 4 + e) ^ (r & 7)) << 4)) =
                make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
        fence_proxy_async_smem();
        // O_t may now be overwritten by the next item's first product, and
        // the staged tile stored.
        tc_fence_before();
        mbar_arrive(&sm.o_empty[t]);
        mbar_arrive(&sm.staged[t]);
        if (valid) p.lse[row_g] = any ? (m_ref + __log2f(l)) * kLn2 : ninf;
        ++n_staged;
        ++n_done;
        continue;
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orow[32];
        tmem_ld32(colO + c * 32, orow);
        tmem_wait_ld(orow);
        if (!valid) continue;
        if (splits == 1) {
          uint4 v[4];
          uint32_t* w = reinterpret_cast<uint32_t*>(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = any ? pack_bf16x2(__uint_as_float(orow[2 * i]) * inv_l,
                                     __uint_as_float(orow[2 * i + 1]) * inv_l)
                       : 0u;
          uint4* dst =
              reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + row_g * D + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = v[i];
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.o_part + ((size_t)item.split * p.BH * p.rows + row_g) * D + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = any ? make_float4(__uint_as_float(orow[4 * i]) * inv_l,
                                       __uint_as_float(orow[4 * i + 1]) * inv_l,
                                       __uint_as_float(orow[4 * i + 2]) * inv_l,
                                       __uint_as_float(orow[4 * i + 3]) * inv_l)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (valid) {
        const float lse_row = any ? (m_ref + __log2f(l)) * kLn2 : ninf;
        if (splits == 1)
          p.lse[row_g] = lse_row;
        else
          p.lse_part[(size_t)item.split * p.BH * p.rows + row_g] = lse_row;
      }
      // O_t may now be overwritten by the next item's first product.
      tc_fence_before();
      mbar_arrive(&sm.o_empty[t]);
      ++n_done;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  if (dyn && tid == 0) {
    // This CTA's claims are over (the producer made them before the barrier
    // above): count the CTA out, and the last one out zeroes the counter
    // for the next launch on the stream.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == G - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

// Merge the key splits of the general forward pass: per row,
// lse = ln sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s (the split-KV
// combine of cs2680 Lecture 9 sec. 9.8, the rescaling of sec. 9.4).  One
// warp per row; lane l owns the d/32 consecutive columns starting at
// l * d/32.  The split lse values are read 32 at a time, one per lane, and
// reduced across the warp; the split O rows are then read eight splits at a
// time with all eight loads in flight, so a row costs a few memory
// latencies rather than one per split.
template <int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const FwdParams p) {
  wait_prior_grid();  // the forward kernel's split results
  constexpr int kPer = D / 32;  // 4 or 2 columns per lane
  constexpr int kBatch = 8;     // split O rows loaded together
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows_total = (long long)p.BH * p.rows;
  if (row >= rows_total) return;  // whole warps: row is uniform in a warp
  const float ninf = __int_as_float(0xff800000);
  constexpr float kL2e = 1.4426950408889634f;
  const int S = p.splits;
  int no_abort = 0;
  if (!bound_ok(S >= 1 && row >= 0, p.status, &no_abort, kChkCombine)) return;
  const float* lse_row_s = p.lse_part + row;  // split s at lse_row_s[s * rows_total]
  float m = ninf;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lse_row_s[s * rows_total]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float lse_row = ninf;
  if (m != ninf) {
    float sum = 0.f;
    for (int s = lane; s < S; s += 32) sum += exp2f((lse_row_s[s * rows_total] - m) * kL2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse_row = m + logf(sum);
    for (int s0 = 0; s0 < S; s0 += 32) {
      // Lane u's weight is split s0 + u's; a split with weight 0 adds nothing.
      const float wl =
          s0 + lane < S ? exp2f((lse_row_s[(s0 + lane) * rows_total] - lse_row) * kL2e) : 0.f;
      const int n = min(32, S - s0);
      for (int u0 = 0; u0 < n; u0 += kBatch) {
        float v[kBatch][kPer];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const float* src = p.o_part + ((s0 + u0 + b) * rows_total + row) * D + lane * kPer;
#pragma unroll
          for (int i = 0; i < kPer; ++i) v[b][i] = 0.f;
          if (u0 + b < n) {
            if constexpr (kPer == 4) {
              const float4 x = *reinterpret_cast<const float4*>(src);
              v[b][0] = x.x, v[b][1] = x.y, v[b][kPer - 2] = x.z, v[b][kPer - 1] = x.w;
            } else {
              const float2 x = *reinterpret_cast<const float2*>(src);
              v[b][0] = x.x, v[b][1] = x.y;
            }
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const float w = __shfl_sync(0xffffffffu, wl, (u0 + b) & 31);
          if (u0 + b < n && w != 0.f) {
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc[i] += w * v[b][i];
          }
        }
      }
    }
  }
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + (size_t)row * D + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[kPer - 2], acc[kPer - 1]);
    *reinterpret_cast<uint2*>(dst) = out;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
  }
  if (lane == 0) p.lse[row] = lse_row;
}

template <int D, bool kNeg, bool kGeneral, bool kSparse, bool kFp8, bool kStage, bool kDyn>
int launch_fwd_dn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& to, const FwdParams& p, cudaStream_t stream) {
  if (kDyn != (p.sched != nullptr)) return FA_ERR_LAUNCH;
  static_assert(sizeof(FwdSmem<D, kFp8>) + 1024 <= 232448,
                "forward shared memory above the 227 KB a CTA may have");
  const size_t smem = sizeof(FwdSmem<D, kFp8>) + 1024;
  if (cudaFuncSetAttribute(fa_fwd_kernel<D, kNeg, kGeneral, kSparse, kFp8, kStage, kDyn>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if constexpr (FwdCfg<D, kFp8>::realloc(kStage) || FwdCfg<D, kFp8>::epi(kStage)) {
    // The softmax warpgroups' setmaxnreg.inc waits for the registers the
    // other warpgroups release, which suffice only at the launch register
    // count the split assumes: refuse to launch otherwise.
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, fa_fwd_kernel<D, kNeg, kGeneral, kSparse, kFp8, kStage, kDyn>) !=
            cudaSuccess ||
        attr.numRegs < (FwdCfg<D, kFp8>::epi(kStage) ? FwdCfg<D, kFp8>::kEpiRegsLaunch
                                                     : FwdCfg<D, kFp8>::kRegsLaunch))
      return FA_ERR_LAUNCH;
  }
  // Launched with programmatic stream serialization: the kernel's launch
  // and setup overlap the end of the previous kernel on the stream, and it
  // waits for that kernel (wait_prior_grid) before reading any input.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3((unsigned)p.grid, 1, 1);
  c.blockDim = dim3(FwdCfg<D, kFp8>::threads(kStage), 1, 1);
  c.dynamicSmemBytes = smem;
  c.stream = stream;
  c.attrs = pdl;
  c.numAttrs = 1;
  if (cudaLaunchKernelEx(&c, fa_fwd_kernel<D, kNeg, kGeneral, kSparse, kFp8, kStage, kDyn>, tq, tk, tv, to,
                         p) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  if (p.splits > 1) {
    const long long threads = (long long)p.BH * p.rows * 32;
    c.gridDim = dim3((unsigned)((threads + 255) / 256), 1, 1);
    c.blockDim = dim3(256, 1, 1);
    c.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&c, fa_combine_kernel<D>, p) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
  }
  return FA_OK;
}

// The kernel for the sign of the scale (kNeg: a negative scale turns the
// row maximum into a minimum).
template <int D, bool kGeneral, bool kSparse, bool kFp8, bool kStage, bool kDyn>
int launch_fwd_signed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& to, const FwdParams& p, cudaStream_t stream) {
  if (p.scale_log2 < 0.f)
    return launch_fwd_dn<D, true, kGeneral, kSparse, kFp8, kStage, kDyn>(tq, tk, tv, to, p, stream);
  return launch_fwd_dn<D, false, kGeneral, kSparse, kFp8, kStage, kDyn>(tq, tk, tv, to, p, stream);
}

template <int D>
int launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& to, FwdParams p, cudaStream_t stream) {
  // A zero scale makes every unmasked probability equal; it runs as the
  // smallest normal positive scale, whose exponents round to exactly 0.
  if (p.scale_log2 == 0.f) p.scale_log2 = 1.17549435e-38f;
  const bool general = p.splits > 1 || p.Nq != p.rows || p.Nkv != p.rows;
  const bool dyn = p.sched != nullptr;
  if (p.fp8_amax) {  // square case, d = 128 only (checked by the caller); static split
    if constexpr (D == 128) {
      if (dyn) return FA_ERR_LAUNCH;
      return launch_fwd_signed<D, false, false, true, false, false>(tq, tk, tv, to, p, stream);
    }
    return FA_ERR_UNSUPPORTED_D;
  }
  if (p.block_mask) {  // square case only (checked by the caller)
    if (dyn) return launch_fwd_signed<D, false, true, false, false, true>(tq, tk, tv, to, p, stream);
    return launch_fwd_signed<D, false, true, false, false, false>(tq, tk, tv, to, p, stream);
  }
  if (general) {
    if (dyn) return launch_fwd_signed<D, true, false, false, false, true>(tq, tk, tv, to, p, stream);
    return launch_fwd_signed<D, true, false, false, false, false>(tq, tk, tv, to, p, stream);
  }
  // Staged O stores (at d = 128 with the epilogue warpgroup) pay at every
  // length; they need persistent CTAs (more items than CTAs).
  const long long items = (long long)p.BH * p.n_pairs;
  if (p.grid < items) {
    if (dyn) return launch_fwd_signed<D, false, false, false, true, true>(tq, tk, tv, to, p, stream);
    return launch_fwd_signed<D, false, false, false, true, false>(tq, tk, tv, to, p, stream);
  }
  if (dyn) return FA_ERR_LAUNCH;  // a work counter comes with a persistent grid
  return launch_fwd_signed<D, false, false, false, false, false>(tq, tk, tv, to, p, stream);
}

}  // namespace

int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_fwd_d<128>(tq, tk, tv, to, p, stream);
  if (d == 64) return launch_fwd_d<64>(tq, tk, tv, to, p, stream);
  return FA_ERR_UNSUPPORTED_D;
}

}  // namespace fa
