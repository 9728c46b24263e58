// fa_bwd.cu -- backward pass of exact attention on sm_103a, by recomputation.
//
// The forward pass kept only O and the per-row logsumexp; this pass
// recomputes the scores and probabilities tile by tile on chip from Q, K, V
// and lse instead of reading a stored N x N matrix (cs2680 Lecture 9,
// sec. 9.6; "Reading CMU 11-868 LLM Systems: FlashAttention", slide page 14).
// The gradient formulas are the softmax Jacobian (the pages print none):
//     P = exp(scale Q K^T - lse),  dV = P^T dO,  dP = dO V^T,
//     D_i = sum_k dO_ik O_ik,  dS = P o (dP - D),
//     dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels:
//   1. prep: per row -D_i and -lse_i * log2(e) into the workspace, negated
//      so that the main kernel adds them (padded rows get 0 and -inf, which
//      makes their probabilities exactly 0), the fp32 dQ accumulator zeroed
//      and the main kernel's work-item counter reset.  HBM-bound.
//   2. main: one persistent CTA per SM; a work item is (head, 128-key tile
//      j), claimed from the counter in longest-first list order when the CTA
//      is ready for one.  K_j, V_j stay in shared memory; dK_j, dV_j
//      accumulate in tensor memory while the CTA walks the query tiles i
//      (all of them, or i >= j under a causal mask).  The next item's K and
//      V load as soon as the last product has read the current ones, and
//      its first products run while the compute warps store dK_j, dV_j.
//      Per step:
//        S^T  = K_j Q_i^T           (tcgen05, both operands in smem)
//        dP^T = V_j dO_i^T
//        P^T  = exp2(S^T c - lse_i log2 e)  -> bf16 in TMEM over S^T
//               (masked scores replaced by the value whose exponent is -inf)
//        dV  += P^T dO_i                    (A operand from TMEM)
//        dS^T = P^T o (dP^T - D_i)          -> bf16 in smem (128B swizzle)
//        dQ_i = dS K_j  -> TMEM (over dP^T) -> fp32 vector atomics into the
//                          workspace, by the compute warpgroups, spread
//                          over the next step
//        dK  += dS^T Q_i                   (A operand from TMEM)
//   3. convert: dQ = bf16(scale * accumulator).
//
// Warp roles of the main kernel (640 threads):
//   warps 0-15 compute: four warpgroups, warpgroup g owning query columns
//              [32g, 32g+32) (thread r owns key row r of the tile): P, dS,
//              then d/4 of dQ_i's columns from TMEM to the fp32 accumulator
//              with atomic adds (part of them held in registers until the
//              next step's P and dS phases); finally the epilogue
//              (warpgroups 0-1 store halves of dV, 2-3 halves of dK).  Four compute warps per SM
//              sub-partition hide the latency of the exponent and dS phases
//              better than two (measured +3% at d = 128, +7% at d = 64).
//   warp 16    TMA producer;  warp 17 MMA issuer and TMEM owner;
//   warps 18-19 idle: they complete the fifth warpgroup, which gives its
//              registers to the compute warpgroups (setmaxnreg: five warps
//              per SM sub-partition cap a thread at 96 registers at launch;
//              the compute warps then run with 104, the others with 56).
// Tensor memory: [0,128) S^T; warpgroup g's 32 columns [32g, 32g+32) take
// P^T (bf16 pairs) over their first 16 and dS^T over the last 16, so that
// dV += P^T dO and dK += dS^T Q take their A operand from tensor memory;
// [128,256) dP^T, then dQ; [256,256+d) dV; [256+d, 256+2d) dK.  At d = 64
// the free columns [384,512) are a second S^T region: step i+1's S^T is
// issued right after step i's dP^T, the compute warps run P(i+1) while the
// tensor core does dK(i) and dQ(i), and read dQ(i) out after P(i+1).
#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x d bf16 tile
  static constexpr int kStages = 2;                  // Q/dO ring
  static constexpr int kWG = 4;                      // compute warpgroups
  static constexpr int kQ = kTile / kWG;             // query columns per warpgroup
  static constexpr int kThreads = kWG * 128 + 128;   // compute, producer, MMA, 2 idle
  // Registers per thread at launch, after the fifth warpgroup's setmaxnreg.dec
  // and after the compute warpgroups' setmaxnreg.inc; the split must fit in
  // the launch's registers, or the increase would wait forever.
  static constexpr int kRegsLaunch = 96, kRegsCtl = 64, kRegsCompute = 104;
  static_assert(kWG * 128 * kRegsCompute + 128 * kRegsCtl <= kThreads * kRegsLaunch,
                "register split above the launch's total");
  static constexpr int kWarpLoad = kWG * 4, kWarpMma = kWG * 4 + 1;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  // d = 64 leaves 128 columns free: a second S^T region, so that the next
  // step's S^T and P phase overlap this step's dK and dQ products.
  static constexpr bool kDbl = D == 64;
  static constexpr uint32_t kColS2 = 256 + 2 * D;
};

template <int D>
struct BwdSmem {
  uint8_t k[BwdCfg<D>::kTileBytes];
  uint8_t v[BwdCfg<D>::kTileBytes];
  uint8_t q[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  uint8_t dO[BwdCfg<D>::kStages][BwdCfg<D>::kTileBytes];
  uint8_t ds[kTile * kTile * 2];  // dS^T [key][query] bf16, 128B swizzle
  float lse2[BwdCfg<D>::kStages][kTile];
  float delta[BwdCfg<D>::kStages][kTile];
  uint64_t kv_full, kv_empty;
  uint64_t item_full[2], item_empty[2];  // work-item handoff from the producer
  int item_idx[2];
  uint64_t q_full[BwdCfg<D>::kStages];
  uint64_t q_empty[BwdCfg<D>::kStages];
  uint64_t s_full[2];  // per S^T region (one region unless BwdCfg::kDbl)
  uint64_t dp_full, p_ready, ds_ready, dq_full, dq_empty, acc_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};


enum : int {
  kSiteKvFull = 201, kSiteQFull, kSiteQEmpty, kSiteSFull, kSiteDpFull, kSitePReady,
  kSiteDsReady, kSiteDqFull, kSiteDqEmpty, kSiteAccFull, kSiteAlign, kSiteKvEmpty,
  kSiteItemFull, kSiteItemEmpty
};
// Bounds checks of the checked build (FA_CHECKS).
enum : int {
  kChkItem = 1201,  // a work item's head, key tile or step count
  kChkQTile,        // a query tile a key tile visits
  kChkDqRow,        // a row of the dQ accumulator
  kChkKvRow,        // a key row of dK / dV
  kChkPrepRow,      // a row of the prep kernel
  kChkConvRow,      // a row of the convert kernel
  kChkMask          // an entry of the block mask
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, 16384, 1024);
}
// Byte offsets of K-step kk in a K-major tile and in an MN-major tile.
__host__ __device__ constexpr uint32_t kmajor_off(int kk) { return (kk >> 2) * 16384 + (kk & 3) * 32; }
__host__ __device__ constexpr uint32_t mnmajor_off(int kk) { return kk * 2048; }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > 100000000ull) return;
  }
}

// Non-tensor bulk copy global -> shared, completing `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Work order of the main kernel: heads in groups of kHeadGroup; inside a
// group the key tiles go first to last (under a causal mask key tile j
// visits n_kv - j query tiles, so the longest work items start first).
__device__ __forceinline__ void bwd_item(int t, int BH, int n_kv, int* bh, int* j) {
  const int per_group = kHeadGroup * n_kv;
  const int g = t / per_group;
  const int gsize = (BH - g * kHeadGroup) < kHeadGroup ? (BH - g * kHeadGroup) : kHeadGroup;
  const int idx = t - g * per_group;
  *j = idx / gsize;
  *bh = g * kHeadGroup + idx % gsize;
}

// Address (in floats) of element (row, 4*c4 .. 4*c4+3) of the dQ accumulator.
// The accumulator is blocked per 128-row tile as [tile][d/4][128][4] so that
// the 32 rows of a warp add to 512 contiguous bytes.
template <int D>
__device__ __forceinline__ size_t dqacc_index(int bh, int n_kv, int row, int c4) {
  const int tile = row >> 7, r = row & 127;
  return ((((size_t)bh * n_kv + tile) * (D / 4) + c4) * kTile + r) * 4;
}

// ------------------------------------------------------------------ prep

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdParams p) {
  wait_prior_grid();  // O (and the workspace) belong to the previous kernel until it ends
  constexpr int kLanesPerRow = D / 8;  // 16-byte loads of 8 bf16
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.sched = 0;
  const int npad = p.n_kv * kTile;
  const long long total_rows = (long long)p.BH * npad;
  const long long row_g = (long long)warp_global * kRowsPerWarp + lane / kLanesPerRow;
  const int sub = lane % kLanesPerRow;
  float acc = 0.f;
  int bh = 0, row = 0;
  bool in_range = row_g < total_rows;
  if (in_range) {
    bh = (int)(row_g / npad);
    row = (int)(row_g % npad);
    int no_abort = 0;
    in_range = bound_ok(bh < p.BH && row < npad, p.status, &no_abort, kChkPrepRow);
  }
  if (in_range) {
    if (row < p.N) {
      const size_t off = ((size_t)bh * p.N + row) * D + sub * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.o) + off);
      const uint4 b = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.dout) + off);
      const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa2 = __bfloat1622float2(ha[i]);
        const float2 fb2 = __bfloat1622float2(hb[i]);
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
    }
  }
#pragma unroll
  for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (in_range) {
    if (sub == 0) {
      const size_t ri = (size_t)bh * npad + row;
      p.delta[ri] = -acc;
      p.lse2[ri] = row < p.N ? -(p.lse[(size_t)bh * p.N + row] * kLog2e) : __int_as_float(0xff800000);
    }
  }
  // Zero the dQ accumulator (BH * npad * D floats, contiguous) with
  // consecutive threads on consecutive 16-byte words.
  const size_t n4 = (size_t)p.BH * npad * (D / 4);
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x)
    acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ convert

// One CTA per (head, 128-row tile, 64 columns): the accumulator's block of
// [16 column groups][128 rows][4] floats is read with consecutive threads on
// consecutive 16-byte words, turned into rows in shared memory (one word of
// padding per row keeps eight consecutive rows on different banks), and
// written out as rows of bf16, eight threads per 128-byte row segment.
constexpr int kConvThreads = 256;
template <int D>
__global__ void __launch_bounds__(kConvThreads) fa_bwd_convert_kernel(const BwdParams p) {
  wait_prior_grid();  // the main kernel's dQ reductions
  constexpr int kGroups = 16;  // float4 column groups per CTA (64 columns)
  constexpr int kHalves = D / 64;
  __shared__ float4 buf[kTile][kGroups + 1];
  const int half = blockIdx.x % kHalves;
  const int tile = (blockIdx.x / kHalves) % p.n_kv;
  const int bh = blockIdx.x / kHalves / p.n_kv;
  int no_abort = 0;
  if (!bound_ok(bh < p.BH, p.status, &no_abort, kChkConvRow)) return;
  const float4* src = reinterpret_cast<const float4*>(
      p.dq_acc + dqacc_index<D>(bh, p.n_kv, tile * kTile, half * kGroups));
#pragma unroll
  for (int k = 0; k < kTile * kGroups / kConvThreads; ++k) {
    const int idx = threadIdx.x + k * kConvThreads;  // = group * 128 + row
    buf[idx % kTile][idx / kTile] = src[idx];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kTile * 8 / kConvThreads; ++k) {
    const int idx = threadIdx.x + k * kConvThreads;
    const int r = idx / 8, q = idx % 8;  // row, 8-column chunk
    const int row = tile * kTile + r;
    if (row >= p.N) continue;
    const float4 a = buf[r][2 * q], b = buf[r][2 * q + 1];
    uint4 out;
    out.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    out.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    out.z = pack_bf16x2(b.x * p.scale, b.y * p.scale);
    out.w = pack_bf16x2(b.z * p.scale, b.w * p.scale);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq) +
                              ((size_t)bh * p.N + row) * D + half * 64 + q * 8) = out;
  }
}

// ------------------------------------------------------------------ main

// kSparse: a block mask over (128-query tile, 128-key tile) pairs; key tile
// j visits only the query tiles i whose block (i, j) is active.
template <int D, bool kSparse>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                       const BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int NS = Cfg::kStages;
  constexpr int kWarpLoad = Cfg::kWarpLoad, kWarpMma = Cfg::kWarpMma;
  constexpr int kWG = Cfg::kWG, kQ = Cfg::kQ;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The swizzled tiles need 1024-byte alignment; the dynamic window starts
  // there on this architecture, and the size leaves no slack to realign.
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) {
      atomicCAS(p.status, 0, FA_ERR_LAUNCH);
      atomicCAS(p.status + 1, 0, kSiteAlign);
    }
    return;
  }
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  volatile int* abortf = &sm.abort_flag;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], 1 + kWG * 4);  // the MMA thread and every compute warp
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.p_ready, kWG * 128);
    mbar_init(&sm.ds_ready, kWG * 128);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, kWG * 128);
    mbar_init(&sm.acc_full, 1);
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
  // The setup above overlaps the prep kernel's end; its outputs (the work
  // counter, the row terms, the zeroed accumulator) are read only after it.
  wait_prior_grid();

  // Work items t = (head, key tile j) in the order of bwd_item.  The
  // producer claims them one at a time from the workspace counter and hands
  // each to the MMA thread and the compute warps through a two-slot ring in
  // shared memory (a claimed index >= total ends the CTA).  Every role walks
  // the same item sequence, so the barrier phases carry over from one item
  // to the next: gstep counts the query-tile steps of all items so far, kvc
  // the K/V loads, m the items.
  const int total = p.BH * p.n_kv;
  const int npad = p.n_kv * kTile;
  struct ItemInfo {
    int bh, j, i0, n_iter;
  };
  auto item_info = [&](int t) -> ItemInfo {
    ItemInfo w;
    bwd_item(t, p.BH, p.n_kv, &w.bh, &w.j);
    w.i0 = p.causal ? w.j : 0;
    w.n_iter = p.n_kv - w.i0;
    if (kSparse) {
      w.n_iter = 0;
      if (bound_ok(w.j < p.n_kv, p.status, abortf, kChkMask))
        for (int i = w.i0; i < p.n_kv; ++i) w.n_iter += p.block_mask[(size_t)i * p.n_kv + w.j] != 0;
    }
    return w;
  };
  // Checked build: the item's head and key tile exist and it has at most
  // n_kv steps starting at a query tile that exists.
  auto item_ok = [&](const ItemInfo& w) -> bool {
    return bound_ok(w.bh >= 0 && w.bh < p.BH && w.j >= 0 && w.j < p.n_kv && w.i0 >= 0 &&
                        w.n_iter >= 0 && w.n_iter <= p.n_kv - w.i0,
                    p.status, abortf, kChkItem);
  };
  // The next query tile at or after c that key tile j visits (callers ask
  // only for tiles that exist; the scan stops at the last tile anyway).
  auto next_i = [&](int c, int j) -> int {
    if (kSparse)
      while (c < p.n_kv && p.block_mask[(size_t)c * p.n_kv + j] == 0) ++c;
    return c;
  };
  // Consumers: the index of the m-th item (waits for the producer's handoff).
  auto take_item = [&](int m, bool* ok) -> int {
    const int slot = m & 1;
    *ok = mbar_wait(&sm.item_full[slot], (m >> 1) & 1, p.status, abortf, kSiteItemFull);
    return *ok ? *reinterpret_cast<volatile int*>(&sm.item_idx[slot]) : total;
  };

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<Cfg::kRegsCtl>();
    if (lane_id() == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      int gstep = 0, kvc = 0;
      bool ok = true;
      for (int m = 0; ok; ++m) {
        const int slot = m & 1;
        if (m >= 2 &&
            !mbar_wait(&sm.item_empty[slot], ((m - 2) >> 1) & 1, p.status, abortf, kSiteItemEmpty)) {
          ok = false;
          break;
        }
        const int t = atomicAdd(p.sched, 1);
        *reinterpret_cast<volatile int*>(&sm.item_idx[slot]) = t;
        mbar_arrive(&sm.item_full[slot]);
        if (t >= total) break;
        const ItemInfo w = item_info(t);
        if (!item_ok(w)) {
          ok = false;
          break;
        }
        int cur = w.i0;
        for (int it = 0; it < w.n_iter; ++it) {
          const int s = gstep % NS, use = gstep / NS;
          if (use > 0 && !mbar_wait(&sm.q_empty[s], (use - 1) & 1, p.status, abortf, kSiteQEmpty)) {
            ok = false;
            break;
          }
          const int i = next_i(cur, w.j);
          cur = i + 1;
          if (!bound_ok(i < p.n_kv, p.status, abortf, kChkQTile)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.q_full[s], 2 * Cfg::kTileBytes + 2 * kTile * 4);
          for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(sm.q[s] + h * 16384, &tq, &sm.q_full[s], h * 64, i * kTile, w.bh);
            tma_load_3d(sm.dO[s] + h * 16384, &tdo, &sm.q_full[s], h * 64, i * kTile, w.bh);
          }
          bulk_load(sm.lse2[s], p.lse2 + (size_t)w.bh * npad + i * kTile, kTile * 4, &sm.q_full[s]);
          bulk_load(sm.delta[s], p.delta + (size_t)w.bh * npad + i * kTile, kTile * 4, &sm.q_full[s]);
          ++gstep;
          if (it == 0) {
            // K_j, V_j replace the previous item's once its last product
            // has read them (kv_empty).
            if (kvc > 0 &&
                !mbar_wait(&sm.kv_empty, (kvc - 1) & 1, p.status, abortf, kSiteKvEmpty)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.kv_full, 2 * Cfg::kTileBytes);
            for (int h = 0; h < D / 64; ++h) {
              tma_load_3d(sm.k + h * 16384, &tk, &sm.kv_full, h * 64, w.j * kTile, w.bh);
              tma_load_3d(sm.v + h * 16384, &tv, &sm.kv_full, h * 64, w.j * kTile, w.bh);
            }
            ++kvc;
          }
        }
      }
      if (!ok) {
        // Aborting: wait (bounded) for the copies in flight before the CTA
        // releases its shared memory.
        if (kvc > 0) drain_wait(&sm.kv_full, (kvc - 1) & 1);
        for (int c = gstep - 1; c >= 0 && c >= gstep - NS; --c)
          drain_wait(&sm.q_full[c % NS], (c / NS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_dec<Cfg::kRegsCtl>();
    if (lane_id() == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false, false);   // S^T, dP^T
      const uint32_t id_acc = idesc_bf16(128, D, false, true);    // dV, dK
      const uint32_t id_dq = idesc_bf16(128, D, true, true);      // dQ
      const uint32_t kb = smem_u32(sm.k), vb = smem_u32(sm.v), dsb = smem_u32(sm.ds);
      int gstep = 0, kvc = 0;
      bool ok = true;
      for (int m = 0; ok; ++m) {
        const int t = take_item(m, &ok);
        if (!ok) break;
        mbar_arrive(&sm.item_empty[m & 1]);
        if (t >= total) break;
        const ItemInfo w = item_info(t);
        if (!item_ok(w)) {
          ok = false;
          break;
        }
        if (w.n_iter > 0) {
          ok = mbar_wait(&sm.kv_full, kvc & 1, p.status, abortf, kSiteKvFull);
          if (!ok) break;
        }
        if constexpr (Cfg::kDbl) {
          // S^T of global step gs into region gs & 1.
          auto issue_st = [&](int gs) -> bool {
            const int s2 = gs % NS;
            if (!mbar_wait(&sm.q_full[s2], (gs / NS) & 1, p.status, abortf, kSiteQFull))
              return false;
            tc_fence_after();
            const uint32_t qb2 = smem_u32(sm.q[s2]);
            const uint32_t col = (gs & 1) ? Cfg::kColS2 : Cfg::kColS;
            const uint64_t kd = desc_here(kmajor_desc(kb, 0)), qd = desc_here(kmajor_desc(qb2, 0));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + col, desc_plus(kd, kmajor_off(kk)), desc_plus(qd, kmajor_off(kk)), id_s,
                     kk > 0);
            tc_commit(&sm.s_full[gs & 1]);
            return true;
          };
          if (w.n_iter > 0 && !(ok = issue_st(gstep))) break;
          for (int it = 0; it < w.n_iter; ++it, ++gstep) {
            const int s = gstep % NS;
            const uint32_t par = gstep & 1;
            const uint32_t cs = par ? Cfg::kColS2 : Cfg::kColS;
            const uint32_t qb = smem_u32(sm.q[s]), dob = smem_u32(sm.dO[s]);
            // dP^T into the columns the previous step's dQ occupied
            if (gstep > 0) {
              ok = mbar_wait(&sm.dq_empty, (gstep - 1) & 1, p.status, abortf, kSiteDqEmpty);
              if (!ok) break;
              tc_fence_after();
            }
            {
              const uint64_t vd = desc_here(kmajor_desc(vb, 0)), dd = desc_here(kmajor_desc(dob, 0));
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + Cfg::kColDP, desc_plus(vd, kmajor_off(kk)),
                       desc_plus(dd, kmajor_off(kk)), id_s, kk > 0);
            }
            tc_commit(&sm.dp_full);
            // The next step's S^T into the other region (its previous step's
            // dV and dK, issued earlier, have read it).  It must not reach
            // the compute warps before all of them have arrived on p_ready
            // for this step: a warp that ran ahead would finish this dS
            // phase and the next P phase and arrive again, completing this
            // step's phase before a slower warpgroup's P^T is in tensor
            // memory.  From an item's second step on, this dP^T already
            // waited for every warp's dQ drain, which follows its P phase;
            // at the first step nothing orders them, so the S^T waits for
            // p_ready there.
            if (it > 0 && it + 1 < w.n_iter && !(ok = issue_st(gstep + 1))) break;
            ok = mbar_wait(&sm.p_ready, par, p.status, abortf, kSitePReady);
            if (!ok) break;
            if (it == 0 && it + 1 < w.n_iter && !(ok = issue_st(gstep + 1))) break;
            tc_fence_after();
            {
              const uint64_t dd = desc_here(mnmajor_desc(dob, 0));
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + Cfg::kColDV, tmem + cs + (kk * 16 / kQ) * kQ + (kk * 16 % kQ) / 2,
                       desc_plus(dd, mnmajor_off(kk)), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
            }
            ok = mbar_wait(&sm.ds_ready, par, p.status, abortf, kSiteDsReady);
            if (!ok) break;
            tc_fence_after();
            {
              const uint64_t qd = desc_here(mnmajor_desc(qb, 0));
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + Cfg::kColDK,
                       tmem + cs + kQ / 2 + (kk * 16 / kQ) * kQ + (kk * 16 % kQ) / 2,
                       desc_plus(qd, mnmajor_off(kk)), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&sm.q_empty[s]);
            {
              const uint64_t sd = desc_here(mnmajor_desc(dsb, 0)), kd = desc_here(mnmajor_desc(kb, 0));
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ss(tmem + Cfg::kColDP, desc_plus(sd, mnmajor_off(kk)),
                       desc_plus(kd, mnmajor_off(kk)), id_dq, kk > 0);
            }
            tc_commit(&sm.dq_full);
          }
        } else
        for (int it = 0; it < w.n_iter; ++it, ++gstep) {
          const int s = gstep % NS;
          const uint32_t par = gstep & 1;
          const uint32_t qb = smem_u32(sm.q[s]), dob = smem_u32(sm.dO[s]);
          ok = mbar_wait(&sm.q_full[s], (gstep / NS) & 1, p.status, abortf, kSiteQFull);
          if (!ok) break;
          tc_fence_after();
          // S^T = K_j Q_i^T
          {
            const uint64_t kd = desc_here(kmajor_desc(kb, 0)), qd = desc_here(kmajor_desc(qb, 0));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + Cfg::kColS, desc_plus(kd, kmajor_off(kk)), desc_plus(qd, kmajor_off(kk)),
                     id_s, kk > 0);
          }
          tc_commit(&sm.s_full[0]);
          // dP^T = V_j dO_i^T, into the columns the previous step's dQ occupied
          if (gstep > 0) {
            ok = mbar_wait(&sm.dq_empty, (gstep - 1) & 1, p.status, abortf, kSiteDqEmpty);
            if (!ok) break;
            tc_fence_after();
          }
          {
            const uint64_t vd = desc_here(kmajor_desc(vb, 0)), dd = desc_here(kmajor_desc(dob, 0));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + Cfg::kColDP, desc_plus(vd, kmajor_off(kk)),
                     desc_plus(dd, kmajor_off(kk)), id_s, kk > 0);
          }
          tc_commit(&sm.dp_full);
          // dV += P^T dO_i.  Warpgroup g's P^T sits in TMEM columns
          // [kQ g, kQ g + kQ/2) as bf16 pairs.
          ok = mbar_wait(&sm.p_ready, par, p.status, abortf, kSitePReady);
          if (!ok) break;
          tc_fence_after();
          {
            const uint64_t dd = desc_here(mnmajor_desc(dob, 0));
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + Cfg::kColDV,
                     tmem + Cfg::kColS + (kk * 16 / kQ) * kQ + (kk * 16 % kQ) / 2,
                     desc_plus(dd, mnmajor_off(kk)), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
          }
          // dQ_i = dS K_j ; dK += dS^T Q_i.  dQ goes first: the compute
          // warps then read it out and start its reductions while the tensor
          // core runs dK and the next S^T.
          ok = mbar_wait(&sm.ds_ready, par, p.status, abortf, kSiteDsReady);
          if (!ok) break;
          tc_fence_after();
          {
            const uint64_t sd = desc_here(mnmajor_desc(dsb, 0)), kd = desc_here(mnmajor_desc(kb, 0));
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tmem + Cfg::kColDP, desc_plus(sd, mnmajor_off(kk)),
                     desc_plus(kd, mnmajor_off(kk)), id_dq, kk > 0);
          }
          tc_commit(&sm.dq_full);
          {
            const uint64_t qd = desc_here(mnmajor_desc(qb, 0));
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + Cfg::kColDK,
                     tmem + Cfg::kColS + kQ / 2 + (kk * 16 / kQ) * kQ + (kk * 16 % kQ) / 2,
                     desc_plus(qd, mnmajor_off(kk)), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&sm.q_empty[s]);
        }
        if (!ok) break;
        if (w.n_iter > 0) {
          tc_commit(&sm.kv_empty);  // the item's last product has read K_j, V_j
          ++kvc;
        }
        tc_commit(&sm.acc_full);    // dK_j, dV_j complete
      }
      tc_commit(&sm.drain);
      drain_wait(&sm.drain, 0);
    }
    __syncwarp();
  } else if (warp >= kWG * 4 + 2) {
    // Idle: its registers go to the compute warpgroups.
    setmaxnreg_dec<Cfg::kRegsCtl>();
  } else if (warp < kWG * 4) {
    // ------------------------------------------------------------ compute
    setmaxnreg_inc<Cfg::kRegsCompute>();
    // Warpgroup g handles query columns [kQ g, kQ g + kQ) of the tile;
    // thread r of every warpgroup owns key row r (TMEM lane r).
    const int g = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = tmem + lane_base + Cfg::kColS + g * kQ;
    const uint32_t colDP = tmem + lane_base + Cfg::kColDP + g * kQ;
    const uint32_t colDQ = tmem + lane_base + Cfg::kColDP + g * (D / kWG);
    const uint32_t colS2 = tmem + lane_base + Cfg::kColS2 + g * kQ;
    const float c2 = p.scale_log2;
    // dQ_i leaves the SM as float4 reductions into the accumulator, 64 KB
    // per step at d = 128.  Issued all at once they queue on the SM's
    // outbound write path and hold the compute warps back from the next
    // step's P phase, while the path idles during the rest of the step.  So
    // kNow of a thread's kGroups float4 groups go out as soon as dQ_i is read;
    // the rest wait in registers and go out after the next step's P phase
    // (kAfterP of them) and after its dS phase (the others) -- the next
    // item's first step for an item's last row -- or at the end.  Measured (main kernel, TFLOP/s): d = 128, N = 8K 1115
    // with all at once, 1272 spread 4/2/2; d = 64 827 -> 887 spread 2/0/2.
    constexpr int kGroups = D / kWG / 4;
    constexpr int kNow = Cfg::kDbl ? 2 : 4;
    constexpr int kAfterP = Cfg::kDbl ? 0 : 2;
    constexpr int kHeld = kGroups - kNow;
    uint32_t held[4 * kHeld];
    float* held_base = nullptr;  // accumulator address of group kNow of the held row, or null
    auto red4 = [&](float* base, int e, const uint32_t* v) {
      atomicAdd(reinterpret_cast<float4*>(base + (size_t)e * kTile * 4),
                make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                            __uint_as_float(v[3])));
    };
    // Row r's dQ values a[] for accumulator address `base` (group 0).
    auto reduce_dq = [&](float* base, const uint32_t* a) {
#pragma unroll
      for (int e = 0; e < kNow; ++e) red4(base, e, a + 4 * e);
#pragma unroll
      for (int e = 0; e < 4 * kHeld; ++e) held[e] = a[4 * kNow + e];
      held_base = base + (size_t)kNow * kTile * 4;
    };
    // Issue held groups [e0, e1) (compile-time bounds at every call site);
    // e1 == kHeld ends the held row.
    auto flush_held = [&](int e0, int e1) {
      if (held_base != nullptr) {
#pragma unroll
        for (int e = 0; e < kHeld; ++e)
          if (e >= e0 && e < e1) red4(held_base, e, held + 4 * e);
        if (e1 == kHeld) held_base = nullptr;
      }
    };
    // Read dQ of global step gs (query tile qi) out of tensor memory and add
    // it to the accumulator (BwdCfg::kDbl: done one step late, after the
    // next step's P phase).
    auto drain_dq = [&](int gs, int bh, int qi) -> bool {
      bool okd = mbar_wait(&sm.dq_full, gs & 1, p.status, abortf, kSiteDqFull);
      okd = __all_sync(0xffffffffu, okd);
      if (!okd) return false;
      tc_fence_after();
      uint32_t a[16];
      tmem_ld16(colDQ, a);
      tmem_wait_ld16(a);
      tc_fence_before();
      mbar_arrive(&sm.dq_empty);
      reduce_dq(p.dq_acc + dqacc_index<D>(bh, p.n_kv, qi * kTile + r, g * (D / kWG) / 4), a);
      return true;
    };
    const float neutral = c2 < 0.f ? __int_as_float(0x7f800000) : __int_as_float(0xff800000);
    int gstep = 0;
    bool ok = true;
    for (int m = 0;; ++m) {
      const int t = take_item(m, &ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(&sm.item_empty[m & 1]);
      if (t >= total) {
        flush_held(0, kHeld);  // the last item's held groups
        break;
      }
      const ItemInfo w = item_info(t);
      if (!warp_bound_ok(item_ok(w), p.status, abortf, kChkItem)) {
        ok = false;
        break;
      }
      const int j = w.j, bh = w.bh;
      const int kv_row = j * kTile + r;
      int cur = w.i0;
      int i_prev = 0;
      for (int it = 0; it < w.n_iter; ++it, ++gstep) {
        const int s = gstep % NS;
        const uint32_t par = gstep & 1;
        const int i = next_i(cur, j);
        cur = i + 1;
        // The query tile, hence the dQ accumulator rows it adds to.
        if (!warp_bound_ok(i < p.n_kv && i * kTile + r < npad, p.status, abortf, kChkDqRow)) {
          ok = false;
          break;
        }
        const uint32_t cS = (Cfg::kDbl && par) ? colS2 : colS;
        ok = mbar_wait(&sm.q_full[s], (gstep / NS) & 1, p.status, abortf, kSiteQFull);
        if (ok)
          ok = mbar_wait(&sm.s_full[Cfg::kDbl ? par : 0], Cfg::kDbl ? (gstep >> 1) & 1 : par,
                         p.status, abortf, kSiteSFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kQ];
        {
          uint32_t (&h)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          static_assert(kQ == 32, "the compute code is written for 32 query columns per warpgroup");
          tmem_ld32(cS, h);
          tmem_wait_ld(h);
        }
        if (p.causal && i == j) {
  #pragma unroll
          for (int e = 0; e < kQ; ++e)
            if (r > g * kQ + e) sr[e] = __float_as_uint(neutral);
        }
        const uint64_t* lse2x2 = reinterpret_cast<const uint64_t*>(sm.lse2[s] + g * kQ);
        const uint64_t c2x2 = f2_pack(c2, c2);
        uint32_t pk[kQ / 2];
  #pragma unroll
        for (int e = 0; e < kQ; e += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2x2,
                           lse2x2[e / 2]),
                    x0, x1);
          pk[e / 2] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
        }
        tmem_st16(cS, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_ready);
        flush_held(0, kAfterP);
        if constexpr (Cfg::kDbl) {
          if (it > 0 && !(ok = drain_dq(gstep - 1, bh, i_prev))) break;
          i_prev = i;
        }

        ok = mbar_wait(&sm.dp_full, par, p.status, abortf, kSiteDpFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t dp[kQ];
        {
          uint32_t (&h)[32] = *reinterpret_cast<uint32_t(*)[32]>(&dp[0]);
          tmem_ld32(colDP, h);
          tmem_wait_ld(h);
        }
        const uint64_t* dlx2 = reinterpret_cast<const uint64_t*>(sm.delta[s] + g * kQ);
        // dS^T row r, query columns [kQ g, kQ g + kQ): in the 128B-swizzled
        // [key][query] tile, column block (kQ g) / 64, 16-byte chunks from
        // ((kQ g) % 64) / 8.
        uint8_t* ds_row = sm.ds + (g * kQ / 64) * 16384 + r * 128;
        const int ch0 = (g * kQ % 64) / 8;
        uint32_t dsw[kQ / 2];
  #pragma unroll
        for (int ch = 0; ch < kQ / 8; ++ch) {
  #pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = ch * 8 + 2 * e;
            const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[col / 2]));
            const uint64_t dpd = f2_add(f2_pack(__uint_as_float(dp[col]), __uint_as_float(dp[col + 1])),
                                        dlx2[col / 2]);
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(pf.x, pf.y), dpd), d0, d1);
            dsw[ch * 4 + e] = pack_bf16x2(d0, d1);
          }
          *reinterpret_cast<uint4*>(ds_row + (((ch0 + ch) ^ (r & 7)) << 4)) =
              make_uint4(dsw[ch * 4], dsw[ch * 4 + 1], dsw[ch * 4 + 2], dsw[ch * 4 + 3]);
        }
        tmem_st16(cS + kQ / 2, dsw);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_ready);
        flush_held(kAfterP, kHeld);
        if constexpr (Cfg::kDbl) continue;

        ok = mbar_wait(&sm.dq_full, par, p.status, abortf, kSiteDqFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        static_assert(Cfg::kDbl || D / kWG == 32, "the single-region path is written for d = 128");
        uint32_t a[32];
        tmem_ld32(colDQ, a);
        tmem_wait_ld(a);
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        reduce_dq(p.dq_acc + dqacc_index<D>(bh, p.n_kv, i * kTile + r, g * (D / kWG) / 4), a);
      }
      if (!ok) break;
      if constexpr (Cfg::kDbl) {
        if (w.n_iter > 0 && !(ok = drain_dq(gstep - 1, bh, i_prev))) break;
      }
      // The held groups of the item's last dQ row go out during the next
      // item's first step, after its P and dS phases (as within an item), or
      // at the end: at an item boundary the SM's write path is busy with the
      // last row's other reductions and the dK, dV stores below (measured:
      // +2.6% on the main kernel at N = 1K, +2.5% for B16 H12 N1K d64).
      // Epilogue: the first half of the warpgroups stores dV, the second half
      // scale * dK, each a D / (kWG / 2)-column slice.  The next item's first
      // dV and dK products overwrite these columns only after this warp's
      // P-ready and dS-ready arrivals for that item, which come after the
      // loads below.
      ok = mbar_wait(&sm.acc_full, m & 1, p.status, abortf, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) ok = warp_bound_ok(kv_row < npad, p.status, abortf, kChkKvRow);
      if (!ok) break;
      tc_fence_after();
      constexpr int kCols = D / (kWG / 2);
      const bool is_dv = g < kWG / 2;
      const int c0 = (g % (kWG / 2)) * kCols;
      const uint32_t col = tmem + lane_base + (is_dv ? Cfg::kColDV : Cfg::kColDK) + c0;
      const float mul = is_dv ? 1.f : p.scale;
      void* out = is_dv ? p.dv : p.dk;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out) + ((size_t)bh * p.N + kv_row) * D + c0;
      // Rows are 32-byte multiples, so 32-byte stores (half as many store
      // instructions queued behind the dQ reductions: measured +4% on the
      // N = 1K pass) need only a 32-byte aligned tensor.
      const bool wide = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(col + c * 32, a);
        tmem_wait_ld(a);
        if (kv_row < p.N) {
          uint4 v[4];
          uint32_t* wv = reinterpret_cast<uint32_t*>(v);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = w.n_iter == 0 ? 0u
                                  : pack_bf16x2(__uint_as_float(a[2 * e]) * mul,
                                                __uint_as_float(a[2 * e + 1]) * mul);
          if (wide) {
            st_global_v8(dst + c * 32, wv);
            st_global_v8(dst + c * 32 + 16, wv + 8);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = v[e];
          }
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int D>
int launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tdo, BwdParams p, cudaStream_t stream, int mask) {
  // As in the forward pass, a zero scale runs its exponents with the smallest
  // normal positive scale (they round to exactly the same values); dQ and dK
  // are still multiplied by the exact scale.
  if (p.scale_log2 == 0.f) p.scale_log2 = 1.17549435e-38f;
  const long long npad = (long long)p.n_kv * kTile;
  // Each kernel is launched with programmatic stream serialization: its
  // launch (and the main kernel's setup) overlaps the end of the kernel
  // before it on the stream, and it waits for that kernel's completion
  // (wait_prior_grid) before it touches memory that kernel writes.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  auto config = [&](unsigned grid, unsigned block, size_t smem) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(grid, 1, 1);
    c.blockDim = dim3(block, 1, 1);
    c.dynamicSmemBytes = smem;
    c.stream = stream;
    c.attrs = pdl;
    c.numAttrs = 1;
    return c;
  };
  // 1. prep: one warp per (32 / (D/8)) rows.
  if (mask & 1) {
    const long long rows = (long long)p.BH * npad;
    const long long warps = (rows + (32 / (D / 8)) - 1) / (32 / (D / 8));
    const long long blocks = (warps * 32 + 255) / 256;
    const cudaLaunchConfig_t c = config((unsigned)blocks, 256, 0);
    if (cudaLaunchKernelEx(&c, fa_bwd_prep_kernel<D>, p) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
  }
  // 2. main
  if (mask & 2) {
    const size_t smem = sizeof(BwdSmem<D>);
    auto kern = p.block_mask ? fa_bwd_main_kernel<D, true> : fa_bwd_main_kernel<D, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    {
      // The compute warpgroups' setmaxnreg.inc waits for the registers the
      // fifth warpgroup releases, which suffice only at the launch register
      // count the split assumes: refuse to launch otherwise.
      cudaFuncAttributes attr;
      if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess ||
          attr.numRegs < BwdCfg<D>::kRegsLaunch)
        return FA_ERR_LAUNCH;
    }
    // One persistent CTA per SM; each claims the next item of the list
    // from the workspace counter when it is ready for one (greedy list
    // scheduling, which under a causal or block mask is the LPT rule).
    const long long items = (long long)p.BH * p.n_kv;
    const unsigned grid = (unsigned)(p.sm_count < 1 || items <= p.sm_count ? items : p.sm_count);
    const cudaLaunchConfig_t c = config(grid, BwdCfg<D>::kThreads, smem);
    if (cudaLaunchKernelEx(&c, kern, tq, tk, tv, tdo, p) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
  }
  // 3. convert
  if (mask & 4) {
    const long long blocks = (long long)p.BH * p.n_kv * (D / 64);
    const cudaLaunchConfig_t c = config((unsigned)blocks, kConvThreads, 0);
    if (cudaLaunchKernelEx(&c, fa_bwd_convert_kernel<D>, p) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
  }
  return FA_OK;
}

}  // namespace

int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const BwdParams& p, int d, cudaStream_t stream,
               int phase_mask) {
  if (d == 128) return launch_bwd_d<128>(tq, tk, tv, tdo, p, stream, phase_mask);
  if (d == 64) return launch_bwd_d<64>(tq, tk, tv, tdo, p, stream, phase_mask);
  return FA_ERR_UNSUPPORTED_D;
}

}  // namespace fa
