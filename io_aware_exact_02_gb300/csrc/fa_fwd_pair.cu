// fa_fwd_pair.cu -- forward pass of exact attention on CTA pairs (sm_103a
// tcgen05 cta_group::2), d = 128, square shapes without a mask.
//
// The pages' answer to Blackwell's shared-memory bound is to let two CTAs
// cooperate on each tensor-core product ("Reading CMU 11-868 LLM Systems:
// FlashAttention", slide pages 50-52).  In the one-CTA forward kernel every
// 128 x 128 x 128 S product reads its Q tile and its K tile from shared
// memory (128 B/clk, the whole bandwidth at the products' full rate), and
// the P V products and the TMA fills of K and V add to it, so the products
// run at about three quarters of their nominal rate.  Here a cluster of two
// CTAs (a pair) computes each product as one M = 256 instruction issued by
// the even CTA (the leader): each CTA supplies its own 128 query rows of Q
// (A operand) and half of the B operand -- 64 keys of K for S = Q K^T, 64 of
// the d columns of V for O += P V -- and receives its own 128 rows of the
// result in its tensor memory.  Per key tile a CTA then reads 96 KB of
// shared memory for its two S products (2 x (32 KB Q + 16 KB K)) and 32 KB
// for its two P V products, and takes in 32 KB of K and V halves, against
// 128 + 64 + 64 KB in the one-CTA kernel.
//
// The host runs this kernel for square shapes with d = 128 and no mask when
// FA_FWD_PAIR=1 is in the environment: the one-CTA kernel, whose epilogue
// runs in its own warpgroup, measured faster at every length.
//
// A work item is 512 query rows of one head.  CTA c of a pair holds Q tiles
// t = 0, 1: rows row0 + (2t + c) * 128, so that pair tile t (the M = 256 rows
// of one product) is the contiguous rows row0 + 256 t .. + 255.  Each CTA
// runs its own softmax warpgroups on its own rows exactly as the one-CTA
// kernel does (fa_softmax.cuh); only the leader issues MMAs.
//
// Warp roles (320 threads per CTA):
//   warps 0-3  softmax of Q tile 0 (thread r owns row r),  warps 4-7 tile 1
//   warp 8     TMA producer: the CTA's two Q tiles, then its halves of K_0,
//              V_0, K_1, V_1, ...; every load signals the LEADER's barrier
//              (cta_group::2 TMA), which counts both CTAs' bytes
//   warp 9     leader: MMA issuer; both CTAs: TMEM allocation (cta_group::2)
// Barriers: the leader's q_full, kv_full, p_full and o_empty gather both
// CTAs (TMA bytes; the peer's softmax warps arrive remotely, one arrival per
// warp); the leader's tcgen05.commit arrives on s_full, o_full, kv_empty,
// q_empty and drain in both CTAs (multicast).  Every wait is bounded and
// acquires at CTA scope, as the barriers' completions publish tensor memory
// and TMA-written shared memory, which the tcgen05 fences and the TMA
// byte counts order.
#include "fa_internal.h"
#include "fa_softmax.cuh"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kPD = 128;                  // head dimension of the pair kernel
constexpr int kQuadRows = 4 * kTile;      // query rows of one work item
constexpr int kQTileBytes = kTile * kPD * 2;   // 32 KB
constexpr int kHalfBytes = kQTileBytes / 2;    // half a K or V tile: 16 KB
constexpr int kPairStages = 10;           // K/V half-tile ring slots
constexpr int kPairThreads = 320;
constexpr uint32_t kPairTmemCols = 512;
constexpr float kLn2p = 0.69314718055994530942f;

struct alignas(1024) PairSmem {
  uint8_t q[2][kQTileBytes];
  uint8_t kv[kPairStages][kHalfBytes];
  uint64_t q_full, q_empty;
  uint64_t kv_full[kPairStages], kv_empty[kPairStages];
  uint64_t s_full[2], p_half[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

enum : int {
  kSitePQFull = 151, kSitePKvEmpty, kSitePKvFull, kSitePPFull, kSitePSFull, kSitePOFull,
  kSitePQEmpty, kSitePOEmpty, kSitePPHalf
};
enum : int { kChkPItem = 1151, kChkPRow };

// ---------------------------------------------------------------- cluster PTX

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster.  The default (CTA
// scope) semantics: what the arrival publishes is tensor memory the arriving
// warp has finished writing (tcgen05.wait::st, then
// tcgen05.fence::before_thread_sync), which the peer SM's tensor core reads
// for the leader's product.  A release at cluster scope costs a memory
// barrier per arrival instead: measured 1122 against 1497 TFLOP/s.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Wait without the abort shortcut: used while winding down after an abort.
__device__ __forceinline__ void drain_wait_c(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > 100000000ull) return;
  }
}
// 3-D TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D(tmem of both CTAs) (+)= A B over the pair: A from each CTA's shared memory
// (SS) or tensor memory (TS) at the same address, B halves from each CTA.
__device__ __forceinline__ void mma_pair_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "setp.ne.b32 P, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, P;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_pair_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "setp.ne.b32 P, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, P;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive on `bar` in both CTAs once the pair products issued so far are done.
__device__ __forceinline__ void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// K-major, 128B-swizzled tile with 64-column blocks `block` bytes apart.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk, uint32_t block) {
  return sdesc_sw128(base + (kk >> 2) * block + (kk & 3) * 32, 16, 1024);
}
// [keys][64 columns] 128B-swizzled tile as the MN-major B operand, K-step kk.
__device__ __forceinline__ uint64_t vdesc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, 16384, 1024);
}

template <bool kNeg>
__global__ void __launch_bounds__(kPairThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tkh,
                       const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  PairSmem& sm = *reinterpret_cast<PairSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abortf = &sm.abort_flag;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  constexpr int S = kPairStages;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      // the leader's own 128 threads plus one arrival per peer warp
      mbar_init(&sm.p_half[t], 128 + 4);
      mbar_init(&sm.p_full[t], 128 + 4);
      mbar_init(&sm.o_full[t], 1);
      mbar_init(&sm.o_empty[t], 128 + 4);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(&sm.tmem_base, kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // Items: (head, 512-row quad) in the work order of fwd_item, split over
  // the pairs in snake order (as the one-CTA kernel splits them over CTAs).
  const int n_quads = ceil_div(p.rows, kQuadRows);
  const int num_items = p.BH * n_quads;
  const int G = gridDim.x / 2;
  const int pair_id = blockIdx.x / 2;
  auto item_of_round = [&](int k) -> int {
    const int base = k * G;
    return (k & 1) ? base + (G - 1 - pair_id) : base + pair_id;
  };
  const int n_kv = p.n_kv;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane_id() == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tkh);
      prefetch_tmap(&tv);
      const uint32_t lead_q_full = peer_addr(&sm.q_full, 0);
      int c = 0, q_issued = 0;
      bool ok = true;
      for (int k = 0; ok && k * G < num_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= num_items) continue;
        int bh, quad;
        fwd_item(idx, p.BH, n_quads, &bh, &quad);
        if (!bound_ok(bh < p.BH && quad < n_quads, p.status, abortf, kChkPItem)) {
          ok = false;
          break;
        }
        const int row0 = quad * kQuadRows;
        if (q_issued > 0 &&
            !mbar_wait(&sm.q_empty, (q_issued - 1) & 1, p.status, abortf, kSitePQEmpty)) {
          ok = false;
          break;
        }
        if (leader) mbar_arrive_expect_tx(&sm.q_full, 4 * kQTileBytes);  // both CTAs' tiles
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < 2; ++h)
            tma_load_3d_pair(sm.q[t] + h * 16384, &tq, lead_q_full, h * 64,
                             row0 + (2 * t + (int)rank) * kTile, bh);
        ++q_issued;
        for (int j = 0; j < n_kv && ok; ++j) {
          for (int w = 0; w < 2; ++w, ++c) {  // K half, then V half
            const int slot = c % S, use = c / S;
            if (use > 0 &&
                !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, p.status, abortf, kSitePKvEmpty)) {
              ok = false;
              break;
            }
            const uint32_t lead_full = peer_addr(&sm.kv_full[slot], 0);
            if (leader) mbar_arrive_expect_tx(&sm.kv_full[slot], 2 * kHalfBytes);
            if (w == 0) {  // keys [128 j + 64 rank, + 64), all d columns
              for (int h = 0; h < 2; ++h)
                tma_load_3d_pair(sm.kv[slot] + h * 8192, &tkh, lead_full, h * 64,
                                 j * kTile + (int)rank * 64, bh);
            } else {       // all 128 keys, d columns [64 rank, + 64)
              tma_load_3d_pair(sm.kv[slot], &tv, lead_full, (int)rank * 64, j * kTile, bh);
            }
          }
        }
      }
      if (!ok && leader) {
        // Let the copies already issued land before the CTA pair exits.
        if (q_issued > 0) drain_wait_c(&sm.q_full, (q_issued - 1) & 1);
        for (int cc = c - 1; cc >= 0 && cc >= c - S; --cc)
          drain_wait_c(&sm.kv_full[cc % S], (cc / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane_id() == 0) {
      const uint32_t id_s = idesc_bf16(256, 128, false, false);   // S: M = 256, N = 128 keys
      const uint32_t id_pv = idesc_bf16(256, kPD, false, true);   // O += P V: N = d
      const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
      uint32_t p_par[2] = {0, 0};
      int cb = 0, n_done = 0, q_used = 0;
      bool ok = true;
      auto wait_full = [&](int cnt) -> bool {
        return mbar_wait(&sm.kv_full[cnt % S], (cnt / S) & 1, p.status, abortf, kSitePKvFull);
      };
      auto issue_s = [&](int t, int kslot) {
        const uint64_t qd = desc_here(kdesc(q_addr[t], 0, 16384)), kd = desc_here(kdesc(smem_u32(sm.kv[kslot]), 0, 8192));
#pragma unroll
        for (int kk = 0; kk < kPD / 16; ++kk)
          mma_pair_ss(tmem + (uint32_t)t * 128u, desc_plus(qd, (kk >> 2) * 16384 + (kk & 3) * 32),
                      desc_plus(kd, (kk >> 2) * 8192 + (kk & 3) * 32), id_s, kk > 0);
        commit_pair(&sm.s_full[t]);
      };
      // O_t += P_t V; the item's first product overwrites O_t, so it waits
      // until both CTAs' softmax t have stored the previous item's O_t.
      auto issue_pv = [&](int t, int vslot, bool accumulate) -> bool {
        if (!accumulate && n_done > 0) {
          if (!mbar_wait(&sm.o_empty[t], (n_done - 1) & 1, p.status, abortf, kSitePOEmpty))
            return false;
          tc_fence_after();
        }
        const uint64_t vd = desc_here(vdesc(smem_u32(sm.kv[vslot]), 0));
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (kk == kTile / 32) {  // the second half of P (keys 64-127)
            const bool r = mbar_wait(&sm.p_full[t], p_par[t], p.status, abortf, kSitePPFull);
            p_par[t] ^= 1;
            if (!r) return false;
            tc_fence_after();
          }
          mma_pair_ts(tmem + 256u + (uint32_t)t * kPD, tmem + (uint32_t)t * 128u + kk * 8,
                      desc_plus(vd, kk * 2048), id_pv, (accumulate || kk > 0) ? 1u : 0u);
        }
        return true;
      };
      // The first half of P_t (keys 0-63) in both CTAs; issue_pv waits for
      // the second half itself.
      auto wait_p = [&](int t) -> bool {
        return mbar_wait(&sm.p_half[t], p_par[t], p.status, abortf, kSitePPHalf);
      };
      for (int k = 0; ok && k * G < num_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= num_items) continue;
        ok = mbar_wait(&sm.q_full, q_used & 1, p.status, abortf, kSitePQFull);
        if (ok) ok = wait_full(cb);
        if (ok) {
          tc_fence_after();
          issue_s(0, cb % S);
          issue_s(1, cb % S);
          commit_pair(&sm.kv_empty[cb % S]);
          if (n_kv == 1) commit_pair(&sm.q_empty);
        }
        // Key tile j: PV_t(j-1), then S_t(j), for t = 0, 1.
        for (int j = 1; j < n_kv && ok; ++j) {
          const int kc = cb + 2 * j, vc = cb + 2 * j - 1;
          ok = wait_full(kc) && wait_full(vc);
          if (!ok) break;
          for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_p(t);
            if (!ok) break;
            tc_fence_after();
            ok = issue_pv(t, vc % S, j - 1 > 0);
            if (ok) issue_s(t, kc % S);
          }
          if (!ok) break;
          commit_pair(&sm.kv_empty[vc % S]);
          commit_pair(&sm.kv_empty[kc % S]);
          if (j == n_kv - 1) commit_pair(&sm.q_empty);  // last product reading Q
        }
        if (ok) {
          const int vc = cb + 2 * n_kv - 1;
          ok = wait_full(vc);
          for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_p(t);
            if (!ok) break;
            tc_fence_after();
            ok = issue_pv(t, vc % S, n_kv - 1 > 0);
            if (ok) commit_pair(&sm.o_full[t]);
          }
          if (ok) commit_pair(&sm.kv_empty[vc % S]);
        }
        cb += 2 * n_kv;
        ++q_used;
        ++n_done;
      }
      // Every product issued so far must finish before TMEM is released.
      commit_pair(&sm.drain);
      drain_wait_c(&sm.drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c2 = p.scale_log2;
    const float ninf = __int_as_float(0xff800000);
    const uint32_t colS = tmem + lane_base + (uint32_t)t * 128u;
    const uint32_t colO = tmem + lane_base + 256u + (uint32_t)t * kPD;
    // P ready / O read: the leader's threads arrive on their own barrier,
    // the peer's warps once each on the leader's.
    const uint32_t lead_p_half = peer_addr(&sm.p_half[t], 0);
    const uint32_t lead_p_full = peer_addr(&sm.p_full[t], 0);
    const uint32_t lead_o_empty = peer_addr(&sm.o_empty[t], 0);
    auto signal = [&](uint64_t* own, uint32_t lead) {
      if (leader) {
        mbar_arrive(own);
      } else {
        __syncwarp();
        if (lane_id() == 0) mbar_arrive_remote(lead);
      }
    };
    uint32_t s_par = 0;
    int n_done = 0;
    bool ok = true;
    for (int k = 0; ok && k * G < num_items; ++k) {
      const int idx = item_of_round(k);
      if (idx >= num_items) continue;
      int bh, quad;
      fwd_item(idx, p.BH, n_quads, &bh, &quad);
      const int R = quad * kQuadRows + (2 * t + (int)rank) * kTile + r;  // query row
      if (!warp_bound_ok(bh < p.BH && quad < n_quads, p.status, abortf, kChkPItem)) {
        ok = false;
        break;
      }
      float m_ref = ninf;
      float l = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const int tlim = p.Nkv - j * kTile;  // columns >= tlim are past the keys
        ok = mbar_wait(&sm.s_full[t], s_par, p.status, abortf, kSitePSFull);
        ok = __all_sync(0xffffffffu, ok);
        s_par ^= 1;
        if (!ok) break;
        tc_fence_after();
        softmax_tile<kPD, kNeg, false>(colS, colO, c2, tlim, j > 0, m_ref, l,
                                       [&] { signal(&sm.p_half[t], lead_p_half); });
        tc_fence_before();
        signal(&sm.p_full[t], lead_p_full);
      }
      if (ok) ok = mbar_wait(&sm.o_full[t], n_done & 1, p.status, abortf, kSitePOFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // Epilogue: O / l to bf16 and lse, rows past N not stored.
      const bool any = l > 0.f;
      const float inv_l = any ? 1.f / l : 0.f;
      const bool valid = R < p.rows;
      const size_t row_g = (size_t)bh * p.rows + R;
      if (!warp_bound_ok(!valid || row_g < (size_t)p.BH * p.rows, p.status, abortf, kChkPRow)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < kPD / 32; ++c) {
        uint32_t orow[32];
        tmem_ld32(colO + c * 32, orow);
        tmem_wait_ld(orow);
        if (!valid) continue;
        uint4 v[4];
        uint32_t* w = reinterpret_cast<uint32_t*>(v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = any ? pack_bf16x2(__uint_as_float(orow[2 * i]) * inv_l,
                                   __uint_as_float(orow[2 * i + 1]) * inv_l)
                     : 0u;
        uint4* dst =
            reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + row_g * kPD + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = v[i];
      }
      if (valid) p.lse[row_g] = any ? (m_ref + __log2f(l)) * kLn2p : ninf;
      tc_fence_before();
      signal(&sm.o_empty[t], lead_o_empty);  // O_t may now be overwritten
      ++n_done;
    }
  }

  // Neither CTA may leave (or free its tensor memory) while the pair's
  // products or the other CTA's arrivals can still reach it.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

}  // namespace

size_t fwd_pair_smem_bytes() { return sizeof(PairSmem) + 1024; }

int launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tkh, const CUtensorMap& tv,
                    const FwdParams& p, cudaStream_t stream, int max_pairs) {
  const size_t smem = fwd_pair_smem_bytes();
  auto kern = p.scale_log2 < 0.f ? fa_fwd_pair_kernel<true> : fa_fwd_pair_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return FA_ERR_LAUNCH;
  const long long items = (long long)p.BH * ceil_div(p.rows, kQuadRows);
  const long long pairs = items < max_pairs ? items : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tq, tkh, tv, p) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

// Pairs that can be resident at once (one CTA per SM, two SMs per pair).
int fwd_pair_max_active(int sm_count) {
  const size_t smem = fwd_pair_smem_bytes();
  if (cudaFuncSetAttribute(fa_fwd_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return sm_count / 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count & ~1), 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fa_fwd_pair_kernel<false>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return sm_count / 2;
  }
  return n;
}

}  // namespace fa
