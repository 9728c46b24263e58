// fa_internal.h -- declarations shared by the C-ABI front end (fa_api.cu)
// and the kernels (fa_fwd.cu, fa_bwd.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kTile = 128;        // rows of a Q tile and of a K/V tile
constexpr int kPairRows = 2 * kTile;  // query rows of one forward work item
constexpr int kHeadGroup = 8;     // heads whose work items are kept together

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Number of 128-key tiles query tile `qt` (rows 128*qt .. 128*qt+127) visits.
__host__ __device__ inline int fwd_kv_tiles(int qt, int n_kv, int causal) {
  if (!causal) return n_kv;
  const int last = qt + 1;  // keys j <= row: tiles 0 .. qt
  return last < n_kv ? last : n_kv;
}

// The forward kernel's work order.  Items are (head, pair of query tiles).
// Heads are taken in groups of kHeadGroup so that the CTAs running at the
// same time share few heads' K/V in L2; inside a group the pairs go from
// the last (most keys under a causal mask) to the first, so under a causal
// mask the longest items start first and the short ones fill the tail.
__host__ __device__ inline void fwd_item(int t, int BH, int n_pairs, int* bh, int* pair) {
  const int per_group = kHeadGroup * n_pairs;
  const int g = t / per_group;
  const int gsize = (BH - g * kHeadGroup) < kHeadGroup ? (BH - g * kHeadGroup) : kHeadGroup;
  const int idx = t - g * per_group;
  *pair = n_pairs - 1 - idx / gsize;
  *bh = g * kHeadGroup + idx % gsize;
}

// Forward parameters.  The general form has H_q query heads sharing H_kv
// K/V heads in groups of G = H_q / H_kv; the G * N_q query rows of one K/V
// head are contiguous in a [B][H_q][N_q][d] array, so the kernel treats them
// as one packed row space of `rows` rows per K/V head.  Row r is query
// position r % N_q.  The square entry point is G = 1, N_q = N_kv = N.
struct FwdParams {
  void* o;           // [BH][rows][d] bf16
  float* lse;        // [BH][rows] fp32
  float* o_part;     // splits > 1: [splits][BH][rows][d] fp32, each split's O
  float* lse_part;   // splits > 1: [splits][BH][rows] fp32, each split's lse
  const uint8_t* block_mask;  // optional [n_kv][n_kv] 0/1 over (query tile, key tile)
  const float* fp8_amax;      // FP8 forward: [3][BH] amax of the (rotated) Q, K and of V
  int fp8_hadamard;           // FP8 forward: Q and K were rotated by H_d
  int* status;       // device status word (2 ints: code, site)
  int BH;            // B * H_kv
  int rows;          // packed query rows per K/V head: G * N_q
  int Nq;            // query positions per query head
  int Nkv;           // keys per K/V head
  int causal_off;    // N_kv - N_q: query i sees keys j <= i + causal_off
  int n_kv;          // ceil(N_kv / 128)
  int n_pairs;       // ceil(rows / 256)
  int splits;        // key splits (1: O and lse written directly)
  int tiles_per_split;
  int causal;
  float scale_log2;  // scale * log2(e)
  int grid;          // CTAs launched
  // Dynamic item claiming (persistent CTAs under a causal or block mask):
  // {items claimed, CTAs finished}, zero at launch; the last CTA to finish
  // sets both back to zero.  Null: the static split of the list.
  int* sched;
};

// Slots of the forward's work counters: calls on one stream share a slot
// (they run in order), calls on different streams get different slots.
constexpr int kFwdSchedSlots = 64;
constexpr int kFwdSchedStride = 32;  // ints per slot: one 128-byte line each

// Number of 128-key tiles, counted from key 0, that the query rows
// [r0, min(r0 + 128, rows)) of a K/V head need: all of them without a mask,
// else up to the last key visible to the row with the largest position.
__host__ __device__ inline int fwd_tile_key_tiles(int r0, const FwdParams& p) {
  if (r0 >= p.rows) return 0;
  if (!p.causal) return p.n_kv;
  const int len = (r0 + kTile < p.rows ? r0 + kTile : p.rows) - r0;
  const int i0 = r0 % p.Nq;
  const int maxi = (i0 + len - 1 >= p.Nq) ? p.Nq - 1 : i0 + len - 1;
  long long lim = (long long)maxi + p.causal_off + 1;
  if (lim <= 0) return 0;
  if (lim > p.Nkv) lim = p.Nkv;
  return ceil_div((int)lim, kTile);
}

// CTA that runs work item `idx` of a longest-first list on `ctas` persistent
// CTAs: round k = idx / ctas is taken in order when k is even and in
// reverse when k is odd ("snake" order).
__host__ __device__ inline int snake_cta(int idx, int ctas) {
  const int k = idx / ctas, pos = idx % ctas;
  return (k & 1) ? ctas - 1 - pos : pos;
}

// The forward kernel's grid.  Without a mask every item costs the same and
// min(items, SMs) persistent CTAs split the list statically.  Under a causal
// mask item costs differ by up to N/128, so a static split cannot balance
// them: the CTAs take the longest-first list greedily instead (the LPT
// rule).  With a work counter (FwdParams::sched) min(items, SMs) persistent
// CTAs claim the items in list order as they become ready for one; without
// one every item gets its own CTA and the hardware hands CTAs to SMs in
// list order as SMs free up.  This function gives the grid of the latter.
__host__ __device__ inline int fwd_grid(int BH, int n_pairs, int causal, int sm_count) {
  const long long items = (long long)BH * n_pairs;
  if (causal) return (int)items;
  return (int)(items < sm_count ? items : sm_count);
}

struct BwdParams {
  const void* o;     // [BH][N][d] bf16 (forward output)
  const void* dout;  // [BH][N][d] bf16
  const float* lse;  // [BH][N] fp32
  void* dq;          // [BH][N][d] bf16
  void* dk;
  void* dv;
  float* dq_acc;     // workspace: [BH][n_kv*128][d] fp32, tile-blocked
  float* delta;      // workspace: [BH][n_kv*128] fp32 (-D_i)
  float* lse2;       // workspace: [BH][n_kv*128] fp32 (-lse_i * log2 e, -inf past N)
  int* status;
  const uint8_t* block_mask;  // optional [n_kv][n_kv] 0/1 over (query tile, key tile)
  int BH, N;
  int n_kv;
  int causal;
  float scale;
  float scale_log2;
  int* sched;    // workspace: the main kernel's work-item counter (zeroed by prep)
  int sm_count;  // persistent grid size of the main kernel
};

// Build a rank-3 tensor map over a [BH][N][d] bf16 array: dims (d, N, BH),
// box (64, 128, 1), 128-byte swizzle, zero fill outside.  Returns 0 or an
// FA_ERR_* code.
int make_tmap_bhnd(const void* base, int BH, int N, int d, CUtensorMap* out);

// The same map with a box of `box_rows` rows (the pair kernel's K halves).
int make_tmap_bhnd_rows(const void* base, int BH, int N, int d, int box_rows, CUtensorMap* out);

// The forward pass on CTA pairs (tcgen05 cta_group::2): square shapes with
// d = 128 and no mask.  tkh is K's map with a 64-row box.  At most
// `max_pairs` pairs are launched (fwd_pair_max_active: pairs that fit at once).
int launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tkh, const CUtensorMap& tv,
                    const FwdParams& p, cudaStream_t stream, int max_pairs);
int fwd_pair_max_active(int sm_count);

// `to` is a tensor map over O with the shape of tq's; only the square bf16
// kernels that stage O for TMA stores use it.
int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdParams& p, int d, cudaStream_t stream);

// Byte offsets of the general forward pass's split workspace: each split's
// fp32 O, then each split's lse, 256-byte aligned.
struct FwdWorkspace {
  size_t o_part, lse_part, total;
};
inline FwdWorkspace fwd_workspace_layout(long long splits, long long BH, long long rows, int d) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  FwdWorkspace w;
  w.o_part = 0;
  w.lse_part = up((size_t)(splits * BH * rows) * (size_t)d * sizeof(float));
  w.total = w.lse_part + up((size_t)(splits * BH * rows) * sizeof(float));
  return w;
}

// Byte offsets of the backward workspace's parts for these sizes:
// the fp32 dQ accumulator, then -D, then -lse * log2(e), then the main
// kernel's work-item counter (one int in a 256-byte slot), each 256-byte
// aligned.
struct BwdWorkspace {
  size_t dq_acc, delta, lse2, sched, total;
};
inline BwdWorkspace bwd_workspace_layout(long long BH, int N, int d) {
  const size_t rows = (size_t)BH * (size_t)ceil_div(N, kTile) * kTile;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  BwdWorkspace w;
  w.dq_acc = 0;
  w.delta = up(rows * (size_t)d * sizeof(float));
  w.lse2 = w.delta + up(rows * sizeof(float));
  w.sched = w.lse2 + up(rows * sizeof(float));
  w.total = w.sched + 256;
  return w;
}

// Byte offsets of the FP8 forward pass's workspace (d = 128): the E4M3
// codes of the (rotated) Q and K, [BH][N][d]; the codes of V transposed per
// head, [BH][d][n_kv * 128] (keys past N are code 0); then the per-head
// absolute maxima of Q, K and V, [3][BH] fp32.  Parts 256-byte aligned.
struct Fp8Workspace {
  size_t q8, k8, vt8, amax, total;
};
inline Fp8Workspace fp8_workspace_layout(long long BH, int N, int d) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t qk = (size_t)BH * (size_t)N * (size_t)d;
  const size_t vt = (size_t)BH * (size_t)d * (size_t)ceil_div(N, kTile) * kTile;
  Fp8Workspace w;
  w.q8 = 0;
  w.k8 = up(qk);
  w.vt8 = w.k8 + up(qk);
  w.amax = w.vt8 + up(vt);
  w.total = w.amax + up((size_t)3 * BH * sizeof(float));
  return w;
}

// Quantise bf16 Q, K, V ([BH][N][128]) into the FP8 workspace `ws` laid out
// by fp8_workspace_layout; with `hadamard` the rows of Q and K are first
// multiplied by the 128 x 128 Sylvester Hadamard matrix.
int launch_fp8_quantize(const void* q, const void* k, const void* v, int BH, int N, int hadamard,
                        char* ws, const Fp8Workspace& layout, cudaStream_t stream);

// A rank-3 tensor map over a [BH][rows][inner] array of bytes: box
// (128, 128, 1), 128-byte swizzle, zero fill outside.
int make_tmap_u8(const void* base, int BH, int rows, int inner, CUtensorMap* out);

// phase_mask: bit 0 prep, bit 1 main, bit 2 convert.
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const BwdParams& p, int d, cudaStream_t stream,
               int phase_mask);

}  // namespace fa
