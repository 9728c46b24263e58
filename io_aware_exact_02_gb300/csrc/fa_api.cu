// fa_api.cu -- the C-ABI front end of libfa.so: argument checks, TMA tensor
// maps, the per-device status word and the exported entry points declared in
// include/fa.h.  No entry point allocates device memory; fa_bwd uses the
// caller's workspace.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

// The status word: [0] = first error code a kernel recorded, [1] = the wait
// site that raised it.  One per device, part of the module's static data.
__device__ int g_status[2];
// The forward's work counters for dynamic item claiming, one 128-byte slot
// per stream (FwdParams::sched); zero at load, and each launch leaves its
// slot at zero.
__device__ int g_fwd_sched[kFwdSchedSlots * kFwdSchedStride];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  int* status = nullptr;  // device address of g_status
  int sm_count = 0;
  int pair_max = 0;       // forward CTA pairs resident at once (0: not yet known)
  int* fwd_sched = nullptr;                  // device address of g_fwd_sched
  unsigned long long sched_stream[kFwdSchedSlots];  // the stream each slot serves (its id)
  int sched_used = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device setup: architecture check and the status word's address.
int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    s.supported = (major == 10 && minor == 3);
    if (s.supported &&
        (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
         s.sm_count < 1)) {
      cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    if (s.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_DEVICE;
      }
      s.status = static_cast<int*>(addr);
      if (cudaGetSymbolAddress(&addr, g_fwd_sched) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_DEVICE;
      }
      s.fwd_sched = static_cast<int*>(addr);
    }
    s.checked = true;
  }
  if (!s.supported) return FA_ERR_DEVICE;
  *out = &s;
  return FA_OK;
}

// The forward's grid and work counter.  Items of equal cost (no mask) or
// no more items than SMs: the static grid of fwd_grid.  Uneven items (a
// causal or block mask) on more items than SMs: one persistent CTA per SM
// claiming items from the stream's counter slot (bf16 kernels; the FP8
// kernel gives every item its own CTA).  Launches on one stream run in
// order, so one slot per stream is never used by two launches at once; a
// launch leaves its slot at zero.  When every slot is taken (more than
// kFwdSchedSlots streams have run masked forward passes on the device)
// the call falls back to one CTA per item.
void set_fwd_grid(FwdParams* p, DeviceState* ds, long long items, bool uneven, bool claim,
                  cudaStream_t stream) {
  p->sched = nullptr;
  p->grid = fwd_grid(1, (int)items, uneven ? 1 : 0, ds->sm_count);
  if (!uneven || !claim || items <= ds->sm_count) return;
  // Streams are told apart by their handle, except the per-thread default
  // stream, whose one handle value names a different stream in every host
  // thread: it gets a key of the calling thread's own.  (No CUDA call here,
  // so the lookup is safe while the stream is being captured into a graph.)
  static std::atomic<unsigned long long> next_thread_key{1};
  thread_local const unsigned long long thread_key = next_thread_key++;
  const unsigned long long key =
      stream == cudaStreamPerThread ? (thread_key | (1ull << 63))
                                    : (unsigned long long)reinterpret_cast<uintptr_t>(stream);
  std::lock_guard<std::mutex> lk(g_mu);
  int slot = -1;
  for (int i = 0; i < ds->sched_used; ++i)
    if (ds->sched_stream[i] == key) slot = i;
  if (slot < 0 && ds->sched_used < kFwdSchedSlots) {
    slot = ds->sched_used++;
    ds->sched_stream[slot] = key;
  }
  if (slot < 0) return;
  p->sched = ds->fwd_sched + slot * kFwdSchedStride;
  p->grid = ds->sm_count;
}

int get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr) {
      cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of the shape arguments.
int check_shape(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_ARG;
  if (!std::isfinite(scale)) return FA_ERR_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  // Element counts of a [B][H][Npad][d] array must fit in int64 and the
  // tensor map's 32-bit coordinates must reach every row.
  const long long bh = (long long)B * H;
  if (bh > (1LL << 30)) return FA_ERR_ARG;
  const long long npad = (long long)ceil_div(N, kTile) * kTile;
  if ((double)bh * (double)npad * (double)d > 9.0e18) return FA_ERR_ARG;
  if ((unsigned long long)bh * (unsigned long long)ceil_div(N, kPairRows) > 0x7fffffffULL)
    return FA_ERR_ARG;
  return FA_OK;
}

// Shape checks and derived sizes of the general forward pass.
struct GqaShape {
  int BH, rows, n_kv, n_pairs, splits, tiles_per_split;
  FwdWorkspace ws;
};

int gqa_shape(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int num_splits, float scale,
              GqaShape* g) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || num_splits < 1) return FA_ERR_ARG;
  if (Hq % Hkv != 0) return FA_ERR_ARG;
  if (!std::isfinite(scale)) return FA_ERR_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  const long long bh = (long long)B * Hkv;
  const long long rows = (long long)(Hq / Hkv) * Nq;
  if (bh > (1LL << 30) || rows > (1LL << 30)) return FA_ERR_ARG;
  const int n_kv = ceil_div(Nkv, kTile);
  const int tps = ceil_div(n_kv, num_splits < n_kv ? num_splits : n_kv);
  const int splits = ceil_div(n_kv, tps);
  const long long n_pairs = (rows + kPairRows - 1) / kPairRows;
  if (bh * n_pairs * splits > 0x7fffffffLL) return FA_ERR_ARG;
  if ((double)splits * (double)bh * (double)rows * (double)d * 4.0 > 9.0e18) return FA_ERR_ARG;
  g->BH = (int)bh;
  g->rows = (int)rows;
  g->n_kv = n_kv;
  g->n_pairs = (int)n_pairs;
  g->splits = splits;
  g->tiles_per_split = tps;
  g->ws = fwd_workspace_layout(splits, bh, (long long)rows, d);
  return FA_OK;
}

}  // namespace

int make_tmap_bhnd(const void* base, int BH, int N, int d, CUtensorMap* out) {
  return make_tmap_bhnd_rows(base, BH, N, d, kTile, out);
}

int make_tmap_bhnd_rows(const void* base, int BH, int N, int d, int box_rows, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = get_encode(&enc);
  if (rc != FA_OK) return rc;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ARG;
}

// The self test's kernel: one thread waits on a barrier nothing arrives on
// until the limit passes, then records the timeout like any kernel wait.
__global__ void fa_selftest_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  abort_flag = 0;
  const uint32_t a = smem_u32(&bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      report_timeout(status, &abort_flag, FA_SITE_SELFTEST);
      return;
    }
  }
}

// The bounds-check self test: one thread checks an index one past its range
// (n = 1, index 1) through the kernels' check; it touches no memory but the
// status word, which the check writes only in the checked build.
__global__ void fa_selftest_bounds_kernel(int* status, int n) {
  int abort_flag = 0;
  const int index = n;
  if (!bound_ok(index < n, status, &abort_flag, FA_SITE_SELFTEST_BOUNDS)) return;
}

int make_tmap_u8(const void* base, int BH, int rows, int inner, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = get_encode(&enc);
  if (rc != FA_OK) return rc;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)rows * inner};
  cuuint32_t box[3] = {128, kTile, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_ARG;
}

namespace {

// Shape checks of the FP8 forward pass: the square shape with d = 128.
int fp8_shape(int B, int H, int N, int d, float scale) {
  int rc = check_shape(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED_D;
  if ((long long)B * H * ceil_div(N, kTile) > 0x7fffffffLL) return FA_ERR_ARG;
  return FA_OK;
}

int fp8_workspace_ok(const void* workspace, size_t workspace_bytes, const Fp8Workspace& w) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  return FA_OK;
}

// The FP8 attention kernel over a quantised workspace.
int fwd_fp8_quantized_impl(void* o, float* lse, int B, int H, int N, int d, int causal,
                           float scale, int hadamard, const void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!o || !lse) return FA_ERR_ARG;
  if ((causal != 0 && causal != 1) || (hadamard != 0 && hadamard != 1)) return FA_ERR_ARG;
  int rc = fp8_shape(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
  const int BH = B * H;
  const Fp8Workspace w = fp8_workspace_layout(BH, N, d);
  if ((rc = fp8_workspace_ok(workspace, workspace_bytes, w)) != FA_OK) return rc;
  DeviceState* ds;
  if ((rc = device_state(&ds)) != FA_OK) return rc;
  const char* ws = static_cast<const char*>(workspace);
  CUtensorMap tq, tk, tv;
  if ((rc = make_tmap_u8(ws + w.q8, BH, N, d, &tq)) != FA_OK) return rc;
  if ((rc = make_tmap_u8(ws + w.k8, BH, N, d, &tk)) != FA_OK) return rc;
  if ((rc = make_tmap_u8(ws + w.vt8, BH, d, ceil_div(N, kTile) * kTile, &tv)) != FA_OK) return rc;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.block_mask = nullptr;
  p.fp8_amax = reinterpret_cast<const float*>(ws + w.amax);
  p.fp8_hadamard = hadamard;
  p.status = ds->status;
  p.BH = BH;
  p.rows = N;
  p.Nq = N;
  p.Nkv = N;
  p.causal_off = 0;
  p.n_kv = ceil_div(N, kTile);
  p.n_pairs = ceil_div(N, kPairRows);
  p.splits = 1;
  p.tiles_per_split = p.n_kv;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  set_fwd_grid(&p, ds, (long long)BH * p.n_pairs, causal != 0, false,
               static_cast<cudaStream_t>(stream));
  return launch_fwd(tq, tk, tv, tq, p, d, static_cast<cudaStream_t>(stream));  // O stored directly
}

int fp8_quantize_impl(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                      int hadamard, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v) return FA_ERR_ARG;
  if (hadamard != 0 && hadamard != 1) return FA_ERR_ARG;
  int rc = fp8_shape(B, H, N, d, 1.0f);
  if (rc != FA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA_ERR_ALIGN;
  const int BH = B * H;
  const Fp8Workspace w = fp8_workspace_layout(BH, N, d);
  if ((rc = fp8_workspace_ok(workspace, workspace_bytes, w)) != FA_OK) return rc;
  DeviceState* ds;
  if ((rc = device_state(&ds)) != FA_OK) return rc;
  return launch_fp8_quantize(q, k, v, BH, N, hadamard, static_cast<char*>(workspace), w,
                             static_cast<cudaStream_t>(stream));
}

// The forward pass over a general shape; block_mask is null for dense attention.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nkv, int d, int causal, float scale, int num_splits,
             void* workspace, size_t workspace_bytes, const uint8_t* block_mask, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_ARG;
  GqaShape g;
  int rc = gqa_shape(B, Hq, Hkv, Nq, Nkv, d, num_splits, scale, &g);
  if (rc != FA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if (g.splits > 1 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                       workspace_bytes < g.ws.total))
    return FA_ERR_WORKSPACE;
  DeviceState* ds;
  if ((rc = device_state(&ds)) != FA_OK) return rc;
  CUtensorMap tq, tk, tv, to;
  if ((rc = make_tmap_bhnd(q, g.BH, g.rows, d, &tq)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(k, g.BH, Nkv, d, &tk)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(v, g.BH, Nkv, d, &tv)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(o, g.BH, g.rows, d, &to)) != FA_OK) return rc;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.block_mask = block_mask;
  p.fp8_amax = nullptr;
  p.fp8_hadamard = 0;
  if (g.splits > 1) {
    p.o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + g.ws.o_part);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + g.ws.lse_part);
  }
  p.status = ds->status;
  p.BH = g.BH;
  p.rows = g.rows;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.causal_off = Nkv - Nq;
  p.n_kv = g.n_kv;
  p.n_pairs = g.n_pairs;
  p.splits = g.splits;
  p.tiles_per_split = g.tiles_per_split;
  p.causal = causal;
  p.scale_log2 = scale * 1.4426950408889634f;
  // Block-sparse items differ in cost like causal ones and are claimed
  // dynamically.  Under the bottom-right causal mask, items cost the same
  // when the query rows are few (decode, N_q <= 16: every row sees about all
  // keys), and the static split serves them.
  const bool uneven = block_mask != nullptr || (causal && Nq > 16);
  set_fwd_grid(&p, ds, (long long)g.BH * g.n_pairs * g.splits, uneven, true,
               static_cast<cudaStream_t>(stream));
  // Square, d = 128, no mask: the CTA-pair kernel (tcgen05 cta_group::2),
  // whose products read half the shared memory per CTA, runs only when
  // FA_FWD_PAIR=1 is in the environment (0 or unset: the one-CTA kernel;
  // the library reads it once).  It was the faster one at N > 2K (B8 H16,
  // TFLOP/s, pair / one CTA: 4K 1666 / 1564, 8K 1753 / 1663) until the
  // one-CTA kernel's epilogue moved to its own warpgroup (then, on one box:
  // 4K 1655 / 1697, 8K 1635 / 1712, 16K 1632 / 1664).
  static const int pair_mode = [] {
    const char* e = std::getenv("FA_FWD_PAIR");
    if (e != nullptr && (e[0] == '0' || e[0] == '1') && e[1] == 0) return e[0] - '0';
    return -1;
  }();
  const bool pair_shape = d == 128 && !causal && block_mask == nullptr && g.splits == 1 &&
                          Hq == Hkv && Nq == Nkv;
  if (pair_shape && pair_mode == 1) {
    CUtensorMap tkh;
    if ((rc = make_tmap_bhnd_rows(k, g.BH, Nkv, d, 64, &tkh)) != FA_OK) return rc;
    if (p.scale_log2 == 0.f) p.scale_log2 = 1.17549435e-38f;  // as launch_fwd does
    int pairs;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (ds->pair_max == 0) ds->pair_max = fwd_pair_max_active(ds->sm_count);
      pairs = ds->pair_max;
    }
    return launch_fwd_pair(tq, tkh, tv, p, static_cast<cudaStream_t>(stream), pairs);
  }
  return launch_fwd(tq, tk, tv, to, p, d, static_cast<cudaStream_t>(stream));
}

// The backward pass; block_mask is null for dense attention.
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             int causal, float scale, void* workspace, size_t workspace_bytes, void* stream,
             int phase_mask, const uint8_t* block_mask) {
  if (phase_mask < 1 || phase_mask > 7) return FA_ERR_ARG;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_ARG;
  int rc = check_shape(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGN;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  DeviceState* ds;
  if ((rc = device_state(&ds)) != FA_OK) return rc;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = make_tmap_bhnd(q, BH, N, d, &tq)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(k, BH, N, d, &tk)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(v, BH, N, d, &tv)) != FA_OK) return rc;
  if ((rc = make_tmap_bhnd(dout, BH, N, d, &tdo)) != FA_OK) return rc;
  const BwdWorkspace ws = bwd_workspace_layout(BH, N, d);
  BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.dq_acc);
  p.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.delta);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.lse2);
  p.status = ds->status;
  p.block_mask = block_mask;
  p.BH = BH;
  p.N = N;
  p.n_kv = ceil_div(N, kTile);
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.sm_count = ds->sm_count;
  p.sched = reinterpret_cast<int*>(static_cast<char*>(workspace) + ws.sched);
  return launch_bwd(tq, tk, tv, tdo, p, d, static_cast<cudaStream_t>(stream), phase_mask);
}

}  // namespace

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 1; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_ARG: return "invalid argument (null pointer, size < 1, non-finite scale or overflow)";
    case FA_ERR_UNSUPPORTED_D: return "unsupported head dimension (d must be 64 or 128)";
    case FA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_DEVICE: return "no usable device (needs sm_103 with tcgen05)";
    case FA_ERR_LAUNCH: return "CUDA launch error";
    case FA_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    case FA_ERR_BOUNDS: return "a kernel computed an out-of-range index (bounds-checked build)";
    default: return "unknown status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, N, d, causal, scale, 1, nullptr, 0, stream);
}

size_t fa_fwd_gqa_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int num_splits) {
  GqaShape g;
  if (gqa_shape(B, Hq, Hkv, Nq, Nkv, d, num_splits, 1.0f, &g) != FA_OK) return 0;
  return g.splits > 1 ? g.ws.total : 0;
}

int fa_fwd_gqa_splits(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal, int sm_count) {
  GqaShape g;
  int rc = gqa_shape(B, Hq, Hkv, Nq, Nkv, d, 1, 1.0f, &g);
  if (rc != FA_OK) return rc;
  if (sm_count < 1 || (causal != 0 && causal != 1)) return FA_ERR_ARG;
  // The split count whose items fill whole waves of SMs best: for s splits
  // of at least two 128-key tiles, wave efficiency = items*s /
  // (ceil(items*s / sms) * sms); take the smallest s within 90% of the best
  // (more splits also cost more combine work).
  const long long items = (long long)g.BH * g.n_pairs;
  int max_splits = g.n_kv / 2 > 1 ? g.n_kv / 2 : 1;
  if (max_splits > 128) max_splits = 128;
  auto eff = [&](int sp) {
    const long long n = items * sp;
    const long long waves = (n + sm_count - 1) / sm_count;
    return (double)n / (double)(waves * sm_count);
  };
  double best = 0.0;
  for (int sp = 1; sp <= max_splits; ++sp) best = eff(sp) > best ? eff(sp) : best;
  for (int sp = 1; sp <= max_splits; ++sp)
    if (eff(sp) >= 0.9 * best) return sp;
  return 1;
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int Nq, int Nkv, int d, int causal, float scale, int num_splits,
               void* workspace, size_t workspace_bytes, void* stream) {
  return fa::fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, causal, scale, num_splits,
                      workspace, workspace_bytes, nullptr, stream);
}

int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, int causal, float scale, const void* block_mask,
                       void* stream) {
  if (!block_mask) return FA_ERR_ARG;
  return fa::fwd_impl(q, k, v, o, lse, B, H, H, N, N, d, causal, scale, 1, nullptr, 0,
                      static_cast<const uint8_t*>(block_mask), stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 1.0f) != FA_OK) return 0;
  return bwd_workspace_layout((long long)B * H, N, d).total;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
           float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_phases(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                       workspace_bytes, stream, 7);
}

int fa_bwd_phases(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t workspace_bytes, void* stream,
                  int phase_mask) {
  return fa::bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                      workspace_bytes, stream, phase_mask, nullptr);
}

int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, int causal, float scale, const void* block_mask,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!block_mask) return FA_ERR_ARG;
  return fa::bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                      workspace_bytes, stream, 7, static_cast<const uint8_t*>(block_mask));
}

size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d) {
  if (fp8_shape(B, H, N, d, 1.0f) != FA_OK) return 0;
  return fp8_workspace_layout((long long)B * H, N, d).total;
}

int fa_fp8_workspace_offsets(int B, int H, int N, int d, size_t* offsets) {
  if (!offsets) return FA_ERR_ARG;
  int rc = fp8_shape(B, H, N, d, 1.0f);
  if (rc != FA_OK) return rc;
  const Fp8Workspace w = fp8_workspace_layout((long long)B * H, N, d);
  offsets[0] = w.q8;
  offsets[1] = w.k8;
  offsets[2] = w.vt8;
  offsets[3] = w.amax;
  return FA_OK;
}

int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    int hadamard, void* workspace, size_t workspace_bytes, void* stream) {
  return fp8_quantize_impl(q, k, v, B, H, N, d, hadamard, workspace, workspace_bytes, stream);
}

int fa_fwd_fp8_quantized(void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                         int hadamard, const void* workspace, size_t workspace_bytes,
                         void* stream) {
  return fwd_fp8_quantized_impl(o, lse, B, H, N, d, causal, scale, hadamard, workspace,
                                workspace_bytes, stream);
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, int causal, float scale, int hadamard, void* workspace,
               size_t workspace_bytes, void* stream) {
  if (!o || !lse) return FA_ERR_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_ARG;
  int rc = fp8_shape(B, H, N, d, scale);
  if (rc != FA_OK) return rc;
  if (!aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
  rc = fp8_quantize_impl(q, k, v, B, H, N, d, hadamard, workspace, workspace_bytes, stream);
  if (rc != FA_OK) return rc;
  return fwd_fp8_quantized_impl(o, lse, B, H, N, d, causal, scale, hadamard, workspace,
                                workspace_bytes, stream);
}

int fa_device_status(void* stream, int* site) {
  if (site) *site = 0;
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  int h[2] = {0, 0};
  const int zero[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  if (site) *site = h[1];
  return h[0];
}

int fa_selftest_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return FA_ERR_ARG;
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  fa_selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      ds->status, (unsigned long long)timeout_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_checks_enabled(void) { return kChecks ? 1 : 0; }

int fa_selftest_bounds(void* stream) {
  DeviceState* ds;
  int rc = device_state(&ds);
  if (rc != FA_OK) return rc;
  fa_selftest_bounds_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(ds->status, 1);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_schedule(int B, int H, int N, int causal, int num_ctas, int* item_bh, int* item_pair,
                    int* item_cost, int* item_cta, int max_items) {
  if (causal != 0 && causal != 1) return FA_ERR_ARG;
  if (num_ctas < 1) return FA_ERR_ARG;
  int rc = check_shape(B, H, N, 64, 1.0f);
  if (rc != FA_OK) return rc;
  const int BH = B * H;
  const int n_pairs = ceil_div(N, kPairRows);
  const int n_kv = ceil_div(N, kTile);
  const long long total = (long long)BH * n_pairs;
  const int ctas = fwd_grid(BH, n_pairs, causal, num_ctas);
  // Under a causal mask with more items than CTAs, persistent CTAs claim
  // the items in list order at run time: no CTA is fixed in advance.
  const bool claimed = causal && total > num_ctas;
  for (long long t = 0; t < total && t < max_items; ++t) {
    int bh, pair;
    fwd_item((int)t, BH, n_pairs, &bh, &pair);
    if (item_bh) item_bh[t] = bh;
    if (item_pair) item_pair[t] = pair;
    if (item_cost)
      item_cost[t] = fwd_kv_tiles(2 * pair, n_kv, causal) + fwd_kv_tiles(2 * pair + 1, n_kv, causal);
    if (item_cta) item_cta[t] = claimed ? -1 : snake_cta((int)t, ctas);
  }
  return (int)total;
}

int fa_snake_assign(int n, int workers, int* worker_of_item) {
  if (n < 0 || workers < 1 || (n > 0 && !worker_of_item)) return FA_ERR_ARG;
  for (int i = 0; i < n; ++i) worker_of_item[i] = snake_cta(i, workers);
  return FA_OK;
}

}  // extern "C"
