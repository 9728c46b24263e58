// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// fa_bwd needs a workspace (an fp32 dQ accumulator and two per-row fp32
// terms) that the caller allocates.  Some callers cannot do that: code that
// runs under a memory manager owning all of the device's memory (a
// framework's caching allocator, a serving engine that reserves HBM up front)
// may not allocate outside it; latency-critical callers cannot afford
// cudaMalloc's implicit device-wide synchronisation on their hot path; and a
// plugin loaded into another program may be handed no allocator at all.
// For them this entry point takes its workspace from a fixed scratch array
// that is part of the library's static device data.
//
// The array is kNoAllocScratchBytes (32 MiB) on every GPU that loads the
// library, held until the process exits.  Calls whose workspace would not fit
// are rejected with FA_ERR_WORKSPACE before anything is launched.  Every call
// on a device shares the one array: calls that overlap on the GPU (on two
// streams, or from two threads) race on it.  The array keeps the previous
// call's contents; the backward pass's preparation kernel rewrites every part
// it reads (it zeroes the dQ accumulator and writes both per-row terms), so
// no stale value reaches a result.
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol, not a device address: its device address is
// obtained with cudaGetSymbolAddress below and passed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array, looked up once per device
// with that device current.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0 || need > fa::kNoAllocScratchBytes) {
    // Invalid sizes, or a workspace larger than the scratch array: fa_bwd
    // without a workspace reports the same argument and alignment errors it
    // would report with one, checked in the same order, and FA_ERR_WORKSPACE
    // when the arguments are otherwise valid.  Nothing is launched.
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, nullptr, 0,
                  stream);
  }
  void* scratch = nullptr;
  const int rc = fa::scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, scratch,
                fa::kNoAllocScratchBytes, stream);
}
