// decode_static_scratch.cu -- the decode / verify step for callers that
// cannot allocate device memory.
//
// hattn_decode() needs a workspace for the per-chunk partial results when a
// sequence's keys are split over several CTAs, and it expects the caller to
// allocate it.  Some callers cannot call cudaMalloc: code that runs inside a
// host framework which owns all device memory through its own pool and
// forbids side allocations, or a serving loop whose memory budget is fixed at
// start-up and may not grow while requests are in flight.  For them this file
// keeps the scratch in a fixed array in the library's own device memory and
// passes it to the unchanged decode path.
//
// The array lives in every GPU that loads the library, until the process
// exits.  In host code its name is only a host-side stand-in, not a device
// address, so the device address is looked up with cudaGetSymbolAddress once
// per device, with that device current, on the first call made on it.  The
// address is kept for the life of the process: it belongs to the device's
// context, so a cudaDeviceReset() (which ends that context) leaves it stale.
// A process that resets a device must not call this entry point on it again.
#include <mutex>

#include "hattn_internal.h"

namespace hattn {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[HATTN_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of this device's scratch array (nullptr on failure).
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace hattn

extern "C" hattn_status_t hattn_decode_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k,
    const float* sink, void* out, float* lse, int B, int T, int hq, int hkv, int dqk, int dv,
    int cap, int is_ring, int window, int max_seqlen_k, int rope_dim, float rope_base,
    float softmax_scale, void* stream) {
  // a malformed call reports its argument error, not a scratch shortfall
  bool empty = false;
  const hattn_status_t st = hattn::decode_check_args(
      q, nullptr, nullptr, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv, dqk, dv,
      cap, is_ring, window, max_seqlen_k, rope_dim, rope_base, softmax_scale, &empty);
  if (st != HATTN_OK || empty) return st;
  const size_t need =
      hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window, cap, is_ring);
  if (need > size_t(HATTN_DECODE_STATIC_SCRATCH_BYTES)) return HATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = hattn::scratch_for_current_device();
    if (scratch == nullptr) return HATTN_ERR_CUDA;
  }
  return hattn_decode(q, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv, dqk, dv, cap,
                      is_ring, window, max_seqlen_k, rope_dim, rope_base, softmax_scale, scratch,
                      need > 0 ? size_t(HATTN_DECODE_STATIC_SCRATCH_BYTES) : 0, stream);
}
