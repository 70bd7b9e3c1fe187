// hattn_api.cu -- the extern "C" entry points declared in include/hattn.h.
//
// Host-side validation (nothing is launched on a bad argument), workspace
// accounting, the device status word, and dispatch to the kernels.  The
// library allocates no device memory; the status word is a file-scope
// __device__ variable.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace hattn {

namespace {

__device__ unsigned int g_status_word;

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
constexpr int kMaxDevices = 64;
unsigned long long g_wait_limit_ns[kMaxDevices];
unsigned int* g_status_addr[kMaxDevices];
std::mutex g_mu;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Device address of this device's status word (looked up once per device,
// with that device current).
bool device_ctl(DeviceCtl* ctl) {
  const int dev = current_device();
  if (dev < 0) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || !p) return false;
    g_status_addr[dev] = static_cast<unsigned int*>(p);
  }
  ctl->status = g_status_addr[dev];
  ctl->wait_limit_ns = g_wait_limit_ns[dev] ? g_wait_limit_ns[dev] : kDefaultWaitLimitNs;
  return true;
}

// Host-side fault injection (hattn_test_fail_next_launches): calls that would
// launch kernels consume one pending failure each and report HATTN_ERR_CUDA
// before touching the device, as a failed launch would.
std::atomic<int> g_fail_launches{0};

bool take_injected_failure() {
  int n = g_fail_launches.load();
  while (n > 0)
    if (g_fail_launches.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

// device_ctl for the entry points that launch kernels.
bool launch_ctl(DeviceCtl* ctl) { return !take_injected_failure() && device_ctl(ctl); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shapes this build supports (the MiMo-V2-Flash attention layer and its
// variants): dqk 192, dv 128, RoPE on 64 dims, G = hq/hkv a power of two <= 16.
hattn_status_t check_heads(int hq, int hkv, int dqk, int dv, int rope_dim) {
  if (hq <= 0 || hkv <= 0 || dqk <= 0 || dv <= 0 || rope_dim < 0) return HATTN_ERR_INVALID_ARG;
  if (hq % hkv) return HATTN_ERR_INVALID_ARG;
  const int G = hq / hkv;
  if (dqk != kDqk || dv != kDv || rope_dim != kRopeDim) return HATTN_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return HATTN_ERR_UNSUPPORTED;
  return HATTN_OK;
}

bool finite_positive(float x) { return isfinite(x) && x > 0.f; }

}  // namespace

void make_rope_freqs(float base, RopeFreqs* f) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kRopeHalf; ++i) {
    const double theta = pow(double(base), -2.0 * double(i) / double(kRopeDim));
    const double turns = theta / two_pi;
    const float hi = float(turns);
    f->hi[i] = hi;
    f->lo[i] = float(turns - double(hi));
  }
}

namespace {

__global__ void lost_arrival_kernel(const DeviceCtl ctl) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none is ever made
    abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, ctl, reinterpret_cast<volatile int*>(&abort));
}

}  // namespace

cudaError_t launch_lost_arrival_selftest(const DeviceCtl& ctl, cudaStream_t s) {
  lost_arrival_kernel<<<1, 32, 0, s>>>(ctl);
  return cudaGetLastError();
}

// The argument checks of a decode step (everything but the workspace);
// *empty is set when there is nothing to launch (B == 0).
hattn_status_t decode_check_args(const void* q, const void* k_new, const void* v_new,
                                 const void* k_cache, const void* v_cache, const int* seqlens_k,
                                 const float* sink, const void* out, const float* lse, int B,
                                 int T, int hq, int hkv, int dqk, int dv, int cap, int is_ring,
                                 int window, int max_seqlen_k, int rope_dim, float rope_base,
                                 float softmax_scale, bool* empty) {
  *empty = false;
  hattn_status_t st = check_heads(hq, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (B < 0 || T <= 0 || cap <= 0 || window < 0 || max_seqlen_k < T ||
      (is_ring != 0 && is_ring != 1))
    return HATTN_ERR_INVALID_ARG;
  if (T > 8 || (hq / hkv) * T > 128) return HATTN_ERR_UNSUPPORTED;
  if (is_ring && window == 0) return HATTN_ERR_INVALID_ARG;  // a ring only holds a window
  // 64-bit: a window near INT_MAX must not wrap around
  if (is_ring && long(cap) < long(window) + T - 1) return HATTN_ERR_RING_TOO_SMALL;
  if (!is_ring && max_seqlen_k > cap) return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base) || !finite_positive(softmax_scale)) return HATTN_ERR_INVALID_ARG;
  if (B == 0) {
    *empty = true;
    return HATTN_OK;
  }
  if (!q || !k_cache || !v_cache || !seqlens_k || !sink || !out) return HATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seqlens_k) & 3u) || (reinterpret_cast<uintptr_t>(sink) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return HATTN_ERR_INVALID_ARG;
  const bool append = k_new != nullptr || v_new != nullptr;
  if (append && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
    return HATTN_ERR_INVALID_ARG;
  return HATTN_OK;
}

}  // namespace hattn

using namespace hattn;

extern "C" {

int hattn_version(void) { return 100; }

const char* hattn_status_string(hattn_status_t s) {
  switch (s) {
    case HATTN_OK: return "HATTN_OK";
    case HATTN_ERR_INVALID_ARG: return "HATTN_ERR_INVALID_ARG";
    case HATTN_ERR_UNSUPPORTED: return "HATTN_ERR_UNSUPPORTED";
    case HATTN_ERR_CUDA: return "HATTN_ERR_CUDA";
    case HATTN_ERR_RING_TOO_SMALL: return "HATTN_ERR_RING_TOO_SMALL";
    case HATTN_ERR_TIMEOUT: return "HATTN_ERR_TIMEOUT";
    case HATTN_ERR_WORKSPACE: return "HATTN_ERR_WORKSPACE";
  }
  return "HATTN_ERR_UNKNOWN";
}

namespace {
// Bytes of the rotated key dims 0..63 in a prefill workspace.
size_t prefill_rot_bytes(long total_tokens, int hkv) {
  return (size_t(total_tokens) * size_t(hkv) * kRopeDim * 2 + 255) / 256 * 256;
}
}  // namespace

size_t hattn_prefill_workspace_size(long total_tokens, int hkv, int dqk) {
  if (total_tokens <= 0 || hkv <= 0 || dqk <= 0) return 0;
  return prefill_rot_bytes(total_tokens, hkv) + 256;  // rotated dims, then the work counter
}

hattn_status_t hattn_prefill(const void* q, const void* k, const void* v, const float* sink,
                             void* out, float* lse, int batch, const int* cu_seqlens,
                             long total_tokens, int max_seqlen, int hq, int hkv, int dqk, int dv,
                             int rope_dim, float rope_base, int window, float softmax_scale,
                             void* workspace, size_t workspace_bytes, void* stream) {
  hattn_status_t st = check_heads(hq, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (batch <= 0 || total_tokens < 0 || max_seqlen < 0 || window < 0) return HATTN_ERR_INVALID_ARG;
  if (total_tokens > 2147483647L || max_seqlen > total_tokens) return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base) || !finite_positive(softmax_scale)) return HATTN_ERR_INVALID_ARG;
  if (total_tokens == 0) return HATTN_OK;
  if (!q || !k || !v || !sink || !out || !cu_seqlens) return HATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(workspace))
    return HATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3u || reinterpret_cast<uintptr_t>(lse) & 3u ||
      reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
    return HATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < hattn_prefill_workspace_size(total_tokens, hkv, dqk))
    return HATTN_ERR_WORKSPACE;
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillArgs a;
  a.q = q;
  a.k_rot = workspace;
  a.k_raw = k;
  a.unit_ctr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) +
                                               prefill_rot_bytes(total_tokens, hkv));
  a.v = v;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.cu_seqlens = cu_seqlens;
  a.batch = batch;
  a.total = total_tokens;
  a.max_seqlen = max_seqlen;
  a.hq = hq;
  a.hkv = hkv;
  a.window = window >= max_seqlen ? 0 : window;  // a window covering every key is global
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  make_rope_freqs(rope_base, &a.freqs);
  a.ctl = ctl;
  if (launch_rope_keys_packed(k, workspace, cu_seqlens, batch, total_tokens, hkv, a.freqs, ctl, s,
                              a.unit_ctr) != cudaSuccess)
    return HATTN_ERR_CUDA;
  a.after_pass = total_tokens > 0;  // the pass launched
  if (max_seqlen == 0) return HATTN_OK;
  if (launch_prefill(a, s) != cudaSuccess) return HATTN_ERR_CUDA;
  return HATTN_OK;
}

hattn_status_t hattn_prefill_shard(const void* q, const void* k, const void* v,
                                   const float* sink, void* out, float* lse, long shard_tokens,
                                   int halo, long pos0, int hq, int hkv, int dqk, int dv,
                                   int rope_dim, float rope_base, int window, float softmax_scale,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  hattn_status_t st = check_heads(hq, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (shard_tokens < 0 || halo < 0 || pos0 < halo || window < 0) return HATTN_ERR_INVALID_ARG;
  // positions are int on the device
  if (pos0 + shard_tokens > 2147483647L) return HATTN_ERR_INVALID_ARG;
  // the halo must hold every key a query of the shard can see: the last
  // window - 1 positions before the shard (a window layer), or all of them
  if (window > 0 ? long(halo) < (long(window) - 1 < pos0 ? long(window) - 1 : pos0)
                 : long(halo) != pos0)
    return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base) || !finite_positive(softmax_scale)) return HATTN_ERR_INVALID_ARG;
  if (shard_tokens == 0) return HATTN_OK;
  const long total_k = long(halo) + shard_tokens;
  if (!q || !k || !v || !sink || !out) return HATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(workspace))
    return HATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3u || reinterpret_cast<uintptr_t>(lse) & 3u)
    return HATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < hattn_prefill_workspace_size(total_k, hkv, dqk))
    return HATTN_ERR_WORKSPACE;
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillArgs a;
  a.q = q;
  a.k_rot = workspace;
  a.k_raw = k;
  a.unit_ctr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) +
                                               prefill_rot_bytes(total_k, hkv));
  a.v = v;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.cu_seqlens = nullptr;  // one sequence: the shard
  a.batch = 1;
  a.total = shard_tokens;
  a.max_seqlen = int(shard_tokens);
  a.hq = hq;
  a.hkv = hkv;
  // a window covering every key the shard holds is global
  a.window = long(window) >= total_k ? 0 : window;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  make_rope_freqs(rope_base, &a.freqs);
  a.ctl = ctl;
  a.total_k = total_k;
  a.lead = halo;
  a.rope_off = int(pos0 - halo);
  if (launch_rope_keys_packed(k, workspace, nullptr, 1, total_k, hkv, a.freqs, ctl, s, a.unit_ctr,
                              a.rope_off) != cudaSuccess)
    return HATTN_ERR_CUDA;
  a.after_pass = total_k > 0;  // the pass launched
  if (launch_prefill(a, s) != cudaSuccess) return HATTN_ERR_CUDA;
  return HATTN_OK;
}

size_t hattn_prefill_backward_workspace_size(long total_tokens, int hq, int hkv) {
  if (total_tokens <= 0 || hq <= 0 || hkv <= 0) return 0;
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t t = size_t(total_tokens);
  return r256(t * hq * kRopeDim * 2) + r256(t * hkv * kRopeDim * 2) + r256(t * hq * 4) +
         r256(size_t(backward_prep_blocks(total_tokens)) * hq * 4);
}

hattn_status_t hattn_prefill_backward(const void* q, const void* k, const void* v,
                                      const float* sink, const void* out, const float* lse,
                                      const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                      float* grad_sink, int batch, const int* cu_seqlens,
                                      long total_tokens, int max_seqlen, int hq, int hkv, int dqk,
                                      int dv, int rope_dim, float rope_base, int window,
                                      float softmax_scale, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  hattn_status_t st = check_heads(hq, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (batch <= 0 || total_tokens < 0 || max_seqlen < 0 || window < 0) return HATTN_ERR_INVALID_ARG;
  if (total_tokens > 2147483647L || max_seqlen > total_tokens) return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base) || !finite_positive(softmax_scale)) return HATTN_ERR_INVALID_ARG;
  if (!grad_sink || reinterpret_cast<uintptr_t>(grad_sink) & 3u) return HATTN_ERR_INVALID_ARG;
  if (total_tokens == 0) {
    // no rows: the sink gradient is an empty sum
    return cudaMemsetAsync(grad_sink, 0, size_t(hq) * 4, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? HATTN_OK
               : HATTN_ERR_CUDA;
  }
  if (!q || !k || !v || !sink || !out || !lse || !dout || !grad_q || !grad_k || !grad_v ||
      !cu_seqlens)
    return HATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(grad_q) || !aligned16(grad_k) || !aligned16(grad_v) || !aligned16(workspace))
    return HATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3u || reinterpret_cast<uintptr_t>(lse) & 3u ||
      reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
    return HATTN_ERR_INVALID_ARG;
  if (size_t(8) * hq * 4 > 48 * 1024) return HATTN_ERR_UNSUPPORTED;  // prep-pass partials
  if (!workspace ||
      workspace_bytes < hattn_prefill_backward_workspace_size(total_tokens, hq, hkv))
    return HATTN_ERR_WORKSPACE;
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t t = size_t(total_tokens);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BackwardArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  a.dq = grad_q;
  a.dk = grad_k;
  a.dv = grad_v;
  a.dsink = grad_sink;
  a.cu_seqlens = cu_seqlens;
  a.batch = batch;
  a.total = total_tokens;
  a.max_seqlen = max_seqlen;
  a.hq = hq;
  a.hkv = hkv;
  a.window = window >= max_seqlen ? 0 : window;  // a window covering every key is global
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  make_rope_freqs(rope_base, &a.freqs);
  a.ctl = ctl;
  a.q_rot = ws;
  ws += r256(t * hq * kRopeDim * 2);
  a.k_rot = ws;
  ws += r256(t * hkv * kRopeDim * 2);
  a.delta = reinterpret_cast<float*>(ws);
  ws += r256(t * hq * 4);
  a.sink_part = reinterpret_cast<float*>(ws);
  a.nprep = backward_prep_blocks(total_tokens);
  if (launch_backward(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return HATTN_ERR_CUDA;
  return HATTN_OK;
}

hattn_status_t hattn_prefill_cached(const void* q, const void* k_new, const void* v_new,
                                    void* k_cache, void* v_cache, const int* cu_seqlens,
                                    const int* prefix_lens, const float* sink, void* out,
                                    float* lse, int batch, long total_tokens, int max_seqlen,
                                    int max_prefix, int cap, int hq, int hkv, int dqk, int dv,
                                    int rope_dim, float rope_base, int window,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  hattn_status_t st = check_heads(hq, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (batch <= 0 || total_tokens < 0 || max_seqlen < 0 || max_prefix < 0 || window < 0 ||
      cap <= 0)
    return HATTN_ERR_INVALID_ARG;
  if (total_tokens > 2147483647L || max_seqlen > total_tokens) return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base) || !finite_positive(softmax_scale)) return HATTN_ERR_INVALID_ARG;
  if (total_tokens == 0) return HATTN_OK;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !cu_seqlens || !prefix_lens || !sink ||
      !out)
    return HATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
    return HATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3u || reinterpret_cast<uintptr_t>(lse) & 3u ||
      reinterpret_cast<uintptr_t>(cu_seqlens) & 3u || reinterpret_cast<uintptr_t>(prefix_lens) & 3u)
    return HATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < 256) return HATTN_ERR_WORKSPACE;
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillArgs a;
  a.q = q;
  a.k_rot = k_cache;
  a.k_raw = k_cache;
  a.unit_ctr = static_cast<unsigned int*>(workspace);
  a.v = v_cache;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.cu_seqlens = cu_seqlens;
  a.batch = batch;
  a.total = total_tokens;
  a.max_seqlen = max_seqlen;
  a.hq = hq;
  a.hkv = hkv;
  // a window covering every key of every sequence is global
  a.window = long(window) >= long(max_prefix) + max_seqlen ? 0 : window;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  make_rope_freqs(rope_base, &a.freqs);
  a.ctl = ctl;
  a.prefix = prefix_lens;
  a.cap = cap;
  if (launch_kv_append_packed(k_new, v_new, cu_seqlens, prefix_lens, k_cache, v_cache, batch,
                              total_tokens, hkv, cap, a.freqs, ctl, a.unit_ctr, s) != cudaSuccess)
    return HATTN_ERR_CUDA;
  a.after_pass = (total_tokens + batch) * long(hkv) > 0;  // the append launched
  if (max_seqlen == 0) return HATTN_OK;
  if (launch_prefill(a, s) != cudaSuccess) return HATTN_ERR_CUDA;
  return HATTN_OK;
}

hattn_status_t hattn_rope_kv_append(const void* k_new, const void* v_new, const int* start_pos,
                                    void* k_cache, void* v_cache, int B, int T, int hkv, int dqk,
                                    int dv, int cap, int is_ring, int rope_dim, float rope_base,
                                    void* stream) {
  hattn_status_t st = check_heads(hkv, hkv, dqk, dv, rope_dim);
  if (st != HATTN_OK) return st;
  if (B < 0 || T <= 0 || cap <= 0 || T > cap || (is_ring != 0 && is_ring != 1))
    return HATTN_ERR_INVALID_ARG;
  if (!finite_positive(rope_base)) return HATTN_ERR_INVALID_ARG;
  if (B == 0) return HATTN_OK;
  if (!k_new || !v_new || !start_pos || !k_cache || !v_cache) return HATTN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(start_pos) & 3u))
    return HATTN_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  RopeFreqs f;
  make_rope_freqs(rope_base, &f);
  if (launch_kv_append(k_new, v_new, start_pos, k_cache, v_cache, B, T, hkv, cap, is_ring, f,
                       ctl, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return HATTN_ERR_CUDA;
  return HATTN_OK;
}

size_t hattn_decode_workspace_size(int B, int T, int hq, int hkv, int dv, int max_seqlen_k,
                                   int window, int cap, int is_ring) {
  (void)hkv;
  (void)dv;
  if (B <= 0 || T <= 0 || hq <= 0 || max_seqlen_k <= 0 || window < 0 || cap <= 0) return 0;
  int chunk = 0;
  const int nsplit = decode_num_splits(max_seqlen_k, T, window, is_ring != 0, cap, &chunk);
  return decode_workspace_bytes(B, T, hq, nsplit);
}

namespace {

// hattn_decode() and hattn_decode_append(): k_new / v_new null for the former.
hattn_status_t decode_step(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                           const void* v_cache, const int* seqlens_k, const float* sink, void* out,
                           float* lse, int B, int T, int hq, int hkv, int dqk, int dv, int cap,
                           int is_ring, int window, int max_seqlen_k, int rope_dim,
                           float rope_base, float softmax_scale, void* workspace,
                           size_t workspace_bytes, void* stream, const Paging& pg = Paging()) {
  bool empty = false;
  hattn_status_t st = decode_check_args(q, k_new, v_new, k_cache, v_cache, seqlens_k, sink, out,
                                        lse, B, T, hq, hkv, dqk, dv, cap, is_ring, window,
                                        max_seqlen_k, rope_dim, rope_base, softmax_scale, &empty);
  if (st != HATTN_OK || empty) return st;
  // a window covering every key of a linear cache is global attention
  if (!is_ring && long(window) >= long(max_seqlen_k)) window = 0;
  DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seqlens = seqlens_k;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.T = T;
  a.hq = hq;
  a.hkv = hkv;
  a.cap = cap;
  a.is_ring = is_ring;
  a.window = window;
  a.max_seqlen_k = max_seqlen_k;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  make_rope_freqs(rope_base, &a.freqs);
  a.nsplit = decode_num_splits(max_seqlen_k, T, window, is_ring, cap, &a.chunk);
  a.k_new = k_new;
  a.v_new = v_new;
  a.pg = pg;
  const size_t need = decode_workspace_bytes(B, T, hq, a.nsplit);
  a.part_o = nullptr;
  a.part_lse = nullptr;
  if (need) {
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return HATTN_ERR_WORKSPACE;
    const size_t rows = size_t(B) * hq * T * a.nsplit;
    const size_t o_bytes = (rows * kDv * sizeof(float) + 255) / 256 * 256;
    const size_t l_bytes = (rows * sizeof(float) + 255) / 256 * 256;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + o_bytes);
    a.item_ctr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + o_bytes +
                                                 l_bytes);
  }
  if (!launch_ctl(&a.ctl)) return HATTN_ERR_CUDA;
  if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return HATTN_ERR_CUDA;
  return HATTN_OK;
}

}  // namespace

hattn_status_t hattn_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int* seqlens_k, const float* sink, void* out, float* lse, int B,
                            int T, int hq, int hkv, int dqk, int dv, int cap, int is_ring,
                            int window, int max_seqlen_k, int rope_dim, float rope_base,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return decode_step(q, nullptr, nullptr, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq,
                     hkv, dqk, dv, cap, is_ring, window, max_seqlen_k, rope_dim, rope_base,
                     softmax_scale, workspace, workspace_bytes, stream);
}

hattn_status_t hattn_decode_append(const void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, const int* seqlens_k,
                                   const float* sink, void* out, float* lse, int B, int T, int hq,
                                   int hkv, int dqk, int dv, int cap, int is_ring, int window,
                                   int max_seqlen_k, int rope_dim, float rope_base,
                                   float softmax_scale, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  if (B > 0 && (!k_new || !v_new)) return HATTN_ERR_INVALID_ARG;
  return decode_step(q, k_new, v_new, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv,
                     dqk, dv, cap, is_ring, window, max_seqlen_k, rope_dim, rope_base,
                     softmax_scale, workspace, workspace_bytes, stream);
}

hattn_status_t hattn_decode_append_paged(const void* q, const void* k_new, const void* v_new,
                                         void* k_pages, void* v_pages, const int* block_table,
                                         int table_stride, int num_pages, int page,
                                         const int* seqlens_k, const float* sink, void* out,
                                         float* lse, int B, int T, int hq, int hkv, int dqk,
                                         int dv, int window, int max_seqlen_k, int rope_dim,
                                         float rope_base, float softmax_scale, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (page <= 0 || page % 64 != 0 || table_stride <= 0 || num_pages <= 0)
    return HATTN_ERR_INVALID_ARG;
  if (long(table_stride) * page > 2147483647L) return HATTN_ERR_INVALID_ARG;
  if (B > 0 && (!k_new || !v_new || !block_table)) return HATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_table) & 3u) return HATTN_ERR_INVALID_ARG;
  Paging pg;
  pg.table = block_table;
  pg.stride = table_stride;
  pg.page = page;
  pg.num_pages = num_pages;
  return decode_step(q, k_new, v_new, k_pages, v_pages, seqlens_k, sink, out, lse, B, T, hq, hkv,
                     dqk, dv, table_stride * page, 0, window, max_seqlen_k, rope_dim, rope_base,
                     softmax_scale, workspace, workspace_bytes, stream, pg);
}

hattn_status_t hattn_check_device_status(void* stream) {
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return HATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ctl.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return HATTN_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(ctl.status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return HATTN_ERR_CUDA;
  }
  return static_cast<hattn_status_t>(word);
}

hattn_status_t hattn_set_wait_limit_ns(unsigned long long limit_ns) {
  const int dev = current_device();
  if (dev < 0) return HATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  g_wait_limit_ns[dev] = limit_ns;
  return HATTN_OK;
}

hattn_status_t hattn_selftest_lost_arrival(void* stream) {
  DeviceCtl ctl;
  if (!launch_ctl(&ctl)) return HATTN_ERR_CUDA;
  if (launch_lost_arrival_selftest(ctl, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return HATTN_ERR_CUDA;
  return HATTN_OK;
}

int hattn_test_fail_next_launches(int n) { return g_fail_launches.exchange(n > 0 ? n : 0); }

}  // extern "C"
