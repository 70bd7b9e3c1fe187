// rope_append.cu -- partial RoPE of key rows and the KV-cache append.
//
// MiMo-V2-Flash paper review, section 3.1: RoPE is applied to the first 64 of
// the 192 Q/K dims; section 4: base 10K (SWA layers) / 5M (GA layers).
// plmsmile notes, MiMo-V2-Flash "local window": an SWA layer's KV cache does
// not grow with the history (a ring of `cap` slots here, slot = pos % cap);
// a GA layer's cache grows (slot = pos).
//
// Rotated keys are stored mixed-precision: dims 0..63 (the rotated ones) as
// IEEE fp16, dims 64..191 unchanged as bf16.  fp16 keeps 11 significant bits
// of the rotated values where bf16 keeps 8, which holds the logit error of
// the bf16/fp16 tensor-core path to a few 1e-4 (rotation changes the values,
// so unlike the untouched dims they are no longer exact bf16 numbers).  A
// rotated value beyond the fp16 range is recorded as HATTN_ERR_INVALID_ARG.
//
// The append kernels give one warp one 192-element key row: lane l < 24 holds
// the 16-byte chunk of dims 8l..8l+7, so the rotated pair (i, i + 32) of a
// lane l < 4 sits in lane l + 4 and one shuffle brings the partner over.
// Loads and stores are 128-bit and coalesced along the row.
#include "common.cuh"

namespace hattn {

namespace {

__device__ __forceinline__ uint4 rope_chunk(uint4 x, uint4 partner, int lane, int pos,
                                            const RopeFreqs& f, bool* overflow) {
  if (lane >= 8) return x;
  const bool first = lane < 4;  // dims i (first half) vs i + 32 (second half)
  const int i0 = 8 * (lane & 3);
  uint32_t xs[4] = {x.x, x.y, x.z, x.w};
  uint32_t ps[4] = {partner.x, partner.y, partner.z, partner.w};
  uint32_t ys[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 a = unpack_bf16x2(xs[w]);
    const float2 b = unpack_bf16x2(ps[w]);
    const float2 cs0 = rope_cos_sin(pos, f.hi[i0 + 2 * w], f.lo[i0 + 2 * w]);
    const float2 cs1 = rope_cos_sin(pos, f.hi[i0 + 2 * w + 1], f.lo[i0 + 2 * w + 1]);
    float y0, y1;
    if (first) {  // y[i] = x[i] c - x[i+32] s
      y0 = a.x * cs0.x - b.x * cs0.y;
      y1 = a.y * cs1.x - b.y * cs1.y;
    } else {      // y[i+32] = x[i+32] c + x[i] s
      y0 = a.x * cs0.x + b.x * cs0.y;
      y1 = a.y * cs1.x + b.y * cs1.y;
    }
    if (fabsf(y0) > kF16Max || fabsf(y1) > kF16Max) *overflow = true;
    ys[w] = pack_f16x2(y0, y1);
  }
  return make_uint4(ys[0], ys[1], ys[2], ys[3]);
}

// Rotate the key row at `src` (position pos) into `dst`.  Whole warp calls.
// Returns true (on the lane concerned) if a rotated value left the fp16 range.
__device__ __forceinline__ bool rope_key_row(const uint4* src, uint4* dst, int pos, int lane,
                                             const RopeFreqs& f) {
  uint4 x = make_uint4(0, 0, 0, 0);
  if (lane < 24) x = __ldg(src + lane);
  uint4 p;
  p.x = __shfl_xor_sync(0xffffffffu, x.x, 4);
  p.y = __shfl_xor_sync(0xffffffffu, x.y, 4);
  p.z = __shfl_xor_sync(0xffffffffu, x.z, 4);
  p.w = __shfl_xor_sync(0xffffffffu, x.w, 4);
  bool overflow = false;
  const uint4 y = rope_chunk(x, p, lane, pos, f, &overflow);
  if (lane < 24) dst[lane] = y;
  return overflow;
}

constexpr int kRowsPerBlock = 8;  // one warp per row

// Rotated-key pre-pass of prefill.  Only the rotated dims 0..63 of each key
// row are read and written (as fp16, into k_rot [total, hkv, 64]); the
// attention kernel reads dims 64..191 straight from k.  A task is one head's
// pair of 16-byte chunks (c, c + 4), c < 4 -- the dims i and i + 32 a rotation
// mixes; a block takes the 4 hkv tasks of each of its tokens (at most
// kPassMaxTok of them), TPT tasks per thread.  Each thread first issues all
// its tasks' loads; while they are in flight the block evaluates its tokens'
// 32 (cos, sin) pairs into shared memory, each pair once for all the heads.
// (One warp per token, with a token's loads issued only after its angles,
// took 22-23 us for 32768 tokens whatever the head count; this layout takes
// 18 us for 8 KV heads and 12 us for 4.)
constexpr int kPassThreads = 256;
constexpr int kPassMaxTok = 128;
constexpr int kPassTasks = 8;  // tasks per thread

template <int TPT>
__host__ __device__ inline int pass_tokens(int hkv) {
  const int t = TPT * kPassThreads / (4 * hkv);
  return t < 1 ? 1 : (t > kPassMaxTok ? kPassMaxTok : t);
}

template <int TPT>
__global__ void __launch_bounds__(kPassThreads) rope_keys_packed_kernel(
    const uint4* __restrict__ k, uint4* __restrict__ k_rot, const int* __restrict__ cu_seqlens,
    int batch, long total, int hkv, const RopeFreqs f, const DeviceCtl ctl,
    unsigned int* __restrict__ unit_ctr, int pos_off) {
  extern __shared__ float2 cs_tab[];  // [tokens of the block][32]
  __shared__ int pos_tab[kPassMaxTok];
  grid_dep_launch();  // the attention kernel after this one may start its setup
  if (unit_ctr != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *unit_ctr = 0u;
  const int ntok = pass_tokens<TPT>(hkv);
  const long n0 = long(blockIdx.x) * ntok;
  const int ntask = 4 * hkv * ntok;
  bool overflow = false;
  for (int base = 0; base < ntask; base += TPT * kPassThreads) {
    uint4 x[TPT], y[TPT];
#pragma unroll
    for (int u = 0; u < TPT; ++u) {
      const int task = base + u * kPassThreads + threadIdx.x;
      const int tok = task / (4 * hkv), h = (task >> 2) % hkv, c = task & 3;
      const long n = n0 + tok;
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      y[u] = x[u];
      if (task < ntask && n < total) {
        const uint4* src = k + (n * hkv + h) * 24;
        x[u] = __ldg(src + c);
        y[u] = __ldg(src + c + 4);
      }
    }
    if (base == 0) {
      for (int t = threadIdx.x; t < ntok; t += kPassThreads) {
        const long nt = n0 + t;
        int pos = int(nt) + pos_off;
        if (cu_seqlens != nullptr && nt < total) {
          int lo = 0, hi = batch;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu_seqlens + mid) <= nt) lo = mid; else hi = mid - 1;
          }
          pos = int(nt - __ldg(cu_seqlens + lo));
        }
        pos_tab[t] = pos;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < 32 * ntok; e += kPassThreads)
        cs_tab[e] = rope_cos_sin(pos_tab[e >> 5], f.hi[e & 31], f.lo[e & 31]);
      __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < TPT; ++u) {
      const int task = base + u * kPassThreads + threadIdx.x;
      const int tok = task / (4 * hkv), h = (task >> 2) % hkv, c = task & 3;
      const long n = n0 + tok;
      if (task < ntask && n < total) {
        const float2* cs = cs_tab + tok * 32;
        const uint32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        const uint32_t ys[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
        uint32_t a[4], b[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 8 * c + 2 * e;
          const float2 xv = unpack_bf16x2(xs[e]), yv = unpack_bf16x2(ys[e]);
          const float2 cs0 = cs[i], cs1 = cs[i + 1];
          const float a0 = xv.x * cs0.x - yv.x * cs0.y, a1 = xv.y * cs1.x - yv.y * cs1.y;
          const float b0 = yv.x * cs0.x + xv.x * cs0.y, b1 = yv.y * cs1.x + xv.y * cs1.y;
          if (fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) > kF16Max)
            overflow = true;
          a[e] = pack_f16x2(a0, a1);
          b[e] = pack_f16x2(b0, b1);
        }
        uint4* dst = k_rot + (n * hkv + h) * 8;
        dst[c] = make_uint4(a[0], a[1], a[2], a[3]);
        dst[c + 4] = make_uint4(b[0], b[1], b[2], b[3]);
      }
    }
  }
  if (overflow) record_status(ctl, HATTN_ERR_INVALID_ARG);
}

__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int* __restrict__ start_pos, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    int B, int T, int hkv, int cap, int is_ring, const RopeFreqs f, const DeviceCtl ctl,
    int from_len, const Paging pg) {
  const int lane = threadIdx.x & 31;
  const long row = long(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);  // (b, t, g)
  if (row >= long(B) * T * hkv) return;
  const int g = int(row % hkv);
  const int t = int((row / hkv) % T);
  const int b = int(row / (long(hkv) * T));
  const int pos = __ldg(start_pos + b) + t - (from_len ? T : 0);
  if (pos < 0 || (!is_ring && pos >= cap)) {
    if (lane == 0) record_status(ctl, HATTN_ERR_INVALID_ARG);
    return;  // whole warp leaves together: no shuffle is pending
  }
  long crow;
  if (pg.table != nullptr) {  // paged: the page of this position, its slot there
    const int lp = pos / pg.page;
    const int phys = __ldg(pg.table + long(b) * pg.stride + lp);
    if (phys < 0 || phys >= pg.num_pages) {
      if (lane == 0) record_status(ctl, HATTN_ERR_INVALID_ARG);
      return;
    }
    crow = (long(phys) * hkv + g) * pg.page + (pos - lp * pg.page);
  } else {
    const long slot = is_ring ? (pos % cap) : pos;
    crow = (long(b) * hkv + g) * cap + slot;
  }
  if (rope_key_row(k_new + row * 24, k_cache + crow * 24, pos, lane, f))
    record_status(ctl, HATTN_ERR_INVALID_ARG);
  if (lane < 16) v_cache[crow * 16 + lane] = __ldg(v_new + row * 16 + lane);
}

// Append of packed new tokens for a prefill over a cached prefix: row (token
// n of sequence b, KV head g) goes to slot prefix[b] + (n - cu[b]) of a linear
// cache, rotated like kv_append_kernel.  Rows past total * hkv zero, one warp
// per (sequence, KV head), the V slots [end, end + 256) past the sequence's
// new end: the attention kernel reads whole key blocks, and a stale value
// there must not turn a zero weight into NaN.  Block 0 also zeroes the
// attention kernel's work counter.
__global__ void __launch_bounds__(256) kv_append_packed_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int* __restrict__ cu_seqlens, const int* __restrict__ prefix,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int batch, long total, int hkv,
    int cap, const RopeFreqs f, const DeviceCtl ctl, unsigned int* __restrict__ unit_ctr) {
  grid_dep_launch();  // the attention kernel after this one may start its setup
  if (unit_ctr != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *unit_ctr = 0u;
  const int lane = threadIdx.x & 31;
  const long row = long(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  const long nrows = total * hkv;
  if (row < nrows) {
    const long n = row / hkv;
    const int g = int(row - n * hkv);
    int lo = 0, hi = batch;  // largest b with cu[b] <= n
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(cu_seqlens + mid) <= n) lo = mid; else hi = mid - 1;
    }
    const int pos = __ldg(prefix + lo) + int(n - __ldg(cu_seqlens + lo));
    if (pos < 0 || pos >= cap) {
      if (lane == 0) record_status(ctl, HATTN_ERR_INVALID_ARG);
      return;  // whole warp leaves together: no shuffle is pending
    }
    const long crow = (long(lo) * hkv + g) * cap + pos;
    if (rope_key_row(k_new + row * 24, k_cache + crow * 24, pos, lane, f))
      record_status(ctl, HATTN_ERR_INVALID_ARG);
    if (lane < 16) v_cache[crow * 16 + lane] = __ldg(v_new + row * 16 + lane);
    return;
  }
  const long z = row - nrows;
  if (z >= long(batch) * hkv) return;
  const int b = int(z / hkv), g = int(z - long(b) * hkv);
  const int end = max(0, __ldg(prefix + b) + __ldg(cu_seqlens + b + 1) - __ldg(cu_seqlens + b));
  const int stop = min(cap, end + 256);
  uint4* plane = v_cache + (long(b) * hkv + g) * cap * 16;
  for (int slot = end + (lane >> 4); slot < stop; slot += 2)
    plane[long(slot) * 16 + (lane & 15)] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_kv_append_packed(const void* k_new, const void* v_new, const int* cu_seqlens,
                                    const int* prefix, void* k_cache, void* v_cache, int batch,
                                    long total, int hkv, int cap, const RopeFreqs& f,
                                    const DeviceCtl& ctl, unsigned int* unit_ctr,
                                    cudaStream_t s) {
  const long rows = total * hkv + long(batch) * hkv;
  if (rows == 0) return cudaSuccess;
  const long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  kv_append_packed_kernel<<<dim3(unsigned(blocks)), 256, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), cu_seqlens, prefix,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), batch, total, hkv, cap, f, ctl,
      unit_ctr);
  return cudaGetLastError();
}

cudaError_t launch_rope_keys_packed(const void* k, void* k_rot, const int* cu_seqlens, int batch,
                                    long total, int hkv, const RopeFreqs& f, const DeviceCtl& ctl,
                                    cudaStream_t s, unsigned int* unit_ctr, int pos_off) {
  if (total == 0) return cudaSuccess;
  const int ntok = pass_tokens<kPassTasks>(hkv);
  const long blocks = (total + ntok - 1) / ntok;
  const size_t smem = size_t(ntok) * 32 * sizeof(float2);  // <= 32 KB
  rope_keys_packed_kernel<kPassTasks><<<dim3(unsigned(blocks)), kPassThreads, smem, s>>>(
      static_cast<const uint4*>(k), static_cast<uint4*>(k_rot), cu_seqlens, batch, total, hkv, f,
      ctl, unit_ctr, pos_off);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int* start_pos,
                             void* k_cache, void* v_cache, int B, int T, int hkv, int cap,
                             int is_ring, const RopeFreqs& f, const DeviceCtl& ctl,
                             cudaStream_t s, bool from_len, Paging pg) {
  const long rows = long(B) * T * hkv;
  if (rows == 0) return cudaSuccess;
  const long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  kv_append_kernel<<<dim3(unsigned(blocks)), 256, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), start_pos,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), B, T, hkv, cap, is_ring, f,
      ctl, from_len ? 1 : 0, pg);
  return cudaGetLastError();
}

}  // namespace hattn
