// decode.cu -- decode / MTP-verify attention over a KV cache, split over keys.
//
// Method: plmsmile notes on the MiMo series, MiMo-V2-Flash MTP: drafted
// tokens are verified by one parallel pass of the main model, so each
// sequence brings T = 1..4 query tokens (positions L-T .. L-1) that attend
// causally over the cache; "local window": an SWA layer's cache is a fixed
// ring (slot = pos % cap), a GA layer's cache grows (slot = pos).  The sink
// (paper review, section 3.2) joins the denominator once, in the merge.
//
// Decomposition (ours): one CTA per (sequence, KV head, key chunk).  Its
// G*T query rows (all query heads of the KV head, all T tokens) share every
// K/V byte it loads.  Keys stream through shared memory in blocks of 64 with
// 16-byte cp.async copies (double buffered, XOR-swizzled 16-byte chunks so
// ldmatrix reads are conflict free); QK^T and PV run on mma.sync m16n8k16
// (fp32 accumulate; the 64 rotated dims as fp16, the rest as bf16, matching
// the cache written by the append) with an online softmax in base 2.  Each of the
// four warps owns 16 rows and a slice of every key block; warps sharing rows
// merge by log-sum-exp at the end.  With one chunk the CTA finishes the rows
// itself (sink included); otherwise it writes (O / l, m + log2 l) and a merge
// kernel combines the chunks and the sink with one warp per output row.
#include <math.h>

#include "common.cuh"

namespace hattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBK = 64;                // keys per block
constexpr int kThreads = 128;
constexpr int kKRow = 384;             // bytes per key row (192 bf16)
constexpr int kVRow = 256;             // bytes per value row (128 bf16)
constexpr int kStageBytes = kBK * (kKRow + kVRow);
constexpr int kSmemBytes = 2 * kStageBytes;
constexpr int kSingleChunkMax = 1024;  // ranges up to this many keys use one chunk
constexpr int kChunk = 2048;           // keys per chunk otherwise

__device__ __forceinline__ uint32_t k_off(int key, int chunk) {
  return uint32_t(key * kKRow + ((chunk ^ (key & 7)) << 4));
}
__device__ __forceinline__ uint32_t v_off(int key, int chunk) {
  return uint32_t(key * kVRow + ((chunk ^ (key & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct SplitRange {
  int lo, kbeg, kend, nsplit;
};

// Keys the T queries of a sequence of length L can see, and this chunk's part.
__device__ __forceinline__ SplitRange split_range(int L, int T, int window, int chunk, int split) {
  SplitRange r;
  r.lo = window > 0 ? max(0, L - T - window + 1) : 0;
  r.nsplit = (L - r.lo + chunk - 1) / chunk;
  r.kbeg = r.lo + split * chunk;
  r.kend = min(L, r.kbeg + chunk);
  return r;
}

// MT: 16-row m-tiles per CTA (1, 2 or 4); the 4 warps = MT m-tiles x KW key groups.
template <int MT>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  constexpr int KW = 4 / MT;
  constexpr int KPW = kBK / KW;   // keys per warp per block
  constexpr int NT = KPW / 8;     // n-tiles of 8 keys
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int mt = warp % MT, kg = warp / MT;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.hq / a.hkv;
  const int T = a.T;
  const int L = __ldg(a.seqlens + b);
  if (L < T || L > a.max_seqlen_k || (!a.is_ring && L > a.cap)) {
    // a device-resident length the host could not check: skip, and say so
    if (threadIdx.x == 0 && split == 0 && kvh == 0) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
    return;
  }
  const int chunk = a.nsplit > 1 ? a.chunk : (1 << 30);
  const SplitRange sr = split_range(L, T, a.window, chunk, split);
  if (sr.kbeg >= sr.kend) return;  // no keys in this chunk (short sequence)

  // ---- the warp's 16 query rows: r = t * G + hh
  const int rows = G * T;
  const int r0 = mt * 16 + gid, r1 = r0 + 8;
  const bool v0 = r0 < rows, v1 = r1 < rows;
  const int t0r = v0 ? r0 / G : T - 1, t1r = v1 ? r1 / G : T - 1;
  const int p0 = L - T + t0r, p1 = L - T + t1r;  // query positions
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const long q0 = ((long(b) * T + t0r) * a.hq + kvh * G + (v0 ? r0 % G : 0)) * kDqk;
  const long q1 = ((long(b) * T + t1r) * a.hq + kvh * G + (v1 ? r1 % G : 0)) * kDqk;
  uint32_t qa[12][4];
#pragma unroll
  for (int kk = 0; kk < 12; ++kk) {
    const int c = kk * 16 + 2 * tig;
    qa[kk][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q + q0 + c)) : 0u;
    qa[kk][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q + q1 + c)) : 0u;
    qa[kk][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q + q0 + c + 8)) : 0u;
    qa[kk][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q + q1 + c + 8)) : 0u;
  }
  // RoPE on dims 0..63: dim d (k-step d/16) pairs with d + 32 (k-step + 2),
  // which this thread holds in the same register slot.
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
    for (int reg = 0; reg < 4; ++reg) {
      const int d = kk * 16 + ((reg & 2) ? 8 : 0) + 2 * tig;
      const int pos = (reg & 1) ? p1 : p0;
      const float2 x = unpack_bf16x2(qa[kk][reg]);
      const float2 y = unpack_bf16x2(qa[kk + 2][reg]);
      const float2 c0 = rope_cos_sin(pos, a.freqs.hi[d], a.freqs.lo[d]);
      const float2 c1 = rope_cos_sin(pos, a.freqs.hi[d + 1], a.freqs.lo[d + 1]);
      const float a0 = x.x * c0.x - y.x * c0.y, a1 = x.y * c1.x - y.y * c1.y;
      const float b0 = y.x * c0.x + x.x * c0.y, b1 = y.y * c1.x + x.y * c1.y;
      if (fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) > kF16Max)
        record_status(a.ctl, HATTN_ERR_INVALID_ARG);
      qa[kk][reg] = pack_f16x2(a0, a1);  // rotated dims are fp16 operands
      qa[kk + 2][reg] = pack_f16x2(b0, b1);
    }
  }

  // ---- key blocks
  const uint8_t* kc = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vc = static_cast<const uint8_t*>(a.v_cache);
  const long head_row0 = (long(b) * a.hkv + kvh) * a.cap;
  const int nb = (sr.kend - sr.kbeg + kBK - 1) / kBK;
  const uint32_t sbase = smem_u32(smem);

  auto load_block = [&](int blk, int stage) {
    const uint32_t ks = sbase + stage * kStageBytes;
    const uint32_t vs = ks + kBK * kKRow;
    const int key0 = sr.kbeg + blk * kBK;
    for (int e = threadIdx.x; e < kBK * 24; e += kThreads) {
      const int key = e / 24, ch = e - key * 24;
      const int kp = key0 + key;
      const bool in = kp < sr.kend;
      const long slot = a.is_ring ? (kp % a.cap) : kp;
      const uint8_t* src = kc + (head_row0 + (in ? slot : 0)) * kKRow + ch * 16;
      cp_async16(ks + k_off(key, ch), src, in ? 16u : 0u);
    }
    for (int e = threadIdx.x; e < kBK * 16; e += kThreads) {
      const int key = e >> 4, ch = e & 15;
      const int kp = key0 + key;
      const bool in = kp < sr.kend;
      const long slot = a.is_ring ? (kp % a.cap) : kp;
      const uint8_t* src = vc + (head_row0 + (in ? slot : 0)) * kVRow + ch * 16;
      cp_async16(vs + v_off(key, ch), src, in ? 16u : 0u);
    }
    cp_async_commit();
  };

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // l: exact sums (for lse); lr: sums of the bf16-rounded weights PV uses (for out)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, lr0 = 0.f, lr1 = 0.f;

  load_block(0, 0);
  for (int blk = 0; blk < nb; ++blk) {
    const int stage = blk & 1;
    if (blk + 1 < nb) {
      load_block(blk + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t ks = sbase + stage * kStageBytes;
    const uint32_t vs = ks + kBK * kKRow;
    const int key_w = kg * KPW;  // warp's first key within the block
    float s[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 12; ++kk) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        const int mi = lane >> 3, rr = lane & 7;
        const int key = key_w + (n + (mi >> 1)) * 8 + rr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks + k_off(key, kk * 2 + (mi & 1)), b0, b1, b2, b3);
        if (kk < 4) {  // rotated dims: fp16 x fp16
          mma_f16(s[n], qa[kk], b0, b1);
          mma_f16(s[n + 1], qa[kk], b2, b3);
        } else {
          mma_bf16(s[n], qa[kk], b0, b1);
          mma_bf16(s[n + 1], qa[kk], b2, b3);
        }
      }
    }
    // mask, block max, online update (base 2)
    const int kp_w = sr.kbeg + blk * kBK + key_w;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kp = kp_w + n * 8 + 2 * tig + e;
        const bool in = kp < sr.kend;
        const bool vis0 = in && kp <= p0 && (a.window == 0 || p0 - kp < a.window);
        const bool vis1 = in && kp <= p1 && (a.window == 0 || p1 - kp < a.window);
        s[n][e] = vis0 ? s[n][e] * a.scale_log2 : -INFINITY;
        s[n][2 + e] = vis1 ? s[n][2 + e] * a.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[n][e]);
        mx1 = fmaxf(mx1, s[n][2 + e]);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m0 - ms0), al1 = fast_exp2(m1 - ms1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f, rr0 = 0.f, rr1 = 0.f;
    uint32_t pa[NT / 2][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float e0 = fast_exp2(s[n][0] - ms0), e1 = fast_exp2(s[n][1] - ms0);
      const float e2 = fast_exp2(s[n][2] - ms1), e3 = fast_exp2(s[n][3] - ms1);
      const uint32_t u01 = pack_bf16x2(e0, e1), u23 = pack_bf16x2(e2, e3);
      const float2 r01 = unpack_bf16x2(u01), r23 = unpack_bf16x2(u23);
      rs0 += e0 + e1;
      rs1 += e2 + e3;
      rr0 += r01.x + r01.y;
      rr1 += r23.x + r23.y;
      pa[n >> 1][(n & 1) * 2 + 0] = u01;
      pa[n >> 1][(n & 1) * 2 + 1] = u23;
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
    lr0 = lr0 * al0 + rr0;
    lr1 = lr1 * al1 + rr1;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }
    // O += P V
#pragma unroll
    for (int j2 = 0; j2 < NT / 2; ++j2) {
      const uint32_t afr[4] = {pa[j2][0], pa[j2][1], pa[j2][2], pa[j2][3]};
      const int k0 = key_w + j2 * 16;
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int mi = lane >> 3, rr = lane & 7;
        const int key = k0 + (mi & 1) * 8 + rr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs + v_off(key, 2 * np + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * np], afr, b0, b1);
        mma_bf16(o[2 * np + 1], afr, b2, b3);
      }
    }
    __syncthreads();  // the stage is refilled next iteration
  }

  // ---- finish: row sums over the quad, then merge the KW key groups
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    lr0 += __shfl_xor_sync(0xffffffffu, lr0, off);
    lr1 += __shfl_xor_sync(0xffffffffu, lr1, off);
  }
  float* red = reinterpret_cast<float*>(smem);  // [4 warps][16 rows][128] + m, l, lr
  if (KW > 1) {
    float* ow = red + warp * (16 * 128);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int c = n * 8 + 2 * tig;
      ow[gid * 128 + c] = o[n][0];
      ow[gid * 128 + c + 1] = o[n][1];
      ow[(gid + 8) * 128 + c] = o[n][2];
      ow[(gid + 8) * 128 + c + 1] = o[n][3];
    }
    float* ml = red + 4 * 16 * 128 + warp * 48;
    if (tig == 0) {
      ml[gid] = m0;
      ml[gid + 8] = m1;
      ml[16 + gid] = l0;
      ml[16 + gid + 8] = l1;
      ml[32 + gid] = lr0;
      ml[32 + gid + 8] = lr1;
    }
    __syncthreads();
    if (kg != 0) return;
    float mm0 = m0, mm1 = m1;
    for (int w = 1; w < KW; ++w) {
      const float* mlw = red + 4 * 16 * 128 + (w * MT + mt) * 48;
      mm0 = fmaxf(mm0, mlw[gid]);
      mm1 = fmaxf(mm1, mlw[gid + 8]);
    }
    const float ms0 = mm0 == -INFINITY ? 0.f : mm0, ms1 = mm1 == -INFINITY ? 0.f : mm1;
    const float f0 = fast_exp2(m0 - ms0), f1 = fast_exp2(m1 - ms1);
    l0 *= f0;
    l1 *= f1;
    lr0 *= f0;
    lr1 *= f1;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= f0;
      o[n][1] *= f0;
      o[n][2] *= f1;
      o[n][3] *= f1;
    }
    for (int w = 1; w < KW; ++w) {
      const int ww = w * MT + mt;
      const float* mlw = red + 4 * 16 * 128 + ww * 48;
      const float g0 = fast_exp2(mlw[gid] - ms0), g1 = fast_exp2(mlw[gid + 8] - ms1);
      l0 += mlw[16 + gid] * g0;
      l1 += mlw[16 + gid + 8] * g1;
      lr0 += mlw[32 + gid] * g0;
      lr1 += mlw[32 + gid + 8] * g1;
      const float* ow2 = red + ww * (16 * 128);
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int c = n * 8 + 2 * tig;
        o[n][0] += ow2[gid * 128 + c] * g0;
        o[n][1] += ow2[gid * 128 + c + 1] * g0;
        o[n][2] += ow2[(gid + 8) * 128 + c] * g1;
        o[n][3] += ow2[(gid + 8) * 128 + c + 1] * g1;
      }
    }
    m0 = mm0;
    m1 = mm1;
  }

  // ---- write
  if (a.nsplit == 1) {
    // add the sink and finish the rows
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool valid = half ? v1 : v0;
      const int r = half ? r1 : r0;
      const float m = half ? m1 : m0;
      const float l = half ? l1 : l0;
      const float lr = half ? lr1 : lr0;
      if (!valid) continue;
      const int t = r / G, hh = r % G, h = kvh * G + hh;
      const float sl2 = __ldg(a.sink + h) * kLog2e;
      const float mt_ = fmaxf(m, sl2);
      const float msub = mt_ == -INFINITY ? 0.f : mt_;
      const float fo = fast_exp2(m - msub);
      const float sw = fast_exp2(sl2 - msub);
      const float lt = l * fo + sw;
      const float sc = fo / (lr * fo + sw);
      const long orow = (long(b) * T + t) * a.hq + h;
      uint32_t* op = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + orow * kDv);
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int c = n * 8 + 2 * tig;
        op[c >> 1] = pack_bf16x2(o[n][half * 2] * sc, o[n][half * 2 + 1] * sc);
      }
      if (tig == 0 && a.lse) a.lse[orow] = (msub + log2f(lt)) * kLn2;
    }
  } else {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool valid = half ? v1 : v0;
      const int r = half ? r1 : r0;
      const float m = half ? m1 : m0;
      const float l = half ? l1 : l0;
      const float lr = half ? lr1 : lr0;
      if (!valid) continue;
      const int t = r / G, hh = r % G, h = kvh * G + hh;
      const long prow = ((long(b) * a.hq + h) * T + t) * a.nsplit + split;
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      float2* pp = reinterpret_cast<float2*>(a.part_o + prow * kDv);
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int c = n * 8 + 2 * tig;
        pp[c >> 1] = make_float2(o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
      }
      if (tig == 0) a.part_lse[prow] = l > 0.f ? m + log2f(l) : -INFINITY;
    }
  }
}

// One warp per output row (b, t, h): combine the chunks' (O_i, lse_i) and the
// sink: lse = log2(sum_i 2^lse_i + 2^s), O = sum_i 2^(lse_i - lse) O_i.
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const long row = long(blockIdx.x) * 8 + (threadIdx.x >> 5);  // (b, t, h)
  const int T = a.T;
  if (row >= long(a.B) * T * a.hq) return;
  const int h = int(row % a.hq);
  const int t = int((row / a.hq) % T);
  const int b = int(row / (long(a.hq) * T));
  const int L = __ldg(a.seqlens + b);
  if (L < T || L > a.max_seqlen_k || (!a.is_ring && L > a.cap)) return;  // reported above
  const SplitRange sr = split_range(L, T, a.window, a.chunk, 0);
  const long prow0 = ((long(b) * a.hq + h) * T + t) * a.nsplit;
  const float sl2 = __ldg(a.sink + h) * kLog2e;
  float M = sl2;
  for (int i = 0; i < sr.nsplit; ++i) M = fmaxf(M, __ldg(a.part_lse + prow0 + i));
  const float msub = M == -INFINITY ? 0.f : M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = fast_exp2(sl2 - msub);
  for (int i = 0; i < sr.nsplit; ++i) {
    const float w = fast_exp2(__ldg(a.part_lse + prow0 + i) - msub);
    den += w;
    const float4 v = __ldg(reinterpret_cast<const float4*>(a.part_o + (prow0 + i) * kDv) + lane);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = 1.f / den;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + row * kDv)[lane] = pk;
  if (lane == 0 && a.lse) a.lse[row] = (msub + log2f(den)) * kLn2;
}

template <int MT>
cudaError_t launch_mt(const DecodeArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.nsplit, a.hkv, a.B);
  decode_kernel<MT><<<grid, kThreads, kSmemBytes, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.nsplit == 1) return e;
  const long rows = long(a.B) * a.T * a.hq;
  decode_merge_kernel<<<dim3(unsigned((rows + 7) / 8)), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(int max_seqlen_k, int T, int window, int* chunk) {
  const int range = window > 0 ? (max_seqlen_k < window + T - 1 ? max_seqlen_k : window + T - 1)
                               : max_seqlen_k;
  if (range <= kSingleChunkMax) {
    *chunk = range > 0 ? range : 1;
    return 1;
  }
  *chunk = kChunk;
  return (range + kChunk - 1) / kChunk;
}

size_t decode_workspace_bytes(int B, int T, int hq, int nsplit) {
  if (nsplit <= 1) return 0;
  const size_t rows = size_t(B) * hq * T * nsplit;
  const size_t o_bytes = rows * kDv * sizeof(float);
  const size_t l_bytes = rows * sizeof(float);
  return ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int rows = (a.hq / a.hkv) * a.T;
  if (rows <= 16) return launch_mt<1>(a, s);
  if (rows <= 32) return launch_mt<2>(a, s);
  return launch_mt<4>(a, s);
}

}  // namespace hattn
