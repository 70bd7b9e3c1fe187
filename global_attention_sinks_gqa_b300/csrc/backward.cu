// backward.cu -- backward of the sliding-window / global sink attention
// prefill on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method (MiMo-V2-Flash paper review, section 3.2: the sink logit is a
// learnable per-head parameter; sections 3.1 and 4 for shapes and RoPE): the
// gradients of sum(dout * out) with respect to q, k, v and the sink.  Per
// row, with p_j = exp(z_j - lse) (lse from the forward, sink included) and
// delta = dout . out:
//   dv_j += p_j dout;  dz_j = p_j (dout . v_j - delta);  dsink = -sum p_sink delta;
//   dq' = scale sum_j dz_j k'_j;  dk'_j += scale dz_j q';
// then dq, dk = the transposed rotation of dq', dk' on dims 0..63.
//
// Passes (ours):
//   bwd_prep_kernel      per token: q' and k' rotated dims (bf16, workspace),
//                        delta = dout . out, and per-block sink partials;
//   bwd_dkdv_kernel      one CTA per (sequence, KV head, 128-key block): keys
//                        are the MMA's 128 rows and the query rows that see
//                        them stream through as 64-column tiles (G heads x
//                        64/G tokens):  S^T = K Q'^T, dP^T = V dout^T, then
//                        P^T, dS^T (bf16, TMEM) and dV += P^T dout,
//                        dK += dS^T Q' with both accumulators in TMEM;
//   bwd_dq_kernel        one CTA per (sequence, KV head, 128-row query tile):
//                        S = Q' K^T, dP = dout V^T over 128-key blocks, dS to
//                        TMEM, dQ += dS K;
//   bwd_dsink_kernel     the sink partials summed in block order.
// Each gradient row is written once, by one thread, so no pass uses atomics
// and the results do not depend on scheduling.  The rotated dims are bf16
// operands here (the forward uses fp16 for them); all products accumulate in
// fp32.
//
// A key block's query tiles are walked from the sequence end down, so the
// CTAs of one KV head that run at the same time read the same query tile
// (L2 hits instead of one DRAM read per CTA).
//
// TMEM (512 columns).  dK/dV: S^T 0..63, dP^T 64..127, P^T 128..159 and dS^T
// 160..191 (bf16 pairs), dV 192..319, dK 320..511; a tile's S^T / dP^T are
// rewritten by the next tile's MMAs as soon as the row threads have read
// them, so the tensor core runs the next tile while they compute.  dQ: S
// 0..127, dP 128..255, dS 256..319, dQ 320..511.  An MMA costs about the same
// to issue at N = 64 as at N = 128, so the dQ kernel takes 128-key blocks;
// the dK/dV kernel stays at 64 query columns because dK (192 columns) and dV
// (128) leave only 192 for the rest.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"

namespace hattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBwdThreads = 256;  // warp 0 loads, warp 1 issues MMAs, warps 4-7 rows
constexpr int kNst = 3;           // pipeline stages of the streamed operand
constexpr int kPrepTok = 32;      // tokens per block of the prep pass
constexpr int kPrepWarps = 8;

// ---- prep ------------------------------------------------------------------

__device__ __forceinline__ int seq_of(const int* cu, int batch, long t) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Rotated dims (2i, 2i+1) and (2i+32, 2i+33) of one head row (i = lane % 16)
// from its raw pairs x = (2i, 2i+1), y = (2i+32, 2i+33).
__device__ __forceinline__ uint2 rotate_pair(uint32_t xr, uint32_t yr, float2 cs0, float2 cs1) {
  const float2 x = unpack_bf16x2(xr), y = unpack_bf16x2(yr);
  const float a0 = x.x * cs0.x - y.x * cs0.y, a1 = x.y * cs1.x - y.y * cs1.y;
  const float b0 = y.x * cs0.x + x.x * cs0.y, b1 = y.y * cs1.x + x.y * cs1.y;
  return make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(b0, b1));
}

// Rotated dims 0..63 of nh head rows of one token: half-warps take alternate
// heads; kU head pairs are loaded before any is stored, so the loads of a
// group are in flight together.
template <int kU>
__device__ __forceinline__ void rotate_heads(const __nv_bfloat16* __restrict__ src,
                                             __nv_bfloat16* __restrict__ dst, int nh, int half,
                                             int i2, float2 cs0, float2 cs1) {
  for (int h0 = 0; h0 < nh; h0 += 2 * kU) {
    uint32_t x[kU], y[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int h = h0 + 2 * u + half;
      x[u] = y[u] = 0u;
      if (h < nh) {
        x[u] = __ldg(reinterpret_cast<const unsigned int*>(src + long(h) * kDqk + i2));
        y[u] = __ldg(reinterpret_cast<const unsigned int*>(src + long(h) * kDqk + i2 + 32));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int h = h0 + 2 * u + half;
      if (h < nh) {
        const uint2 r = rotate_pair(x[u], y[u], cs0, cs1);
        *reinterpret_cast<uint32_t*>(dst + long(h) * kRopeDim + i2) = r.x;
        *reinterpret_cast<uint32_t*>(dst + long(h) * kRopeDim + i2 + 32) = r.y;
      }
    }
  }
}

__global__ void __launch_bounds__(kPrepWarps * 32)
    bwd_prep_kernel(const BackwardArgs a) {
  extern __shared__ float sp[];  // [warp][hq] sink partials
  constexpr int kU = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, i2 = 2 * (lane & 15);
  for (int h = threadIdx.x; h < kPrepWarps * a.hq; h += blockDim.x) sp[h] = 0.f;
  __syncthreads();
  float* spw = sp + warp * a.hq;
  const __nv_bfloat16* __restrict__ q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* __restrict__ kk = static_cast<const __nv_bfloat16*>(a.k);
  __nv_bfloat16* __restrict__ qr = static_cast<__nv_bfloat16*>(a.q_rot);
  __nv_bfloat16* __restrict__ kr = static_cast<__nv_bfloat16*>(a.k_rot);
  const uint4* __restrict__ o4 = static_cast<const uint4*>(a.out);
  const uint4* __restrict__ g4 = static_cast<const uint4*>(a.dout);
  for (int k = 0; k < kPrepTok / kPrepWarps; ++k) {
    const long t = long(blockIdx.x) * kPrepTok + warp + k * kPrepWarps;
    if (t >= a.total) break;
    const int b = seq_of(a.cu_seqlens, a.batch, t);
    const int p = int(t - __ldg(a.cu_seqlens + b));
    const float2 cs0 = rope_cos_sin(p, a.freqs.hi[i2], a.freqs.lo[i2]);
    const float2 cs1 = rope_cos_sin(p, a.freqs.hi[i2 + 1], a.freqs.lo[i2 + 1]);
    rotate_heads<kU>(q + t * a.hq * kDqk, qr + t * a.hq * kRopeDim, a.hq, half, i2, cs0, cs1);
    rotate_heads<kU>(kk + t * a.hkv * kDqk, kr + t * a.hkv * kRopeDim, a.hkv, half, i2, cs0, cs1);
    // delta = dout . out, 16 lanes per head row (8 dims each)
    for (int h0 = 0; h0 < a.hq; h0 += 2 * kU) {
      uint4 ov[kU], gv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int h = h0 + 2 * u + half;
        ov[u] = gv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (h < a.hq) {
          ov[u] = __ldg(o4 + (t * a.hq + h) * 16 + (lane & 15));
          gv[u] = __ldg(g4 + (t * a.hq + h) * 16 + (lane & 15));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int h = h0 + 2 * u + half;
        const uint32_t* ow = reinterpret_cast<const uint32_t*>(&ov[u]);
        const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[u]);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = unpack_bf16x2(ow[e]), y = unpack_bf16x2(gw[e]);
          d = fmaf(x.x, y.x, d);
          d = fmaf(x.y, y.y, d);
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        if ((lane & 15) == 0 && h < a.hq) {
          a.delta[t * a.hq + h] = d;
          const float ps = exp2f((__ldg(a.sink + h) - __ldg(a.lse + t * a.hq + h)) * kLog2e);
          spw[h] -= ps * d;
        }
      }
    }
  }
  __syncthreads();
  for (int h = threadIdx.x; h < a.hq; h += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < kPrepWarps; ++w) s += sp[w * a.hq + h];
    a.sink_part[long(blockIdx.x) * a.hq + h] = s;
  }
}

// One block per head: thread i sums partials i, i + 256, ... in order, then a
// fixed tree over the 256 sums (the same order on every run).
__global__ void __launch_bounds__(256) bwd_dsink_kernel(const BackwardArgs a) {
  __shared__ float red[256];
  const int h = blockIdx.x;
  float s = 0.f;
  for (long i = threadIdx.x; i < a.nprep; i += 256) s += a.sink_part[i * a.hq + h];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.dsink[h] = red[0];
}

// ---- shared pieces of the two MMA kernels -----------------------------------

struct BwdBars {
  uint64_t fixed_full;            // the operand loaded once per CTA
  uint64_t st_full[kNst], st_empty[kNst];
  uint64_t s_full, s_free, p_full, acc_done, drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kBoxBytes128 = 128 * 128;  // [128 rows][64 dims] bf16
constexpr int kBoxBytes64 = 64 * 128;    // [64 rows][64 dims] bf16
constexpr int kFixedBytes = 5 * kBoxBytes128;         // 3 boxes of 192 dims + 2 of 128
constexpr int kStageBytes = 5 * kBoxBytes64;
constexpr int kOffStage = kFixedBytes;
constexpr int kOffRowData = kOffStage + kNst * kStageBytes;   // dK/dV: lse2 / delta per stage
constexpr int kOffBar = kOffRowData + kNst * 2 * 64 * 4;
constexpr int kBwdSmem = kOffBar + 256 + 1024;                 // + alignment slack
static_assert(sizeof(BwdBars) <= 256, "barrier area");
static_assert(kBwdSmem <= 232448, "shared memory");

__device__ __forceinline__ uint8_t* smem_base_1k(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// 32 fp32 TMEM columns of this thread's row -> 16 bf16 pairs, times f.
__device__ __forceinline__ void pack_scaled(const uint32_t* v, float f, uint32_t* o) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    o[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * f, __uint_as_float(v[2 * e + 1]) * f);
}

__device__ __forceinline__ void store_row64(void* dst, const uint32_t* w) {
  uint4* d = static_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
}

// Epilogue pieces of a 192-dim gradient row held in TMEM columns
// taddr..taddr+191 of this thread's lane, times f, to bf16 at dst.  All lanes
// call them (tcgen05.ld is warp-wide); only `write` lanes store.
// Dims 0..63, turned back by the row's RoPE angle (the transpose of the
// forward rotation):
__device__ __forceinline__ void finish_rot64(uint32_t taddr, float f, int pos,
                                             const RopeFreqs& fr, bool write,
                                             __nv_bfloat16* dst) {
  uint32_t x[32], y[32];
  tmem_ld32_nowait(taddr, x);
  tmem_ld32_nowait(taddr + 32, y);
  tmem_ld_wait();
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 c0 = rope_cos_sin(pos, fr.hi[i], fr.lo[i]);
    const float2 c1 = rope_cos_sin(pos, fr.hi[i + 1], fr.lo[i + 1]);
    const float gx0 = __uint_as_float(x[i]) * f, gy0 = __uint_as_float(y[i]) * f;
    const float gx1 = __uint_as_float(x[i + 1]) * f, gy1 = __uint_as_float(y[i + 1]) * f;
    w[i >> 1] = pack_bf16x2(gx0 * c0.x + gy0 * c0.y, gx1 * c1.x + gy1 * c1.y);
    w[16 + (i >> 1)] = pack_bf16x2(gy0 * c0.x - gx0 * c0.y, gy1 * c1.x - gx1 * c1.y);
  }
  if (write) {
    store_row64(dst, w);
    store_row64(dst + 32, w + 16);
  }
}
// 32 plain dims starting at dim d0:
__device__ __forceinline__ void finish_chunk32(uint32_t taddr, float f, bool write,
                                               __nv_bfloat16* dst, int d0) {
  uint32_t v[32], o[16];
  tmem_ld32_nowait(taddr + d0, v);
  tmem_ld_wait();
  pack_scaled(v, f, o);
  if (write) store_row64(dst + d0, o);
}

__device__ __forceinline__ void bwd_init(BwdBars* bars, uint32_t st_full_count) {
  mbar_init(&bars->fixed_full, 1);
  for (int s = 0; s < kNst; ++s) {
    mbar_init(&bars->st_full[s], st_full_count);
    mbar_init(&bars->st_empty[s], 1);
  }
  mbar_init(&bars->s_full, 1);
  mbar_init(&bars->s_free, 4);
  mbar_init(&bars->p_full, 4);
  mbar_init(&bars->acc_done, 1);
  mbar_init(&bars->drain, 1);
  bars->abort = 0;
  mbar_fence_init();
}

// ---- dK / dV -----------------------------------------------------------------

// Unit u: (key block kb, sequence b, KV head g), key blocks in ascending order
// so that a global layer's longest units (its first keys) start first; each
// walks its query tiles from the last one down.
template <int G, bool WIN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mKr, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mQr,
                    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mDO,
                    const BackwardArgs a) {
  constexpr int TQ = 64 / G;  // tokens per 64-column query tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_base_1k(smem_raw);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + kOffBar);
  volatile int* abort = &bars->abort;
  float* rowdata = reinterpret_cast<float*>(smem + kOffRowData);  // [stage][lse2 | delta][64]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int per = a.batch * a.hkv;
  const int kb = blockIdx.x / per, rem = blockIdx.x - kb * per;
  const int b = rem / a.hkv, g = rem - b * a.hkv;
  // a sequence with out-of-range offsets is skipped (its key block 0 reports it)
  int tok0, L;
  if (!seq_slice(a.cu_seqlens, b, a.total, a.max_seqlen, a.ctl, kb == 0 && threadIdx.x == 0,
                 tok0, L))
    return;  // uniform over the CTA, before any barrier or TMEM use
  const int k0 = kb * 128;
  if (k0 >= L) return;  // uniform over the CTA, before any barrier or TMEM use
  const int qend = WIN ? min(L, k0 + 128 + a.window - 1) : L;
  const int ntile = (qend - k0 + TQ - 1) / TQ;

  if (threadIdx.x == 0) {
    bwd_init(bars, 1 + 32);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_map(&mQr);
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mDO);
      mbar_arrive_expect_tx(&bars->fixed_full, kFixedBytes);
      tma_load_3d(smem, &mKr, &bars->fixed_full, 0, g, tok0 + k0);
      tma_load_3d(smem + kBoxBytes128, &mK, &bars->fixed_full, 64, g, tok0 + k0);
      tma_load_3d(smem + 2 * kBoxBytes128, &mK, &bars->fixed_full, 128, g, tok0 + k0);
      tma_load_3d(smem + 3 * kBoxBytes128, &mV, &bars->fixed_full, 0, g, tok0 + k0);
      tma_load_3d(smem + 4 * kBoxBytes128, &mV, &bars->fixed_full, 64, g, tok0 + k0);
    }
    int filled = 0;
    for (int i = 0; i < ntile; ++i) {
      const int s = i % kNst;
      if (i >= kNst && !warp_wait(&bars->st_empty[s], ((i / kNst) - 1) & 1, a.ctl, abort)) break;
      const int tq0 = k0 + (ntile - 1 - i) * TQ;
      uint8_t* st = smem + kOffStage + s * kStageBytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->st_full[s], kStageBytes);
        tma_load_3d(st, &mQr, &bars->st_full[s], 0, g * G, tok0 + tq0);
        tma_load_3d(st + kBoxBytes64, &mQ, &bars->st_full[s], 64, g * G, tok0 + tq0);
        tma_load_3d(st + 2 * kBoxBytes64, &mQ, &bars->st_full[s], 128, g * G, tok0 + tq0);
        tma_load_3d(st + 3 * kBoxBytes64, &mDO, &bars->st_full[s], 0, g * G, tok0 + tq0);
        tma_load_3d(st + 4 * kBoxBytes64, &mDO, &bars->st_full[s], 64, g * G, tok0 + tq0);
      }
      float* rd = rowdata + s * 128;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = lane + 32 * cc;
        const int p = tq0 + c / G;
        float l2 = 0.f, de = 0.f;
        if (p < L) {
          const long idx = long(tok0 + p) * a.hq + g * G + c % G;
          l2 = __ldg(a.lse + idx) * kLog2e;
          de = __ldg(a.delta + idx);
        }
        rd[c] = l2;
        rd[64 + c] = de;
      }
      mbar_arrive(&bars->st_full[s]);
      filled = i + 1;
    }
    // copies still in flight must land before the CTA may exit
    if (lane == 0) {
      mbar_wait_drain(&bars->fixed_full, 0, a.ctl);
      for (int i = max(0, filled - kNst); i < filled; ++i)
        mbar_wait_drain(&bars->st_full[i % kNst], (i / kNst) & 1, a.ctl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_s = make_idesc_bf16(128, 64, 0, 0);
    const uint32_t id_dv = make_idesc_bf16(128, 128, 0, 1);
    const uint32_t id_dk = make_idesc_bf16(128, 192, 0, 1);
    const uint32_t sb = smem_u32(smem);
    const uint64_t dk_a = make_sdesc_sw128(sb, 16, 1024);                       // K, K-major
    const uint64_t dv_a = make_sdesc_sw128(sb + 3 * kBoxBytes128, 16, 1024);    // V, K-major
    bool ok = warp_wait(&bars->fixed_full, 0, a.ctl, abort);
    auto issue_s = [&](int i) {
      const uint32_t st = sb + kOffStage + (i % kNst) * kStageBytes;
      const uint64_t qd = make_sdesc_sw128(st, 16, 1024);
      const uint64_t gd = make_sdesc_sw128(st + 3 * kBoxBytes64, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 12; ++kk)
        umma_ss(tmem, dk_a + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4),
                qd + uint64_t(((kk >> 2) * kBoxBytes64 + (kk & 3) * 32) >> 4), id_s, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ss(tmem + 64, dv_a + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4),
                gd + uint64_t(((kk >> 2) * kBoxBytes64 + (kk & 3) * 32) >> 4), id_s, kk > 0);
      umma_commit(&bars->s_full);
    };
    bool issued = false;
    for (int i = 0; ok && i < ntile; ++i) {
      const int s = i % kNst;
      if (i == 0) {
        if (!warp_wait(&bars->st_full[0], 0, a.ctl, abort)) break;
        tc_fence_after();
        if (lane == 0) issue_s(0);
        issued = true;
      }
      if (i + 1 < ntile) {
        const int s1 = (i + 1) % kNst;
        if (!warp_wait(&bars->st_full[s1], ((i + 1) / kNst) & 1, a.ctl, abort)) break;
        if (!warp_wait(&bars->s_free, i & 1, a.ctl, abort)) break;
        tc_fence_after();
        if (lane == 0) issue_s(i + 1);
      }
      if (!warp_wait(&bars->p_full, i & 1, a.ctl, abort)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sb + kOffStage + s * kStageBytes;
        const uint64_t qb = make_sdesc_sw128(st, kBoxBytes64, 1024);                 // Q', MN-major
        const uint64_t gb = make_sdesc_sw128(st + 3 * kBoxBytes64, kBoxBytes64, 1024);  // dout
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          umma_ts(tmem + 192, tmem + 128 + kk * 8, gb + uint64_t((kk * 2048) >> 4), id_dv, acc);
          umma_ts(tmem + 320, tmem + 160 + kk * 8, qb + uint64_t((kk * 2048) >> 4), id_dk, acc);
        }
        // completes with dV / dK of this tile: its stage may be refilled and its
        // P^T / dS^T columns rewritten
        umma_commit(&bars->st_empty[s]);
        if (i + 1 == ntile) umma_commit(&bars->acc_done);
      }
      __syncwarp();
    }
    // every MMA issued must complete before TMEM is released
    if (issued && lane == 0) {
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.ctl);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ one thread per key
    const int r = (warp & 3) * 32 + lane;
    const int j = k0 + r;  // this thread's key position
    const bool jvalid = j < L;
    const uint32_t t_row = tmem + (uint32_t((warp & 3) * 32) << 16);
    bool ok = true;
    for (int i = 0; i < ntile; ++i) {
      const int s = i % kNst;
      const int tq0 = k0 + (ntile - 1 - i) * TQ;
      if (!warp_wait(&bars->s_full, i & 1, a.ctl, abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[64], dp[64];
      tmem_ld32_nowait(t_row, sv);
      tmem_ld32_nowait(t_row + 32, sv + 32);
      tmem_ld32_nowait(t_row + 64, dp);
      tmem_ld32_nowait(t_row + 96, dp + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free);
      if (!warp_wait(&bars->st_full[s], (i / kNst) & 1, a.ctl, abort)) { ok = false; break; }
      const float* rd = rowdata + s * 128;
      uint32_t pw[32], dw[32];
      const int d0 = tq0 - j;  // query position minus key position, column 0
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float pc[2], dc[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = d0 + (c + e) / G;
          const bool vis = jvalid && d >= 0 && (!WIN || d < a.window) && tq0 + (c + e) / G < L;
          const float x = __uint_as_float(sv[c + e]) * a.scale_log2 - rd[c + e];
          pc[e] = vis ? fast_exp2(x) : 0.f;
          dc[e] = vis ? pc[e] * (__uint_as_float(dp[c + e]) - rd[64 + c + e]) : 0.f;
        }
        pw[c >> 1] = pack_bf16x2(pc[0], pc[1]);
        dw[c >> 1] = pack_bf16x2(dc[0], dc[1]);
      }
      // the previous tile's dV / dK products have read its P^T / dS^T (its
      // stage's empty barrier cannot move on before this tile is handed over)
      if (i > 0 && !warp_wait(&bars->st_empty[(i - 1) % kNst], ((i - 1) / kNst) & 1, a.ctl, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32(t_row + 128, pw);
      tmem_st32(t_row + 160, dw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
    }
    if (ok && warp_wait(&bars->acc_done, 0, a.ctl, abort)) {
      tc_fence_after();
      const long row = long(tok0 + j) * a.hkv + g;
      // dV = sum p dout (no scale)
      __nv_bfloat16* dvr = static_cast<__nv_bfloat16*>(a.dv) + row * kDv;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32], o[16];
        tmem_ld32_nowait(t_row + 192 + 32 * ch, v);
        tmem_ld_wait();
        pack_scaled(v, 1.f, o);
        if (jvalid) store_row64(dvr + 32 * ch, o);
      }
      __nv_bfloat16* dkr = static_cast<__nv_bfloat16*>(a.dk) + row * kDqk;
      finish_rot64(t_row + 320, a.scale, j, a.freqs, jvalid, dkr);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) finish_chunk32(t_row + 320, a.scale, jvalid, dkr, 64 + 32 * ch);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---- dQ ----------------------------------------------------------------------

// Shared memory of the dQ kernel: Q' and dout of the tile (5 boxes of
// [128 rows][64 dims]), two K buffers of 128 keys (3 boxes each: K is read by
// S = Q' K^T and again by dQ += dS K, which runs after the next block's S) and
// one V buffer (2 boxes: V is read only by dP = dout V^T and is refilled as
// soon as that completes).
constexpr int kDqOffK = kFixedBytes;
constexpr int kDqKBytes = 3 * kBoxBytes128;
constexpr int kDqOffV = kDqOffK + 2 * kDqKBytes;
constexpr int kDqOffBar = kDqOffV + 2 * kBoxBytes128;
constexpr int kDqSmem = kDqOffBar + 256 + 1024;
static_assert(kDqSmem <= 232448, "shared memory");

struct DqBars {
  // V(it) is free once dP(it) is done: the producer reads that from the
  // phase of s_full (committed with it; the next phase needs V(it + 1))
  uint64_t fixed_full, fixed_empty, k_full[2], k_empty[2], v_full;
  uint64_t s_full, s_free, p_full, acc_done, acc_free, drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBars) <= 256, "barrier area");

// Unit u: (query tile, sequence b, KV head g); a global layer's latest (longest)
// tiles first.  An empty unit (tile past its sequence's end) is skipped, and
// so is every unit of a sequence whose offsets are out of range (`report`:
// record that; the loader, which walks every unit, reports).
struct DqUnit {
  int b, g, tok0, L, t0, kstart, nblk;
};
template <int G, bool WIN>
__device__ __forceinline__ bool dq_unit(int u, const BackwardArgs& a, int nqt, DqUnit& du,
                                        bool report = false) {
  constexpr int TQ = 128 / G;
  const int per = a.batch * a.hkv;
  const int q_ord = u / per, rem = u - q_ord * per;
  const int qt = WIN ? q_ord : nqt - 1 - q_ord;
  du.b = rem / a.hkv;
  du.g = rem - du.b * a.hkv;
  if (!seq_slice(a.cu_seqlens, du.b, a.total, a.max_seqlen, a.ctl, report && q_ord == 0,
                 du.tok0, du.L))
    return false;
  du.t0 = qt * TQ;
  if (du.t0 >= du.L) return false;
  du.kstart = WIN ? max(0, du.t0 - a.window + 1) : 0;
  const int kend = min(du.L, du.t0 + TQ);
  du.nblk = (kend - du.kstart + 127) / 128;
  return true;
}

// CTA c takes units c, c + grid, ... (a grid of one CTA per unit, or one per
// SM); the block counters (K / V buffers, S / dS hand-offs) run on across
// units, so a unit's loads and first products overlap the previous unit's
// last products and epilogue.
// 128-key blocks: TMEM S 0..127, dP 128..255, dS 256..319 (bf16 pairs), dQ
// 320..511.
template <int G, bool WIN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap mQr, const __grid_constant__ CUtensorMap mQ,
                  const __grid_constant__ CUtensorMap mDO, const __grid_constant__ CUtensorMap mKr,
                  const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                  const BackwardArgs a, int nqt, int nunits) {
  constexpr int BN = 128;  // keys per block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_base_1k(smem_raw);
  DqBars* bars = reinterpret_cast<DqBars*>(smem + kDqOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->fixed_full, 1);
    mbar_init(&bars->fixed_empty, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bars->k_full[j], 1);
      mbar_init(&bars->k_empty[j], 1);
    }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 4);
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->acc_free, 4);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_map(&mQr);
      tma_prefetch_map(&mKr);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
      int it = 0, nu = 0;        // blocks and units whose loads were issued
      int kfill = 0, vfill = 0;  // K and V copies issued
      bool ok = true;
      for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
        DqUnit du;
        if (!dq_unit<G, WIN>(u, a, nqt, du, true)) continue;
        // Q' and dout of the tile, once the previous tile's products are done with them
        if (nu > 0 && !mbar_wait(&bars->fixed_empty, (nu - 1) & 1, a.ctl, abort)) break;
        const int qrow = du.tok0 + du.t0;
        mbar_arrive_expect_tx(&bars->fixed_full, kFixedBytes);
        tma_load_3d(smem, &mQr, &bars->fixed_full, 0, du.g * G, qrow);
        tma_load_3d(smem + kBoxBytes128, &mQ, &bars->fixed_full, 64, du.g * G, qrow);
        tma_load_3d(smem + 2 * kBoxBytes128, &mQ, &bars->fixed_full, 128, du.g * G, qrow);
        tma_load_3d(smem + 3 * kBoxBytes128, &mDO, &bars->fixed_full, 0, du.g * G, qrow);
        tma_load_3d(smem + 4 * kBoxBytes128, &mDO, &bars->fixed_full, 64, du.g * G, qrow);
        ++nu;
        for (int i = 0; i < du.nblk; ++i, ++it) {
          const int kr0 = du.tok0 + du.kstart + BN * i;
          const int j = it & 1;
          if (it >= 2 && !mbar_wait(&bars->k_empty[j], ((it >> 1) - 1) & 1, a.ctl, abort)) {
            ok = false;
            break;
          }
          uint8_t* kb = smem + kDqOffK + j * kDqKBytes;
          mbar_arrive_expect_tx(&bars->k_full[j], kDqKBytes);
          tma_load_3d(kb, &mKr, &bars->k_full[j], 0, du.g, kr0);
          tma_load_3d(kb + kBoxBytes128, &mK, &bars->k_full[j], 64, du.g, kr0);
          tma_load_3d(kb + 2 * kBoxBytes128, &mK, &bars->k_full[j], 128, du.g, kr0);
          ++kfill;
          if (it >= 1 && !mbar_wait(&bars->s_full, (it - 1) & 1, a.ctl, abort)) {
            ok = false;
            break;
          }
          uint8_t* vb = smem + kDqOffV;
          mbar_arrive_expect_tx(&bars->v_full, 2 * kBoxBytes128);
          tma_load_3d(vb, &mV, &bars->v_full, 0, du.g, kr0);
          tma_load_3d(vb + kBoxBytes128, &mV, &bars->v_full, 64, du.g, kr0);
          ++vfill;
        }
      }
      // copies still in flight must land before the CTA may exit: the last
      // fill of each barrier
      if (nu > 0) mbar_wait_drain(&bars->fixed_full, (nu - 1) & 1, a.ctl);
      for (int f = max(0, kfill - 2); f < kfill; ++f)
        mbar_wait_drain(&bars->k_full[f & 1], (f >> 1) & 1, a.ctl);
      if (vfill > 0) mbar_wait_drain(&bars->v_full, (vfill - 1) & 1, a.ctl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_s = make_idesc_bf16(128, BN, 0, 0);
    const uint32_t id_dq = make_idesc_bf16(128, 192, 0, 1);
    const uint32_t sb = smem_u32(smem);
    const uint64_t qa = make_sdesc_sw128(sb, 16, 1024);                      // Q', K-major
    const uint64_t ga = make_sdesc_sw128(sb + 3 * kBoxBytes128, 16, 1024);   // dout, K-major
    const uint64_t vd = make_sdesc_sw128(sb + kDqOffV, 16, 1024);            // V, K-major
    // S(it) = Q' K^T once K has landed, then dP(it) = dout V^T once V has;
    // first: the unit's Q' / dout must have landed; last: they may be refilled
    // once these products complete
    auto issue_s = [&](int it, bool first, int nu, bool last) -> bool {
      if (first && !warp_wait(&bars->fixed_full, nu & 1, a.ctl, abort)) return false;
      if (!warp_wait(&bars->k_full[it & 1], (it >> 1) & 1, a.ctl, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t kd = make_sdesc_sw128(sb + kDqOffK + (it & 1) * kDqKBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk)
          umma_ss(tmem, qa + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4),
                  kd + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4), id_s, kk > 0);
      }
      __syncwarp();
      if (!warp_wait(&bars->v_full, it & 1, a.ctl, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + BN, ga + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4),
                  vd + uint64_t(((kk >> 2) * kBoxBytes128 + (kk & 3) * 32) >> 4), id_s, kk > 0);
        umma_commit(&bars->s_full);
        if (last) umma_commit(&bars->fixed_empty);
      }
      __syncwarp();
      return true;
    };
    // dQ += dS K(it); the unit's first block overwrites dQ, so it waits for the
    // previous unit's epilogue to have read it
    auto issue_dq = [&](int it, bool first, int nu, bool last) -> bool {
      if (first && nu > 0 && !warp_wait(&bars->acc_free, (nu - 1) & 1, a.ctl, abort))
        return false;
      if (!warp_wait(&bars->p_full, it & 1, a.ctl, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t kb = make_sdesc_sw128(sb + kDqOffK + (it & 1) * kDqKBytes, kBoxBytes128,
                                             1024);  // K', MN-major
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts(tmem + 320, tmem + 2 * BN + kk * 8, kb + uint64_t((kk * 2048) >> 4), id_dq,
                  (!first || kk > 0) ? 1u : 0u);
        // completes with this block's dQ product: its K buffer may be refilled
        // and its dS columns rewritten
        umma_commit(&bars->k_empty[it & 1]);
        if (last) umma_commit(&bars->acc_done);
      }
      __syncwarp();
      return true;
    };
    // the CTA's blocks in order: block counter, first / last of its unit, unit counter
    int u = int(blockIdx.x) - int(gridDim.x), i = 0, it = 0, nu = -1;
    DqUnit du;
    du.nblk = 0;
    auto advance = [&](int& bit, bool& bfirst, bool& blast, int& bnu) -> bool {
      while (i >= du.nblk) {
        u += gridDim.x;
        i = 0;
        du.nblk = 0;
        if (u >= nunits) return false;
        if (dq_unit<G, WIN>(u, a, nqt, du)) ++nu;
      }
      bit = it++;
      bfirst = i == 0;
      blast = i + 1 == du.nblk;
      bnu = nu;
      ++i;
      return true;
    };
    bool issued = false, ok = true;
    int c_it = 0, c_nu = 0, n_it = 0, n_nu = 0;  // current block and the next one
    bool c_first = false, c_last = false, n_first = false, n_last = false;
    bool have_c = advance(c_it, c_first, c_last, c_nu);
    if (have_c) {
      issued = true;
      ok = issue_s(c_it, c_first, c_nu, c_last);
    }
    while (ok && have_c) {
      const bool have_n = advance(n_it, n_first, n_last, n_nu);
      if (have_n && !n_first) {
        // same unit: the next block's S / dP first (they overlap this block's row work)
        if (!warp_wait(&bars->s_free, c_it & 1, a.ctl, abort)) break;
        if (!issue_s(n_it, n_first, n_nu, n_last)) break;
        if (!issue_dq(c_it, c_first, c_nu, c_last)) break;
      } else {
        // unit boundary: finish this unit's dQ first
        if (!issue_dq(c_it, c_first, c_nu, c_last)) break;
        if (have_n) {
          if (!warp_wait(&bars->s_free, c_it & 1, a.ctl, abort)) break;
          if (!issue_s(n_it, n_first, n_nu, n_last)) break;
        }
      }
      have_c = have_n;
      c_it = n_it;
      c_first = n_first;
      c_last = n_last;
      c_nu = n_nu;
    }
    if (issued && lane == 0) {
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.ctl);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------- one thread per row
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_row = tmem + (uint32_t((warp & 3) * 32) << 16);
    int it = 0, nu = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
      DqUnit du;
      if (!dq_unit<G, WIN>(u, a, nqt, du)) continue;
      const int p = du.t0 + r / G;  // query position
      const int h = du.g * G + r % G;
      const bool valid = p < du.L;
      const long orow = long(du.tok0 + p) * a.hq + h;
      const float l2 = valid ? __ldg(a.lse + orow) * kLog2e : 0.f;
      const float de = valid ? __ldg(a.delta + orow) : 0.f;
      for (int i = 0; i < du.nblk; ++i, ++it) {
        if (!warp_wait(&bars->s_full, it & 1, a.ctl, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t dw[64];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t sv[64], dp[64];
          tmem_ld32_nowait(t_row + 64 * hb, sv);
          tmem_ld32_nowait(t_row + 64 * hb + 32, sv + 32);
          tmem_ld32_nowait(t_row + BN + 64 * hb, dp);
          tmem_ld32_nowait(t_row + BN + 64 * hb + 32, dp + 32);
          tmem_ld_wait();
          if (hb == 1) {
            // S and dP are in registers: the next block's products may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free);
          }
          const int d0 = p - (du.kstart + BN * i + 64 * hb);  // query minus key position, col 0
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float dc[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int d = d0 - (c + e);
              const bool vis = valid && d >= 0 && (!WIN || d < a.window);
              const float x = __uint_as_float(sv[c + e]) * a.scale_log2 - l2;
              dc[e] = vis ? fast_exp2(x) * (__uint_as_float(dp[c + e]) - de) : 0.f;
            }
            dw[32 * hb + (c >> 1)] = pack_bf16x2(dc[0], dc[1]);
          }
        }
        // the previous block's dQ product has read its dS (that K buffer's empty
        // barrier cannot move on before this block is handed over)
        if (it > 0 &&
            !warp_wait(&bars->k_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, a.ctl, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32(t_row + 2 * BN, dw);
        tmem_st32(t_row + 2 * BN + 32, dw + 32);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
      if (!ok || !warp_wait(&bars->acc_done, nu & 1, a.ctl, abort)) { ok = false; break; }
      tc_fence_after();
      __nv_bfloat16* dqr = static_cast<__nv_bfloat16*>(a.dq) + orow * kDqk;
      finish_rot64(t_row + 320, a.scale, p, a.freqs, valid, dqr);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) finish_chunk32(t_row + 320, a.scale, valid, dqr, 64 + 32 * ch);
      // dQ has been read: the next unit's first product may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_free);
      ++nu;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int G>
cudaError_t launch_g(const BackwardArgs& a, cudaStream_t s) {
  const bool win = a.window > 0;
  auto kv = win ? bwd_dkdv_kernel<G, true> : bwd_dkdv_kernel<G, false>;
  auto qk = win ? bwd_dq_kernel<G, true> : bwd_dq_kernel<G, false>;
  cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qk, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
  if (e != cudaSuccess) return e;
  CUtensorMap mKr128, mK128, mV128, mQr64, mQ64, mDO64;
  if (!make_map(&mKr128, a.k_rot, a.total, a.hkv, kRopeDim, 1, 128) ||
      !make_map(&mK128, a.k, a.total, a.hkv, kDqk, 1, 128) ||
      !make_map(&mV128, a.v, a.total, a.hkv, kDv, 1, 128) ||
      !make_map(&mQr64, a.q_rot, a.total, a.hq, kRopeDim, G, 64 / G) ||
      !make_map(&mQ64, a.q, a.total, a.hq, kDqk, G, 64 / G) ||
      !make_map(&mDO64, a.dout, a.total, a.hq, kDv, G, 64 / G))
    return cudaErrorInvalidValue;
  const long per = long(a.batch) * a.hkv;
  const long nkb = (a.max_seqlen + 127) / 128;
  if (nkb * per > 0x7fffffffL) return cudaErrorInvalidValue;
  kv<<<unsigned(nkb * per), kBwdThreads, kBwdSmem, s>>>(mKr128, mK128, mV128, mQr64, mQ64, mDO64,
                                                         a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mQr128, mQ128, mDO128;
  if (!make_map(&mQr128, a.q_rot, a.total, a.hq, kRopeDim, G, 128 / G) ||
      !make_map(&mQ128, a.q, a.total, a.hq, kDqk, G, 128 / G) ||
      !make_map(&mDO128, a.dout, a.total, a.hq, kDv, G, 128 / G))
    return cudaErrorInvalidValue;
  const int nqt = (a.max_seqlen + 128 / G - 1) / (128 / G);
  if (long(nqt) * per > 0x7fffffffL) return cudaErrorInvalidValue;
  const int nunits = int(nqt * per);
  // window layers: short, equal units, a persistent CTA per SM; global layers:
  // one CTA per unit (their lengths differ, and the hardware's dispatch of the
  // next CTA to the SM that frees first balances them better than a fixed split)
  const int grid = win ? (nunits < num_sms() ? nunits : num_sms()) : nunits;
  qk<<<unsigned(grid), kBwdThreads, kDqSmem, s>>>(mQr128, mQ128, mDO128, mKr128, mK128, mV128, a,
                                                   nqt, nunits);
  return cudaGetLastError();
}

}  // namespace

long backward_prep_blocks(long total) { return (total + kPrepTok - 1) / kPrepTok; }

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s) {
  const size_t prep_smem = size_t(kPrepWarps) * a.hq * sizeof(float);
  if (prep_smem > 48 * 1024) return cudaErrorInvalidValue;
  bwd_prep_kernel<<<unsigned(a.nprep), kPrepWarps * 32, prep_smem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dsink_kernel<<<unsigned(a.hq), 256, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.max_seqlen == 0) return e;
  switch (a.hq / a.hkv) {
    case 1: return launch_g<1>(a, s);
    case 2: return launch_g<2>(a, s);
    case 4: return launch_g<4>(a, s);
    case 8: return launch_g<8>(a, s);
    case 16: return launch_g<16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hattn
