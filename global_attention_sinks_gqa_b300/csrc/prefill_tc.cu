// prefill_tc.cu -- sliding-window / global causal GQA attention with a
// per-head sink, prefill, on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method (MiMo-V2-Flash paper review, sections 3.1, 3.2 and 4; plmsmile notes
// on the MiMo series, MiMo-V2-Flash "local window" and "Learnable Attention
// Sink"): out = softmax over {visible keys, sink} of scale * q'.k' applied to
// the values (the sink has no value), lse = log of that denominator.  q' and
// k' carry RoPE on dims 0..63.  Keys arrive already rotated (the rotation of
// K is a separate pass); Q is rotated here, in shared memory, once per tile.
// The 64 rotated dims are fp16 operands (11 significant bits) and the other
// 128 dims bf16, so QK^T runs as 4 fp16 k-steps plus 8 bf16 k-steps into one
// fp32 accumulator.
//
// Work decomposition (ours): one CTA tile is 128 query rows = TQ = 128/G
// consecutive tokens x the G query heads that share one KV head, so every
// K/V tile fetched from memory serves all G heads (GQA reuse through the M
// dimension of the MMA).  The keys a tile needs are walked in blocks of BN
// rows starting at the window's first key: a sliding-window tile touches only
// the band [t0 - W + 1, t0 + TQ - 1]; a global tile walks up to its diagonal.
//
// CTA roles (192 threads, persistent over tiles):
//   warp 0      TMA producer: Q tile (3 boxes of 64 dims), K/V blocks
//               (2-stage ring), all 128-byte swizzled.
//   warp 1      TMEM allocator and single-thread MMA issuer:
//               S_j = Q K_j^T  (M=128, N=BN, K=192; A, B from smem)
//               O  += P_j V_j  (M=128, N=128, K=BN; P from TMEM, V from smem)
//   warps 2-5   one thread per query row (TMEM lane): RoPE of the Q tile,
//               masked online softmax in base 2 with the running max started
//               at the sink logit, P written back to TMEM as bf16 over the
//               consumed S columns, lazy O rescaling (only when the max grows
//               by more than 2^8), and the epilogue O / (l + 2^(s - m)).
// TMEM: S/P double buffer at columns 0 and 128, O at columns 256..383.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"

namespace hattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past 256x growth

template <int G, int BN, int QS>
struct Cfg {
  static constexpr int TQ = 128 / G;                 // tokens per tile
  static constexpr int kQBytes = 128 * 384;           // 3 boxes [128 rows][64 dims]
  static constexpr int kKBox = BN * 128;              // one 64-dim box of a K/V block
  static constexpr int kKBytes = 3 * kKBox;
  static constexpr int kVBytes = 2 * kKBox;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + QS * kQBytes;
  static constexpr int kOffV = kOffK + 2 * kKBytes;
  static constexpr int kOffBar = kOffV + 2 * kVBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
  static constexpr uint32_t kSCol0 = 0, kSCol1 = 128, kOCol = 256, kTmemCols = 512;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "BN");
  static_assert(kKBox % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Bars {
  uint64_t q_full[2], q_ready[2], q_empty[2];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, o_free, drain;
  uint32_t tmem_base;
  int abort;
};

struct TileInfo {
  int b, g, t0, L, kstart, nblk, tok0;
};

template <int G, int BN, bool GLOBAL>
__device__ __forceinline__ bool tile_info(int t_lin, const PrefillArgs& a, int nqt, TileInfo& ti) {
  constexpr int TQ = 128 / G;
  const int per_qt = a.batch * a.hkv;
  const int q_ord = t_lin / per_qt;
  const int rem = t_lin - q_ord * per_qt;
  // global tiles: longest (latest) first for balance; window tiles: in order
  const int qt = GLOBAL ? (nqt - 1 - q_ord) : q_ord;
  ti.b = rem / a.hkv;
  ti.g = rem - ti.b * a.hkv;
  ti.tok0 = __ldg(a.cu_seqlens + ti.b);
  ti.L = __ldg(a.cu_seqlens + ti.b + 1) - ti.tok0;
  ti.t0 = qt * TQ;
  if (ti.t0 >= ti.L) return false;
  const int qlast = min(ti.t0 + TQ, ti.L) - 1;
  ti.kstart = GLOBAL ? 0 : max(0, ti.t0 - a.window + 1);
  ti.nblk = (qlast + 1 - ti.kstart + BN - 1) / BN;
  return true;
}

template <int G, int BN, int QS, bool GLOBAL>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapV, const PrefillArgs a) {
  using C = Cfg<G, BN, QS>;
  constexpr int TQ = C::TQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (a.max_seqlen + TQ - 1) / TQ;
  const int ntiles = nqt * a.batch * a.hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_ready[i], 128);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapQ);
    tma_prefetch_map(&mapK);
    tma_prefetch_map(&mapV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t q_fills[2] = {0, 0}, kv_fills[2] = {0, 0};
      int tc = 0, it = 0;
      bool ok = true;
      for (int t_lin = blockIdx.x; t_lin < ntiles && ok; t_lin += gridDim.x) {
        TileInfo ti;
        if (!tile_info<G, BN, GLOBAL>(t_lin, a, nqt, ti)) continue;
        const int qs = tc % QS;
        const uint32_t qph = uint32_t(tc / QS) & 1u;
        if (!mbar_wait(&bars->q_empty[qs], qph ^ 1u, a.ctl, abort)) break;
        mbar_arrive_expect_tx(&bars->q_full[qs], C::kQBytes);
        uint8_t* qdst = smem + C::kOffQ + qs * C::kQBytes;
        for (int i = 0; i < 3; ++i)
          tma_load_3d(qdst + i * 16384, &mapQ, &bars->q_full[qs], 64 * i, ti.g * G,
                      ti.tok0 + ti.t0);
        ++q_fills[qs];
        for (int j = 0; j < ti.nblk; ++j, ++it) {
          const int s = it & 1;
          const uint32_t ph = uint32_t(it >> 1) & 1u;
          if (!mbar_wait(&bars->kv_empty[s], ph ^ 1u, a.ctl, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->kv_full[s], C::kKBytes + C::kVBytes);
          const int krow = ti.tok0 + ti.kstart + j * BN;
          uint8_t* kdst = smem + C::kOffK + s * C::kKBytes;
          uint8_t* vdst = smem + C::kOffV + s * C::kVBytes;
          for (int i = 0; i < 3; ++i)
            tma_load_3d(kdst + i * C::kKBox, &mapK, &bars->kv_full[s], 64 * i, ti.g, krow);
          for (int i = 0; i < 2; ++i)
            tma_load_3d(vdst + i * C::kKBox, &mapV, &bars->kv_full[s], 64 * i, ti.g, krow);
          ++kv_fills[s];
        }
        ++tc;
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int i = 0; i < 2; ++i) {
        if (q_fills[i]) mbar_wait_drain(&bars->q_full[i], (q_fills[i] - 1) & 1u, a.ctl);
        if (kv_fills[i]) mbar_wait_drain(&bars->kv_full[i], (kv_fills[i] - 1) & 1u, a.ctl);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_rot = make_idesc_f16(128, BN, 0, 0);   // dims 0..63
      constexpr uint32_t idesc_s = make_idesc_bf16(128, BN, 0, 0);    // dims 64..191
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, 0, 1);
      const uint32_t sbase = smem_u32(smem);
      int tc = 0, it = 0;
      long pv_issued = 0;  // PVs issued so far; PV k completes o_done phase k
      bool ok = true;
      auto issue_pv = [&](int itj, bool first_of_tile) -> bool {
        const int s = itj & 1;
        const uint32_t ph = uint32_t(itj >> 1) & 1u;
        if (!mbar_wait(&bars->p_full[s], ph, a.ctl, abort)) return false;
        if (first_of_tile && tc > 0) {
          if (!mbar_wait(&bars->o_free, uint32_t(tc - 1) & 1u, a.ctl, abort)) return false;
        }
        tc_fence_after();
        const uint32_t p_tmem = tmem + (s ? C::kSCol1 : C::kSCol0);
        const uint32_t v_base = sbase + C::kOffV + s * C::kVBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bdesc = make_sdesc_sw128(v_base + kk * 2048, C::kKBox, 1024);
          umma_ts(tmem + C::kOCol, p_tmem + kk * 8, bdesc, idesc_o,
                  (first_of_tile && kk == 0) ? 0u : 1u);
        }
        umma_commit(&bars->o_done);
        umma_commit(&bars->kv_empty[s]);
        ++pv_issued;
        return true;
      };
      for (int t_lin = blockIdx.x; t_lin < ntiles && ok; t_lin += gridDim.x) {
        TileInfo ti;
        if (!tile_info<G, BN, GLOBAL>(t_lin, a, nqt, ti)) continue;
        const int qs = tc % QS;
        const uint32_t qph = uint32_t(tc / QS) & 1u;
        if (!mbar_wait(&bars->q_ready[qs], qph, a.ctl, abort)) break;
        const uint32_t q_base = sbase + C::kOffQ + qs * C::kQBytes;
        for (int j = 0; j < ti.nblk && ok; ++j) {
          const int itj = it + j;
          const int s = itj & 1;
          const uint32_t ph = uint32_t(itj >> 1) & 1u;
          if (!mbar_wait(&bars->kv_full[s], ph, a.ctl, abort)) { ok = false; break; }
          // S buffer s last held P_{itj-2}; make sure the PV reading it is done
          // (waiting on the latest PV issued, never on an older phase).
          if (pv_issued > 0 && pv_issued - 1 >= itj - 2) {
            if (!mbar_wait(&bars->o_done, uint32_t(pv_issued - 1) & 1u, a.ctl, abort)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t k_base = sbase + C::kOffK + s * C::kKBytes;
          const uint32_t d_tmem = tmem + (s ? C::kSCol1 : C::kSCol0);
#pragma unroll
          for (int kk = 0; kk < 12; ++kk) {
            const uint64_t adesc =
                make_sdesc_sw128(q_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            const uint64_t bdesc =
                make_sdesc_sw128(k_base + (kk >> 2) * C::kKBox + (kk & 3) * 32, 16, 1024);
            umma_ss(d_tmem, adesc, bdesc, kk < 4 ? idesc_rot : idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->s_full[s]);
          if (j == ti.nblk - 1) umma_commit(&bars->q_empty[qs]);
          if (j >= 1 && !issue_pv(itj - 1, j == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(it + ti.nblk - 1, ti.nblk == 1)) break;
        it += ti.nblk;
        ++tc;
      }
      // every MMA issued must be complete before TMEM is released
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;            // query row of the tile
    const int hl = r % G;
    const int tl = r / G;
    const uint32_t lane_addr = uint32_t(quad * 32) << 16;
    int tc = 0, it = 0;
    for (int t_lin = blockIdx.x; t_lin < ntiles; t_lin += gridDim.x) {
      TileInfo ti;
      if (!tile_info<G, BN, GLOBAL>(t_lin, a, nqt, ti)) continue;
      const int qs = tc % QS;
      const uint32_t qph = uint32_t(tc / QS) & 1u;
      if (!warp_wait(&bars->q_full[qs], qph, a.ctl, abort)) break;
      const int qpos = ti.t0 + tl;
      // RoPE of this row's dims 0..63 (box 0, 128-byte row, 16-byte chunks
      // swizzled by row % 8): pairs (i, i + 32) live in chunks c and c + 4.
      {
        uint8_t* qrow = smem + C::kOffQ + qs * C::kQBytes + r * 128;
        uint4 ch[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) ch[c] = *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t* x = reinterpret_cast<uint32_t*>(&ch[c]);
          uint32_t* y = reinterpret_cast<uint32_t*>(&ch[c + 4]);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int i = 8 * c + 2 * w;
            const float2 xv = unpack_bf16x2(x[w]);
            const float2 yv = unpack_bf16x2(y[w]);
            const float2 c0 = rope_cos_sin(qpos, a.freqs.hi[i], a.freqs.lo[i]);
            const float2 c1 = rope_cos_sin(qpos, a.freqs.hi[i + 1], a.freqs.lo[i + 1]);
            const float a0 = xv.x * c0.x - yv.x * c0.y, a1 = xv.y * c1.x - yv.y * c1.y;
            const float b0 = yv.x * c0.x + xv.x * c0.y, b1 = yv.y * c1.x + xv.y * c1.y;
            if (fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) > kF16Max)
              record_status(a.ctl, HATTN_ERR_INVALID_ARG);
            x[w] = pack_f16x2(a0, a1);  // rotated dims are fp16 operands
            y[w] = pack_f16x2(b0, b1);
          }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4)) = ch[c];
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_ready[qs]);
      }
      const int h = ti.g * G + hl;
      const float sink_l2 = __ldg(a.sink + h) * kLog2e;
      float m = sink_l2;  // running max (log2 units), started at the sink logit
      float l = 0.f;      // running sum of exp2(x - m) over visible keys (for lse)
      float lr = 0.f;     // the same sum of the bf16-rounded weights PV uses (for out)
      bool ok = true;
      for (int j = 0; j < ti.nblk; ++j) {
        const int itj = it + j;
        const int s = itj & 1;
        const uint32_t ph = uint32_t(itj >> 1) & 1u;
        if (!warp_wait(&bars->s_full[s], ph, a.ctl, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_s = tmem + lane_addr + (s ? C::kSCol1 : C::kSCol0);
        const int kb = ti.kstart + j * BN;  // position of column 0
        // visible columns: kpos <= qpos and (global or qpos - kpos < W)
        const int c_hi = qpos - kb;                                     // inclusive
        const int c_lo = GLOBAL ? 0 : (qpos - a.window + 1 - kb);       // inclusive
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN; c += 16) {
          uint32_t v[16];
          tmem_ld16(t_s + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = c + e;
            if (col <= c_hi && col >= c_lo) mx = fmaxf(mx, __uint_as_float(v[e]));
          }
        }
        const float m_blk = mx * a.scale_log2;
        const float m_new = fmaxf(m, m_blk);
        const bool resc = (m == -INFINITY) ? (m_new != -INFINITY)
                                           : (m_new > m + kRescaleThreshold);
        const float m_use = resc ? m_new : m;
        const float alpha = resc ? exp2f(m - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O holds sum over earlier blocks scaled by 2^-m: rescale it once the
          // previous PV has landed.
          if (!warp_wait(&bars->o_done, uint32_t(itj - 1) & 1u, a.ctl, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t t_o = tmem + lane_addr + C::kOCol;
#pragma unroll
          for (int c = 0; c < 128; c += 16) {
            uint32_t v[16];
            tmem_ld16(t_o + c, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(t_o + c, v);
          }
          tmem_st_wait();
        }
        l *= alpha;
        lr *= alpha;
        m = m_use;
        const float msub = (m == -INFINITY) ? 0.f : m;
#pragma unroll
        for (int c = 0; c < BN; c += 16) {
          uint32_t v[16];
          tmem_ld16(t_s + c, v);
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int col = c + e;
            float p0 = 0.f, p1 = 0.f;
            if (col <= c_hi && col >= c_lo)
              p0 = fast_exp2(fmaf(__uint_as_float(v[e]), a.scale_log2, -msub));
            if (col + 1 <= c_hi && col + 1 >= c_lo)
              p1 = fast_exp2(fmaf(__uint_as_float(v[e + 1]), a.scale_log2, -msub));
            // out is normalised by the sum of the same bf16-rounded weights the
            // PV product uses; lse uses the exact sum
            pk[e >> 1] = pack_bf16x2(p0, p1);
            const float2 pr = unpack_bf16x2(pk[e >> 1]);
            l += p0 + p1;
            lr += pr.x + pr.y;
          }
          tmem_st8(t_s + (c >> 1), pk);  // P (bf16 pairs) over consumed S columns
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[s]);
      }
      if (!ok) break;
      // --------------------------------------------------------- epilogue
      if (!warp_wait(&bars->o_done, uint32_t(it + ti.nblk - 1) & 1u, a.ctl, abort)) break;
      tc_fence_after();
      const float msub = (m == -INFINITY) ? 0.f : m;
      const float sink_w = exp2f(sink_l2 - msub);
      const float l_tot = l + sink_w;
      const float inv = 1.f / (lr + sink_w);
      const bool valid = qpos < ti.L;
      const long orow = long(ti.tok0 + qpos) * a.hq + h;
      uint4* optr = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + orow * 256);
      const uint32_t t_o = tmem + lane_addr + C::kOCol;
#pragma unroll
      for (int c = 0; c < 128; c += 16) {
        uint32_t v[16];
        tmem_ld16(t_o + c, v);
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
        if (valid) {
          optr[(c >> 3) + 0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          optr[(c >> 3) + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if (valid && a.lse != nullptr) a.lse[orow] = (msub + log2f(l_tot)) * kLn2;
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      it += ti.nblk;
      ++tc;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over a [rows, heads, dim] bf16 tensor, 64-element (128-byte) inner
// box with 128-byte swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, long rows, int heads, int dim, int box_heads,
              int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(dim), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(dim) * 2, cuuint64_t(dim) * 2 * heads};
  cuuint32_t box[3] = {64, cuuint32_t(box_heads), cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int G, int BN, int QS, bool GLOBAL>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  using C = Cfg<G, BN, QS>;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.total, a.hq, kDqk, G, C::TQ) ||
      !make_map(&mk, a.k_rot, a.total, a.hkv, kDqk, 1, BN) ||
      !make_map(&mv, a.v, a.total, a.hkv, kDv, 1, BN))
    return cudaErrorInvalidValue;
  auto kern = prefill_kernel<G, BN, QS, GLOBAL>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long nqt = (a.max_seqlen + C::TQ - 1) / C::TQ;
  const long ntiles = nqt * a.batch * a.hkv;
  if (ntiles == 0) return cudaSuccess;
  const int grid = int(ntiles < num_sms() ? ntiles : num_sms());
  kern<<<grid, 192, C::kSmemBytes, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t s) {
  if (a.window == 0) return launch_t<G, 128, 1, true>(a, s);
  if (a.window <= 256) return launch_t<G, 80, 2, false>(a, s);
  return launch_t<G, 128, 1, false>(a, s);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  switch (a.hq / a.hkv) {
    case 1: return launch_g<1>(a, s);
    case 2: return launch_g<2>(a, s);
    case 4: return launch_g<4>(a, s);
    case 8: return launch_g<8>(a, s);
    case 16: return launch_g<16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hattn
