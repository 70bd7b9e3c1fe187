// decode.cu -- decode / MTP-verify attention over a KV cache, split over keys,
// on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method: plmsmile notes on the MiMo series, MiMo-V2-Flash MTP: drafted
// tokens are verified by one parallel pass of the main model, so each
// sequence brings T = 1..4 query tokens (positions L-T .. L-1) that attend
// causally over the cache; "local window": an SWA layer's cache is a fixed
// ring (slot = pos % cap), a GA layer's cache grows (slot = pos).  The sink
// (paper review, section 3.2) joins the denominator once, when a row is
// finished.
//
// Decomposition (ours).  A work item is (sequence, KV head, chunk of cache
// slots); its G*T query rows (all query heads of the KV head, all T tokens)
// share every K/V byte it loads.  A linear cache splits the visible positions
// into chunks of `chunk` keys; a ring's slots are split the same way (the key
// position of slot s is the one position of the last `cap` that is congruent
// to s).  The kernel is persistent: one CTA per SM walks the items
// round-robin.  The G*T <= 128 rows sit in a 128-row tile whose other rows
// are zero, so QK^T and PV are plain M=128 tensor-core products; the step is
// bound by streaming the cache, not by the multiply.
//
// CTA roles (192 threads):
//   warp 0      TMA producer: blocks of 64 cache slots (K: 3 boxes, V: 2 boxes
//               of [64 slots][64 dims], 128-byte swizzle) into a 5-stage ring,
//               running ahead across item boundaries; a stage is released by a
//               row thread once it has seen S of the block two later (that
//               QK^T was issued after the block's PV).
//   warp 1      TMEM allocator and single-thread MMA issuer:
//                 S_j = Q K_j^T (M=128, N=64, K=192; Q from TMEM) into one of
//                 two S buffers, O += P_j V_j (M=128, N=128, K=64, P from TMEM),
//               in the order QK_0, QK_1, PV_0, QK_2, PV_1, ... (the tensor core
//               runs them in issue order, so S may be rewritten right behind
//               the PV reading the P stored over it).
//   warps 2-5   one thread per tile row (TMEM lane); warps whose 32 rows are
//               all padding only keep the barriers: the row's Q from global
//               memory, RoPE in registers and into one of two TMEM Q buffers,
//               masked online softmax in base 2, P written back to TMEM as
//               bf16, lazy O rescaling, and the epilogue.  A single-chunk item
//               finishes its rows (sink included); otherwise it writes
//               (O / l, m + log2 l) and a merge kernel combines the chunks and
//               the sink with one warp per output row.  The epilogue waits on
//               a barrier committed after the item's last PV (o_done).
// TMEM: S_0 columns 0..63, S_1 64..127, O 128..255, Q buffers 256.. and 352..
#include <math.h>

#include "common.cuh"

namespace hattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past 256x growth
constexpr int kBK = 64;                    // cache slots per block
constexpr int kStages = 5;
constexpr int kBox = kBK * 128;            // [64 slots][64 dims] bf16
constexpr int kStageBytes = 5 * kBox;      // K: 3 boxes, V: 2 boxes
constexpr int kOffStage = 0;
constexpr int kOffBar = kOffStage + kStages * kStageBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr int kThreads = 192;
// TMEM: S_0 0..63, S_1 64..127, O 128..255, Q buffers 256..351 and 352..447
// (192 dims of a row as 96 packed pairs; rows >= G*T are padding).
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t s_col(uint32_t b) { return b ? 64u : 0u; }
constexpr uint32_t kOCol = 128;
__host__ __device__ constexpr uint32_t q_col(uint32_t qb) { return 256u + 96u * qb; }
constexpr int kSingleChunkMax = 1024;  // ranges up to this many keys use one chunk
constexpr int kChunkShort = 2048;      // keys per chunk for caches up to 16K keys
constexpr int kChunkLong = 4096;       // and beyond
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffStage % 1024 == 0 && kBox % 1024 == 0, "swizzle atoms must be 1024-byte aligned");

constexpr int kItemQueue = 4;        // items the producer may publish ahead
constexpr int kItemReaders = 1 + 4;  // the MMA issuer and the four row warps

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_ready[2], q_empty[2];
  // pv_done: after every PV (the rescale of O waits for the previous
  // block's); o_done: after an item's last PV (its epilogue waits on it:
  // pv_done's parity could alias there, since the row warps reach the
  // epilogue having seen only the PVs up to two blocks back complete)
  uint64_t s_full[2], p_full[2], pv_done, o_done, o_free, drain;
  uint64_t item_full[kItemQueue], item_empty[kItemQueue];
  uint32_t tmem_base;
  int abort;
  int item[kItemQueue];  // published virtual item indices, -1: no more
};

// Slots of the cache a work item covers.  Linear cache: the visible positions
// [lo, L) (lo > 0 only for a window), slot = position.  Ring: slots
// [0, min(L, cap)).  Either range is cut into chunks of `chunk` slots.
struct Item {
  int b, kvh, split, L, s_beg, s_end, nsplit;
  int ring_r, ring_off;  // slot s holds position s + ring_off + (s < ring_r ? cap : 0)
};

__device__ __forceinline__ bool slot_range(int L, const DecodeArgs& a, int& lo, int& hi) {
  if (a.is_ring) {
    lo = 0;
    hi = min(L, a.cap);
  } else {
    lo = a.window > 0 ? max(0, L - a.T - a.window + 1) : 0;
    // paged: blocks of 64 slots start on a multiple of 64, so a block never
    // straddles two pages (the extra leading slots are outside the window)
    if (a.pg.table != nullptr) lo &= ~63;
    hi = L;
  }
  return hi > lo;
}

__device__ __forceinline__ bool length_ok(int L, const DecodeArgs& a) {
  return L >= a.T && L <= a.max_seqlen_k && (a.is_ring || L <= a.cap);
}

// Virtual item v = (split, b, kvh), split-major so that the items of one CTA
// mix long and short sequences.  Returns 1 for a work item, 0 for an item past
// a sequence's last chunk, -1 for a sequence whose device-resident length the
// host could not check and that is skipped.
__device__ __forceinline__ int item_info(int v, const DecodeArgs& a, Item& it) {
  const int per = a.B * a.hkv;
  it.split = v / per;
  const int rem = v - it.split * per;
  it.b = rem / a.hkv;
  it.kvh = rem - it.b * a.hkv;
  it.L = __ldg(a.seqlens + it.b);
  if (!length_ok(it.L, a)) return -1;
  int lo, hi;
  if (!slot_range(it.L, a, lo, hi)) return 0;
  const int chunk = a.nsplit > 1 ? a.chunk : (1 << 30);
  it.nsplit = (hi - lo + chunk - 1) / chunk;
  if (it.nsplit > a.nsplit) return -1;  // would not fit the workspace the host sized
  if (it.split >= it.nsplit) return 0;
  it.s_beg = lo + it.split * chunk;
  it.s_end = min(hi, it.s_beg + chunk);
  // a ring keeps the last cap positions [L - cap, L): slot s holds the one
  // congruent to s (never written, and negative, while L < cap)
  it.ring_r = 0;
  it.ring_off = 0;
  if (a.is_ring) {
    const int base = it.L - a.cap;
    int r = base % a.cap;
    if (r < 0) r += a.cap;
    it.ring_r = r;
    it.ring_off = base - r;
  }
  return 1;
}

template <int BN>
__device__ __forceinline__ void ld_row(uint32_t taddr, uint32_t (&s)[BN]) {
#pragma unroll
  for (int c = 0; c < BN; c += 32) tmem_ld32_nowait(taddr + c, s + c);
  tmem_ld_wait();
#pragma unroll
  for (int e = 0; e < BN; ++e) tmem_reg_fence(s[e]);
}

// cos / sin of RoPE frequency i for this lane's token, when the G lanes
// sharing a token (lanes l with equal l / G) hold frequencies hl, hl + G, ...
// in own[] (hl = l % G).  Whole warp calls; i is a compile-time index.
template <int G>
__device__ __forceinline__ float2 shared_cos_sin(const float2 (&own)[32 / G], int i, int lane) {
  if (G == 1) return own[i];
  const int src = (lane & ~(G - 1)) | (i % G);
  return make_float2(__shfl_sync(0xffffffffu, own[i / G].x, src),
                     __shfl_sync(0xffffffffu, own[i / G].y, src));
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                  const __grid_constant__ CUtensorMap mapV, const DecodeArgs a, int nvirt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T;
  const int rows = G * T;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_ready[i], 128);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      // one P barrier per S buffer: QK_{j+1} is issued before PV_j waits for
      // P_j, so the softmax may finish block j+1 before that wait begins
      mbar_init(&bars->p_full[i], 128);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain, 1);
    for (int i = 0; i < kItemQueue; ++i) {
      mbar_init(&bars->item_full[i], 1);
      mbar_init(&bars->item_empty[i], kItemReaders);
    }
    bars->abort = 0;
  }
  if (threadIdx.x == 0) mbar_fence_init();
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapQ);
    tma_prefetch_map(&mapK);
    tma_prefetch_map(&mapV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Items are drawn from a work counter in the workspace when there is one
  // (split caches: SMs that run faster take more items), else round-robin;
  // the producer publishes each item in a small queue that the MMA issuer and
  // the row warps read in the same order (-1: no more).  n: entries read.
  auto read_item = [&](uint32_t& n, bool whole_warp) -> int {
    const uint32_t q = n % kItemQueue, ph = (n / kItemQueue) & 1u;
    const bool ok = whole_warp ? warp_wait(&bars->item_full[q], ph, a.ctl, abort)
                               : mbar_wait(&bars->item_full[q], ph, a.ctl, abort);
    if (!ok) return -1;
    const int v = bars->item[q];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&bars->item_empty[q]);
    ++n;
    return v;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t pos = 0;
      bool ok = true;
      uint32_t pn = 0;  // queue entries published
      int next_static = blockIdx.x;
      while (ok) {
        const uint32_t q = pn % kItemQueue;
        if (pn >= uint32_t(kItemQueue) &&
            !mbar_wait(&bars->item_empty[q], ((pn / kItemQueue) & 1u) ^ 1u, a.ctl, abort))
          break;
        Item it;
        int v;
        while (true) {
          if (a.item_ctr != nullptr) {
            v = int(atomicAdd(a.item_ctr, 1u));
          } else {
            v = next_static;
            next_static += gridDim.x;
          }
          if (v >= nvirt) break;
          const int st_item = item_info(v, a, it);
          if (st_item == 1) break;
          if (st_item < 0) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
        }
        if (v >= nvirt) v = -1;
        bars->item[q] = v;
        mbar_arrive(&bars->item_full[q]);
        ++pn;
        if (v < 0) break;
        const int plane = it.b * a.hkv + it.kvh;
        const int nb = (it.s_end - it.s_beg + kBK - 1) / kBK;
        for (int blk = 0; blk < nb; ++blk, ++pos) {
          const uint32_t st = pos % kStages;
          if (!mbar_wait(&bars->empty[st], ((pos / kStages) & 1u) ^ 1u, a.ctl, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
          uint8_t* dst = smem + kOffStage + st * kStageBytes;
          int row = it.s_beg + blk * kBK, pl = plane;
          if (a.pg.table != nullptr) {  // paged: blocks never straddle a page
            const int lp = row / a.pg.page;
            const int phys = __ldg(a.pg.table + long(it.b) * a.pg.stride + lp);
            if (phys < 0 || phys >= a.pg.num_pages) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
            row -= lp * a.pg.page;
            pl = phys * a.hkv + it.kvh;  // out of range reads as zeros
          }
          for (int i = 0; i < 3; ++i)
            tma_load_3d(dst + i * kBox, &mapK, &bars->full[st], 64 * i, row, pl);
          for (int i = 0; i < 2; ++i)
            tma_load_3d(dst + (3 + i) * kBox, &mapV, &bars->full[st], 64 * i, row, pl);
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      for (uint32_t s = 0; s < uint32_t(kStages); ++s) {
        const uint32_t fills = pos > s ? (pos - s + kStages - 1) / kStages : 0;
        if (fills) mbar_wait_drain(&bars->full[s], (fills - 1) & 1u, a.ctl);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_rot = make_idesc_f16(128, kBK, 0, 0);   // dims 0..63
      constexpr uint32_t idesc_s = make_idesc_bf16(128, kBK, 0, 0);    // dims 64..191
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, 0, 1);
      const uint32_t sbase = smem_u32(smem);
      uint32_t qc = 0, items = 0;
      uint32_t qk = 0, pv = 0;  // QK / PV products issued so far (global block counters)
      bool ok = true;
      auto issue_qk = [&](uint32_t qb, uint32_t blk_global) -> bool {
        const uint32_t st = blk_global % kStages;
        if (!mbar_wait(&bars->full[st], (blk_global / kStages) & 1u, a.ctl, abort)) return false;
        tc_fence_after();
        const uint32_t kbase = sbase + kOffStage + st * kStageBytes;
        const uint32_t d = tmem + s_col(blk_global & 1u);
        const uint64_t kdesc = make_sdesc_sw128(kbase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk)  // A = Q from TMEM (8 columns per k-step)
          umma_ts(d, tmem + q_col(qb) + kk * 8,
                  kdesc + uint64_t(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                  kk < 4 ? idesc_rot : idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[blk_global & 1u]);
        return true;
      };
      auto issue_pv = [&](uint32_t blk_global, bool first, bool last) -> bool {
        if (!mbar_wait(&bars->p_full[blk_global & 1u], (blk_global >> 1) & 1u, a.ctl, abort))
          return false;
        if (first && items > 0 && !mbar_wait(&bars->o_free, (items - 1) & 1u, a.ctl, abort))
          return false;
        tc_fence_after();
        const uint32_t st = blk_global % kStages;
        const uint32_t vbase = sbase + kOffStage + st * kStageBytes + 3 * kBox;
        const uint32_t p = tmem + s_col(blk_global & 1u);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_ts(tmem + kOCol, p + kk * 8, make_sdesc_sw128(vbase + kk * 2048, kBox, 1024),
                  idesc_o, (!first || kk > 0) ? 1u : 0u);
        umma_commit(&bars->pv_done);
        if (last) umma_commit(&bars->o_done);  // the item's O is complete
        // (the stage is released by a softmax thread once S of block
        // blk_global + 2 is done: that QK^T was issued after this PV)
        return true;
      };
      uint32_t rn = 0;
      while (ok) {
        const int v = read_item(rn, false);
        if (v < 0) break;
        Item it;
        item_info(v, a, it);
        const uint32_t qb = qc & 1u;
        if (!mbar_wait(&bars->q_ready[qb], (qc >> 1) & 1u, a.ctl, abort)) break;
        ++qc;
        const int nb = (it.s_end - it.s_beg + kBK - 1) / kBK;
        const uint32_t b0 = qk;  // global index of this item's block 0
        // QK_0, QK_1, PV_0, QK_2, PV_1, ...; once the item's last QK is
        // issued its Q buffer may be refilled
        if (!issue_qk(qb, qk)) break;
        ++qk;
        if (nb == 1) umma_commit(&bars->q_empty[qb]);
        for (int j = 0; j < nb && ok; ++j) {
          if (j + 1 < nb) {
            if (!issue_qk(qb, qk)) { ok = false; break; }
            ++qk;
            if (j + 2 == nb) umma_commit(&bars->q_empty[qb]);
          }
          if (!issue_pv(b0 + j, j == 0, j + 1 == nb)) { ok = false; break; }
          ++pv;
        }
        ++items;
      }
      // every MMA issued must be complete before TMEM is released
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;            // tile row
    const bool active = quad * 32 < rows;      // warp has at least one real row
    const bool real = r < rows;
    const int hh = r % G;                      // = lane % G
    const int t = real ? r / G : 0;
    const uint32_t lane_addr = uint32_t(quad * 32) << 16;
    uint32_t qc = 0, blk = 0, items = 0;
    // the previous item's row, finished after the next item's Q is rotated
    bool have_prev = false;
    float pm = 0.f, pl = 0.f;
    long porow = 0;
    int pb = 0, ph = 0, psplit = 0, pnsplit = 1;
    bool ok = true;

    auto epilogue = [&]() -> bool {
      // the item's last PV (items: items finished, the previous one included)
      if (!warp_wait(&bars->o_done, (items - 1) & 1u, a.ctl, abort)) return false;
      tc_fence_after();
      if (active) {
        const uint32_t t_o = tmem + lane_addr + kOCol;
        float sc, lse_v = 0.f;
        if (pnsplit == 1) {  // add the sink and finish the row
          const float sl2 = __ldg(a.sink + ph) * kLog2e;
          const float mt_ = fmaxf(pm, sl2);
          const float msub = mt_ == -INFINITY ? 0.f : mt_;
          const float fo = fast_exp2(pm - msub);
          const float sw = fast_exp2(sl2 - msub);
          sc = fo / (pl * fo + sw);
          lse_v = (msub + log2f(pl * fo + sw)) * kLn2;
        } else {
          sc = pl > 0.f ? 1.f / pl : 0.f;
          lse_v = pl > 0.f ? pm + log2f(pl) : -INFINITY;
        }
        const long prow = ((long(pb) * a.hq + ph) * T + t) * a.nsplit + psplit;
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t v[32];
          tmem_ld32_nowait(t_o + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) tmem_reg_fence(v[e]);
          if (real) {
            if (pnsplit == 1) {
              uint4* op = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + porow * 256 + c * 2);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                op[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]) * sc, __uint_as_float(v[8 * e + 1]) * sc),
                                   pack_bf16x2(__uint_as_float(v[8 * e + 2]) * sc, __uint_as_float(v[8 * e + 3]) * sc),
                                   pack_bf16x2(__uint_as_float(v[8 * e + 4]) * sc, __uint_as_float(v[8 * e + 5]) * sc),
                                   pack_bf16x2(__uint_as_float(v[8 * e + 6]) * sc, __uint_as_float(v[8 * e + 7]) * sc));
            } else {
              float4* pp = reinterpret_cast<float4*>(a.part_o + prow * kDv + c);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                pp[e] = make_float4(__uint_as_float(v[4 * e]) * sc, __uint_as_float(v[4 * e + 1]) * sc,
                                    __uint_as_float(v[4 * e + 2]) * sc, __uint_as_float(v[4 * e + 3]) * sc);
            }
          }
        }
        if (real) {
          if (pnsplit == 1) {
            if (a.lse) a.lse[porow] = lse_v;
          } else {
            a.part_lse[prow] = lse_v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      return true;
    };

    uint32_t rn = 0;
    while (true) {
      const int v = read_item(rn, true);
      if (v < 0) {
        ok = ok && !*abort;
        break;
      }
      Item it;
      item_info(v, a, it);
      // ---- Q: this row from global memory, RoPE on dims 0..63 in registers
      // (pairs (i, i + 32); the G lanes holding one token's heads each
      // evaluate 32/G of the 32 angles and exchange them by shuffles), into
      // TMEM Q buffer qb once the item that used it last has issued its
      // final QK^T
      const uint32_t qb = qc & 1u;
      if (!warp_wait(&bars->q_empty[qb], ((qc >> 1) & 1u) ^ 1u, a.ctl, abort)) { ok = false; break; }
      ++qc;
      const int p = it.L - T + t;  // this row's query position
      if (active) {
        float2 cs_own[32 / G];
#pragma unroll
        for (int k2 = 0; k2 < 32 / G; ++k2)
          cs_own[k2] = rope_cos_sin(p, a.freqs.hi[hh + G * k2], a.freqs.lo[hh + G * k2]);
        uint32_t qw[96];
        const uint4* qsrc = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(a.q) +
            ((long(it.b) * T + t) * a.hq + it.kvh * G + hh) * kDqk);
#pragma unroll
        for (int c = 0; c < 24; ++c) {
          const uint4 v = real ? __ldg(qsrc + c) : make_uint4(0u, 0u, 0u, 0u);
          qw[4 * c] = v.x;
          qw[4 * c + 1] = v.y;
          qw[4 * c + 2] = v.z;
          qw[4 * c + 3] = v.w;
        }
        uint32_t big = 0u;  // |rotated| of every pair, as fp16 (inf once out of range)
#pragma unroll
        for (int w = 0; w < 16; ++w) {  // word w holds dims 2w, 2w+1; word w + 16 dims + 32
          const int i = 2 * w;
          const float2 xv = unpack_bf16x2(qw[w]);
          const float2 yv = unpack_bf16x2(qw[w + 16]);
          const float2 c0 = shared_cos_sin<G>(cs_own, i, lane);
          const float2 c1 = shared_cos_sin<G>(cs_own, i + 1, lane);
          const float a0 = xv.x * c0.x - yv.x * c0.y, a1 = xv.y * c1.x - yv.y * c1.y;
          const float b0 = yv.x * c0.x + xv.x * c0.y, b1 = yv.y * c1.x + xv.y * c1.y;
          qw[w] = pack_f16x2(a0, a1);  // rotated dims are fp16 operands
          qw[w + 16] = pack_f16x2(b0, b1);
          big = f16x2_absmax3(big, qw[w], qw[w + 16]);
        }
        if (real && f16x2_any_inf(big)) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
        const uint32_t t_q = tmem + lane_addr + q_col(qb);
        tmem_st32(t_q, qw);
        tmem_st32(t_q + 32, qw + 32);
        tmem_st32(t_q + 64, qw + 64);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars->q_ready[qb]);
      if (have_prev && !epilogue()) { ok = false; break; }
      float m = -INFINITY, l = 0.f;
      const int nb = (it.s_end - it.s_beg + kBK - 1) / kBK;
      for (int j = 0; j < nb; ++j, ++blk) {
        const uint32_t sb = blk & 1u;
        if (!warp_wait(&bars->s_full[sb], (blk >> 1) & 1u, a.ctl, abort)) { ok = false; break; }
        // QK^T of block blk was issued after PV of block blk - 2 (within an
        // item QK_{j} follows PV_{j-2}; an item's first QK^T follows the last
        // PV of the item before), so that block's K / V stage is free now
        if (blk >= 2 && quad == 0 && lane == 0) mbar_arrive(&bars->empty[(blk - 2) % kStages]);
        tc_fence_after();
        const int sbase_slot = it.s_beg + j * kBK;
        const int valid_rows = it.s_end - sbase_slot;
        if (valid_rows < kBK) {
          // Slots past the item's end were loaded from cache memory the item
          // does not own (a linear cache's unwritten tail); their weights are
          // 0, but 0 * NaN is not, so zero those V rows before PV reads them.
          uint8_t* vrow = smem + kOffStage + (blk % kStages) * kStageBytes + 3 * kBox;
          for (int e = threadIdx.x - 64; e < (kBK - valid_rows) * 16; e += 128) {
            const int rr = valid_rows + (e >> 4), c16 = e & 15;
            *reinterpret_cast<uint4*>(vrow + (c16 >> 3) * kBox + rr * 128 + (c16 & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        if (active) {
          const uint32_t t_s = tmem + lane_addr + s_col(sb);
          uint32_t s[kBK];
          ld_row<kBK>(t_s, s);
          // visibility of slot sl for this row
          const bool full = !a.is_ring && a.window == 0 &&
                            sbase_slot + kBK <= min(it.s_end, it.L - T + 1);
          if (!full) {
#pragma unroll
            for (int c = 0; c < kBK; ++c) {
              const int sl = sbase_slot + c;
              const int kp = sl + it.ring_off + (sl < it.ring_r ? a.cap : 0);
              const bool vis = real && sl < it.s_end && kp >= 0 && kp <= p &&
                               (a.window == 0 || p - kp < a.window);
              if (!vis) s[c] = __float_as_uint(-INFINITY);
            }
          }
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBK; c += 2)
            mx = fmax3f(mx, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
          const float m_new = fmaxf(m, mx * a.scale_log2);
          const bool resc = m_new > m + kRescaleThreshold;
          float alpha = 1.f;
          if (resc) {
            alpha = fast_exp2(m - m_new);  // 0 when m was -inf
            m = m_new;
            l *= alpha;
          }
          const float msub = (m == -INFINITY) ? 0.f : m;
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
          const uint64_t nm2 = f2_pack(-msub, -msub);
          uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kBK; c += 16) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 x = f2_unpack(f2_fma(
                  f2_pack(__uint_as_float(s[c + e]), __uint_as_float(s[c + e + 1])), sc2, nm2));
              const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
              pk[e >> 1] = pack_bf16x2(p0, p1);
              acc = f2_add(acc, f2_pack(p0, p1));
            }
            tmem_st8(t_s + (c >> 1), pk);  // P (bf16 pairs) over consumed S columns
          }
          const float2 sum = f2_unpack(acc);
          l += sum.x + sum.y;
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
            // O holds the earlier blocks scaled by 2^-m_old: rescale it once
            // the PV of the previous block has landed
            if (!warp_wait(&bars->pv_done, (blk - 1) & 1u, a.ctl, abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t_o = tmem + lane_addr + kOCol;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
              uint32_t v[32];
              tmem_ld32_nowait(t_o + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                tmem_reg_fence(v[e]);
                v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              }
              tmem_st32(t_o + c, v);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      have_prev = true;
      pm = m;
      pl = l;
      pb = it.b;
      ph = it.kvh * G + hh;
      porow = (long(it.b) * T + t) * a.hq + ph;
      psplit = it.split;
      pnsplit = it.nsplit;
      ++items;
    }
    if (ok && have_prev) epilogue();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One warp per output row (b, t, h) of a sequence cut into several chunks:
// combine the chunks' (O_i, lse_i) and the sink:
// lse = log2(sum_i 2^lse_i + 2^s), O = sum_i 2^(lse_i - lse) O_i.
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const long row = long(blockIdx.x) * 8 + (threadIdx.x >> 5);  // (b, t, h)
  const int T = a.T;
  if (row >= long(a.B) * T * a.hq) return;
  const int h = int(row % a.hq);
  const int t = int((row / a.hq) % T);
  const int b = int(row / (long(a.hq) * T));
  const int L = __ldg(a.seqlens + b);
  if (!length_ok(L, a)) return;  // reported by the decode kernel
  int lo, hi;
  slot_range(L, a, lo, hi);
  const int nsplit = (hi - lo + a.chunk - 1) / a.chunk;
  if (nsplit <= 1) return;  // a one-chunk sequence was finished by the decode kernel
  const long prow0 = ((long(b) * a.hq + h) * T + t) * a.nsplit;
  const float sl2 = __ldg(a.sink + h) * kLog2e;
  float M = sl2;
  for (int i = 0; i < nsplit; ++i) M = fmaxf(M, __ldg(a.part_lse + prow0 + i));
  const float msub = M == -INFINITY ? 0.f : M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = fast_exp2(sl2 - msub);
  for (int i = 0; i < nsplit; ++i) {
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

// ---------------------------------------------------------------------------
// Rings of at most 144 slots with at most 32 query rows (the window layer at
// W = 128, T <= 4, G <= 8) on the tensor cores.  Persistent: one CTA per SM
// walks the items (sequence, KV head) v = blockIdx.x + i * gridDim.x.  Two
// workers take alternate items, each with its own shared-memory buffer (Q,
// the ring's K and V), its own half of TMEM and its own TMEM lane quadrant,
// so that one item's loads, MMAs and softmax overlap the other's.
//   warp 2   TMEM allocator; lane 0 loads item i into buffer i % 2: Q (3
//            boxes of [G*T rows][64 dims]), K (3 boxes of [cap slots][64
//            dims]) and V (2 boxes), each on its own barrier, the Q/K loads
//            of an item ahead of the V loads of the one before (the first
//            two items' Q/K before the rest of the setup).  Q/K and V of a
//            buffer are refilled as soon as the MMAs that read them are done.
//   worker w = warps w and w + 4 (TMEM lane quadrant w, one lane per query
//            row; the two warps split each row's work in halves): RoPE of the
//            Q rows in shared memory; S = Q K^T (M=128, N = cap rounded up to
//            16, K=192); the masked softmax over the whole ring in one pass (a
//            row sees a cyclic interval of slots); P to TMEM; O = P V; the
//            epilogue with the sink.  Lane 0 of warp w issues the MMAs.
// Worker w's query rows are rows 32w.. of its MMA tile (the lanes its warps
// read): its A descriptor starts 32w rows before the Q tile.  Other tile rows
// read whatever shared memory lies there: their S, P and O rows are never
// used.  TMEM of worker w: S at 256w + 0..143, O at 256w + 128..255 over S's
// upper columns (dead once the softmax read them).
// ---------------------------------------------------------------------------
constexpr int kRingTcMaxCap = 144;
constexpr int kRingTcH0 = 80, kRingTcH1 = 64;    // S columns of the two halves
constexpr int kRingTcQBox = 32 * 128;            // [32 rows][64 dims]
constexpr int kRingTcKBox = kRingTcMaxCap * 128; // [144 slots][64 dims]
constexpr int kRingTcOffK = 3 * kRingTcQBox;
constexpr int kRingTcOffV = kRingTcOffK + 3 * kRingTcKBox;
constexpr int kRingTcBuf = kRingTcOffV + 2 * kRingTcKBox;
constexpr int kRingTcOffCs = 2 * kRingTcBuf;     // (cos, sin) of the item's tokens, per worker
constexpr int kRingTcCsRow = 32 * 8 + 16;        // one token's 32 pairs (+16: no bank clash)
constexpr int kRingTcOffRed = kRingTcOffCs + 2 * 4 * kRingTcCsRow;  // [worker][half][max|sum][32]
// the T <= 4 new tokens' K (3 boxes of [T rows][64 dims]) and V (2 boxes) of a
// worker's item, loaded with its Q (the fused append reads them from here)
constexpr int kRingTcNewBox = 1024;
constexpr int kRingTcNewBytes = 5 * kRingTcNewBox;  // per worker
constexpr int kRingTcOffNew = (kRingTcOffRed + 2 * 2 * 2 * 32 * 4 + 1023) / 1024 * 1024;
constexpr int kRingTcOffBar = kRingTcOffNew + 2 * kRingTcNewBytes;
constexpr int kRingTcSmem = kRingTcOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr int kRingTcThreads = 192;
static_assert(kRingTcBuf % 1024 == 0 && kRingTcKBox % 1024 == 0, "swizzle atoms");
static_assert(kRingTcSmem <= 232448, "shared memory");
static_assert(kRingTcH0 + kRingTcH1 == kRingTcMaxCap, "halves cover the ring");
__host__ __device__ constexpr int ring_tc_rows(int cap) { return (cap + 15) & ~15; }

struct RingTcBars {
  // a buffer's Q/K may be refilled once its S product is done and its V
  // once its PV product is: the producer reads both from the phases of
  // s_full and pv_done (the next phase needs the very load being waited for)
  uint64_t q_full[2], k_full[2], v_full[2], s_full[2], pv_done[2];
  uint64_t drain[2], pair[2];  // the two warps of a worker meet here (one arrival per warp)
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(RingTcBars) <= 256, "barrier block");

// Bits [lo, hi) of the 32-bit word holding columns 32k..32k+31.
__device__ __forceinline__ uint32_t ring_bits(int k, int lo, int hi) {
  const int a = min(max(lo - 32 * k, 0), 32), b = min(max(hi - 32 * k, 0), 32);
  const uint32_t below_b = b >= 32 ? 0xffffffffu : (1u << b) - 1u;
  const uint32_t below_a = a >= 32 ? 0xffffffffu : (1u << a) - 1u;
  return below_b & ~below_a;
}

// Both warps of a worker: a bounded rendezvous on an mbarrier of count 2.
__device__ __forceinline__ bool pair_sync(uint64_t* bar, uint32_t& ph, int lane,
                                          const DecodeArgs& a, volatile int* abort) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = warp_wait(bar, ph, a.ctl, abort);
  ph ^= 1u;
  return ok;
}

// One half of a row's softmax: N S columns C0.. from TMEM; invisible columns
// (clear bit in vis[]) to -inf; returns their max (unscaled).
template <int N, int C0>
__device__ __forceinline__ float ring_load_max(uint32_t t_s, uint32_t (&s)[N],
                                               const uint32_t (&vis)[5]) {
#pragma unroll
  for (int c = 0; c + 32 <= N; c += 32) tmem_ld32_nowait(t_s + C0 + c, s + c);
  if constexpr (N % 32 == 16) tmem_ld16_nowait(t_s + C0 + N - 16, s + N - 16);
  tmem_ld_wait();
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int e = 0; e < N; ++e) {
    tmem_reg_fence(s[e]);
    const int c = C0 + e;
    if (!(vis[c >> 5] & (1u << (c & 31)))) s[e] = __float_as_uint(-INFINITY);
  }
#pragma unroll
  for (int e = 0; e < N; e += 8) {
    mx[(e >> 3) & 3] = fmax3f(mx[(e >> 3) & 3], __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
    mx[(e >> 3) & 3] = fmax3f(mx[(e >> 3) & 3], __uint_as_float(s[e + 2]), __uint_as_float(s[e + 3]));
    mx[(e >> 3) & 3] = fmax3f(mx[(e >> 3) & 3], __uint_as_float(s[e + 4]), __uint_as_float(s[e + 5]));
    mx[(e >> 3) & 3] = fmax3f(mx[(e >> 3) & 3], __uint_as_float(s[e + 6]), __uint_as_float(s[e + 7]));
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// exp2(s * scale - m) of N columns as bf16 pairs into TMEM at taddr (masked
// columns hold -inf and give 0); returns the fp32 sum of the weights.
template <int N>
__device__ __forceinline__ float ring_exp_store(const uint32_t (&s)[N], uint32_t taddr,
                                                float scale, float m) {
  const uint64_t sc2 = f2_pack(scale, scale);
  const uint64_t nm2 = f2_pack(-m, -m);
  uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int c = 0; c < N; c += 16) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 x = f2_unpack(
          f2_fma(f2_pack(__uint_as_float(s[c + e]), __uint_as_float(s[c + e + 1])), sc2, nm2));
      const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
      pk[e >> 1] = pack_bf16x2(p0, p1);
      acc[(e >> 1) & 1] = f2_add(acc[(e >> 1) & 1], f2_pack(p0, p1));
    }
    tmem_st8(taddr + (c >> 1), pk);
  }
  const float2 s0 = f2_unpack(acc[0]), s1 = f2_unpack(acc[1]);
  return (s0.x + s0.y) + (s1.x + s1.y);
}

template <int G>
__global__ void __launch_bounds__(kRingTcThreads, 1)
    decode_ring_tc_kernel(const __grid_constant__ CUtensorMap mapQ,
                          const __grid_constant__ CUtensorMap mapK,
                          const __grid_constant__ CUtensorMap mapV,
                          const __grid_constant__ CUtensorMap mapKN,
                          const __grid_constant__ CUtensorMap mapVN, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, rows = G * T;
  const int nitems = a.B * a.hkv;
  const int RR = ring_tc_rows(a.cap);
  RingTcBars* bars = reinterpret_cast<RingTcBars*>(smem + kRingTcOffBar);
  volatile int* abort = &bars->abort;
  // Q (3 boxes of [G*T rows][64 dims]) -- and with a fused append the new
  // tokens' K and V (5 boxes of [T rows][64 dims]) -- on q_full, K (3 boxes
  // of [cap slots][64 dims]) on k_full of buffer j = i % 2
  const bool fused = a.k_new != nullptr;
  auto load_qk = [&](int i) {
    const int v = blockIdx.x + i * gridDim.x;
    const int b = v / a.hkv, kvh = v - b * a.hkv, j = i & 1;
    uint8_t* buf = smem + j * kRingTcBuf;
    mbar_arrive_expect_tx(&bars->q_full[j], uint32_t((3 * rows + (fused ? 5 * T : 0)) * 128));
    for (int k = 0; k < 3; ++k)
      tma_load_3d(buf + k * kRingTcQBox, &mapQ, &bars->q_full[j], 64 * k, kvh * G, b * T);
    if (fused) {
      uint8_t* nb = smem + kRingTcOffNew + j * kRingTcNewBytes;
      for (int k = 0; k < 3; ++k)
        tma_load_3d(nb + k * kRingTcNewBox, &mapKN, &bars->q_full[j], 64 * k, kvh, b * T);
      for (int k = 0; k < 2; ++k)
        tma_load_3d(nb + (3 + k) * kRingTcNewBox, &mapVN, &bars->q_full[j], 64 * k, kvh, b * T);
    }
    mbar_arrive_expect_tx(&bars->k_full[j], uint32_t(3 * a.cap * 128));
    for (int k = 0; k < 3; ++k)
      tma_load_3d(buf + kRingTcOffK + k * kRingTcKBox, &mapK, &bars->k_full[j], 64 * k, 0, v);
  };
  const int nmine = (nitems - 1 - int(blockIdx.x)) / int(gridDim.x) + 1;  // items of this CTA
  if (threadIdx.x == 64) {
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bars->q_full[j], 1);
      mbar_init(&bars->k_full[j], 1);
      mbar_init(&bars->v_full[j], 1);
      mbar_init(&bars->s_full[j], 1);
      mbar_init(&bars->pv_done[j], 1);
      mbar_init(&bars->drain[j], 1);
      mbar_init(&bars->pair[j], 2);
    }
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_map(&mapQ);
    tma_prefetch_map(&mapK);
    tma_prefetch_map(&mapV);
    if (fused) {
      tma_prefetch_map(&mapKN);
      tma_prefetch_map(&mapVN);
    }
  }
  if (warp == 2) {
    __syncwarp();
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  // V rows past cap are read by the last PV k-step and never loaded: zero
  // them once in both buffers
  for (int e = threadIdx.x; e < 2 * (kRingTcMaxCap - a.cap) * 16; e += kRingTcThreads) {
    const int j = e & 1, rr = a.cap + (e >> 5), c16 = (e >> 1) & 15;
    *reinterpret_cast<uint4*>(smem + j * kRingTcBuf + kRingTcOffV + (c16 >> 3) * kRingTcKBox +
                              rr * 128 + (c16 & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Everything above touches only this CTA's shared memory and TMEM, so under
  // a programmatic launch it overlaps the previous kernel's tail; from here on
  // the previous kernel's writes (the queries, new tokens, the caches) are
  // visible.  The next kernel may then start its own setup.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the first two items' Q/K go out first
      for (int i = 0; i < 2 && i < nmine; ++i) load_qk(i);
      int qk_uses[2] = {nmine > 0 ? 1 : 0, nmine > 1 ? 1 : 0}, v_uses[2] = {0, 0};
      // Q/K of item iq once its buffer's Q/K are free; V of item iv once that
      // item's K has landed (the softmax needs it first) and its buffer's V
      // is free.  Q/K run at most two items ahead of V, so that the
      // full-barrier phase V tests is still the current one.
      int iq = nmine < 2 ? nmine : 2, iv = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (iv < nmine) {
        bool prog = false;
        if (iq < nmine && iq < iv + 2) {
          const int j = iq & 1, use = iq >> 1;
          if (mbar_test_wait(&bars->s_full[j], (use - 1) & 1u)) {
            load_qk(iq);
            qk_uses[j] = use + 1;
            ++iq;
            prog = true;
          }
        }
        if (iv < iq) {
          const int j = iv & 1, use = iv >> 1;
          if (mbar_test_wait(&bars->k_full[j], use & 1u) &&
              (use == 0 || mbar_test_wait(&bars->pv_done[j], (use - 1) & 1u))) {
            const int v = blockIdx.x + iv * gridDim.x;
            uint8_t* buf = smem + j * kRingTcBuf;
            mbar_arrive_expect_tx(&bars->v_full[j], uint32_t(2 * a.cap * 128));
            for (int k = 0; k < 2; ++k)
              tma_load_3d(buf + kRingTcOffV + k * kRingTcKBox, &mapV, &bars->v_full[j], 64 * k, 0,
                          v);
            v_uses[j] = use + 1;
            ++iv;
            prog = true;
          }
        }
        if (prog) {
          t_last = globaltimer_ns();
          spins = 0;
        } else if (((++spins) & 15u) == 0u) {
          if (*abort) break;
          if (globaltimer_ns() - t_last > a.ctl.wait_limit_ns) {
            record_status(a.ctl, HATTN_ERR_TIMEOUT);
            *abort = 1;
            break;
          }
        }
      }
      // never leave with copies in flight
      for (int j = 0; j < 2; ++j) {
        if (qk_uses[j]) {
          mbar_wait_drain(&bars->q_full[j], (qk_uses[j] - 1) & 1u, a.ctl);
          mbar_wait_drain(&bars->k_full[j], (qk_uses[j] - 1) & 1u, a.ctl);
        }
        if (v_uses[j]) mbar_wait_drain(&bars->v_full[j], (v_uses[j] - 1) & 1u, a.ctl);
      }
    }
  } else if (warp != 3) {
    // ------------------------------------------------------------ workers
    const int w = warp & 3;          // worker = TMEM lane quadrant
    const int hf = warp >> 2;        // half of the row's work
    const bool issuer = hf == 0 && lane == 0;
    const int r = lane;
    const bool real = r < rows;
    const int t = real ? r / G : 0, hh = r % G;
    uint8_t* buf = smem + w * kRingTcBuf;
    uint8_t* cs_tab = smem + kRingTcOffCs + w * 4 * kRingTcCsRow;
    float* red = reinterpret_cast<float*>(smem + kRingTcOffRed) + w * 128;  // [half][max|sum][32]
    const uint32_t sbuf = smem_u32(buf);
    const uint32_t t_s = tmem + (uint32_t(32 * w) << 16) + 256u * w;
    const uint32_t d_s = tmem + 256u * w;  // MMA accumulator (lane field 0)
    uint32_t pph = 0;                      // phase of this worker's pair barrier
    bool issued = false;
    uint32_t nv = 0;  // items this worker took (computed or skipped): phases of s_full, pv_done
    // the sequence length and this row's sink logit of the worker's next
    // item are loaded one item ahead: their latency hides behind the
    // current item instead of stalling its start and its epilogue
    auto item_len = [&](int i) {
      const int v = blockIdx.x + i * gridDim.x;
      return v < nitems ? __ldg(a.seqlens + v / a.hkv) : 0;
    };
    auto item_sink = [&](int i) {
      const int v = blockIdx.x + i * gridDim.x;
      return v < nitems ? __ldg(a.sink + (v % a.hkv) * G + hh) : 0.f;
    };
    int L_next = item_len(w);
    float sink_next = item_sink(w);
    for (int i = w;; i += 2) {
      const int v = blockIdx.x + i * gridDim.x;
      if (v >= nitems) break;
      const uint32_t ph = uint32_t(i >> 1) & 1u;
      const int b = v / a.hkv, kvh = v - b * a.hkv;
      const int L = L_next;
      const float sink_row = sink_next;
      L_next = item_len(i + 2);
      sink_next = item_sink(i + 2);
      const bool valid = length_ok(L, a);
      // fused append: this lane's share of the T new tokens' K and V, which
      // land with Q (read into registers once Q has, before the S product
      // lets the producer refill the buffer).  K pairs of chunks (c, c + 4),
      // c in this half's two rotated chunks: lanes < 2T; the other 16 K
      // chunks and the 16 V chunks of each token: task e = 32 hf + lane < 16 T.
      const bool fuse = a.k_new != nullptr && valid;
      const int e_task = 32 * hf + lane;
      const int kp_t = lane >> 1, kp_c = 2 * hf + (lane & 1);
      const int pl_t = e_task >> 4, pl_c = 8 + (e_task & 15), v_c = e_task & 15;
      uint4 kp_x = make_uint4(0u, 0u, 0u, 0u), kp_y = kp_x, kpl = kp_x, vpl = kp_x;
      if (valid) {
        // (cos, sin) of the 16 frequencies this half rotates, at each of the
        // T query positions
        const int f = 16 * hf + (lane & 15);
        for (int tt = lane >> 4; tt < T; tt += 2)
          *reinterpret_cast<float2*>(cs_tab + tt * kRingTcCsRow + f * 8) =
              rope_cos_sin(L - T + tt, a.freqs.hi[f], a.freqs.lo[f]);
      }
      __syncwarp();
      if (!warp_wait(&bars->q_full[w], ph, a.ctl, abort)) break;
      if (fuse) {
        // rows of 128 bytes, 16-byte chunks swizzled by row (boxes 1 KB-aligned)
        const uint8_t* nb = smem + kRingTcOffNew + w * kRingTcNewBytes;
        if (lane < 2 * T) {
          kp_x = *reinterpret_cast<const uint4*>(nb + kp_t * 128 + ((kp_c ^ kp_t) << 4));
          kp_y = *reinterpret_cast<const uint4*>(nb + kp_t * 128 + (((kp_c + 4) ^ kp_t) << 4));
        }
        if (e_task < 16 * T) {
          kpl = *reinterpret_cast<const uint4*>(nb + (pl_c >> 3) * kRingTcNewBox + pl_t * 128 +
                                                (((pl_c & 7) ^ pl_t) << 4));
          vpl = *reinterpret_cast<const uint4*>(nb + (3 + (v_c >> 3)) * kRingTcNewBox +
                                                pl_t * 128 + (((v_c & 7) ^ pl_t) << 4));
        }
      }
      const int p = L - T + t;  // this row's query position
      if (valid) {
        // RoPE of this row's dim pairs (f, f + 32), f in this half's 16:
        // chunks c and c + 4 of box 0 (128-byte rows, 16-byte chunks
        // swizzled by row % 8)
        const uint8_t* cs_row = cs_tab + t * kRingTcCsRow;
        uint8_t* qrow = buf + r * 128;
        uint32_t big = 0u;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint4 cx = *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4));
          uint4 cy = *reinterpret_cast<uint4*>(qrow + (((c + 4) ^ (r & 7)) << 4));
          uint32_t* x = reinterpret_cast<uint32_t*>(&cx);
          uint32_t* y = reinterpret_cast<uint32_t*>(&cy);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 cs = *reinterpret_cast<const float4*>(cs_row + (8 * c + 2 * q) * 8);
            const float2 xv = unpack_bf16x2(x[q]);
            const float2 yv = unpack_bf16x2(y[q]);
            const float a0 = xv.x * cs.x - yv.x * cs.y, a1 = xv.y * cs.z - yv.y * cs.w;
            const float b0 = yv.x * cs.x + xv.x * cs.y, b1 = yv.y * cs.z + xv.y * cs.w;
            x[q] = pack_f16x2(a0, a1);  // rotated dims are fp16 operands
            y[q] = pack_f16x2(b0, b1);
            big = f16x2_absmax3(big, x[q], y[q]);
          }
          if (real) {
            *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4)) = cx;
            *reinterpret_cast<uint4*>(qrow + (((c + 4) ^ (r & 7)) << 4)) = cy;
          }
        }
        if (real && f16x2_any_inf(big)) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
        fence_proxy_async_smem();
      } else if (lane == 0 && hf == 0 && kvh == 0) {
        record_status(a.ctl, HATTN_ERR_INVALID_ARG);
      }
      // both halves' Q rows are written, K has landed, and their reads of
      // this TMEM half (the previous item's epilogue) are complete
      if (!warp_wait(&bars->k_full[w], ph, a.ctl, abort)) break;
      const long plane = long(b) * a.hkv + kvh;
      if (fuse) {
        // the new keys over their slots' stale rows: in the loaded ring
        // (after the load, before the MMA reads it) and in the cache
        uint8_t* ks = buf + kRingTcOffK;
        uint4* kc = static_cast<uint4*>(const_cast<void*>(a.k_cache));
        if (lane < 2 * T) {
          const int slot = (L - T + kp_t) % a.cap;
          const uint8_t* cs_row = cs_tab + kp_t * kRingTcCsRow;
          uint32_t* x = reinterpret_cast<uint32_t*>(&kp_x);
          uint32_t* y = reinterpret_cast<uint32_t*>(&kp_y);
          bool over = false;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 cs = *reinterpret_cast<const float4*>(cs_row + (8 * kp_c + 2 * q) * 8);
            const float2 xv = unpack_bf16x2(x[q]);
            const float2 yv = unpack_bf16x2(y[q]);
            const float a0 = xv.x * cs.x - yv.x * cs.y, a1 = xv.y * cs.z - yv.y * cs.w;
            const float b0 = yv.x * cs.x + xv.x * cs.y, b1 = yv.y * cs.z + xv.y * cs.w;
            over |= fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) > kF16Max;
            x[q] = pack_f16x2(a0, a1);  // rotated dims are stored as fp16
            y[q] = pack_f16x2(b0, b1);
          }
          if (over) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
          *reinterpret_cast<uint4*>(ks + slot * 128 + ((kp_c ^ (slot & 7)) << 4)) = kp_x;
          *reinterpret_cast<uint4*>(ks + slot * 128 + (((kp_c + 4) ^ (slot & 7)) << 4)) = kp_y;
          kc[(plane * a.cap + slot) * 24 + kp_c] = kp_x;
          kc[(plane * a.cap + slot) * 24 + kp_c + 4] = kp_y;
        }
        if (e_task < 16 * T) {
          const int slot = (L - T + pl_t) % a.cap;
          *reinterpret_cast<uint4*>(ks + (pl_c >> 3) * kRingTcKBox + slot * 128 +
                                    (((pl_c & 7) ^ (slot & 7)) << 4)) = kpl;
          kc[(plane * a.cap + slot) * 24 + pl_c] = kpl;
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      if (!pair_sync(&bars->pair[w], pph, lane, a, abort)) break;
      if (!valid) {
        // nothing to compute: hand the buffer back once V has landed too,
        // completing the phases of s_full and pv_done the products would have
        const bool ok = warp_wait(&bars->v_full[w], ph, a.ctl, abort);
        if (issuer) {
          mbar_arrive(&bars->s_full[w]);
          mbar_arrive(&bars->pv_done[w]);
        }
        ++nv;
        if (!ok) break;
        continue;
      }
      if (issuer) {
        tc_fence_after();
        const uint32_t idesc_rot = make_idesc_f16(128, RR, 0, 0);
        const uint32_t idesc_s = make_idesc_bf16(128, RR, 0, 0);
        const uint64_t qd = make_sdesc_sw128(sbuf - uint32_t(w * kRingTcQBox), 16, 1024);
        const uint64_t kd = make_sdesc_sw128(sbuf + kRingTcOffK, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk)
          umma_ss(d_s, qd + uint64_t(((kk >> 2) * kRingTcQBox + (kk & 3) * 32) >> 4),
                  kd + uint64_t(((kk >> 2) * kRingTcKBox + (kk & 3) * 32) >> 4),
                  kk < 4 ? idesc_rot : idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[w]);
      }
      issued = true;
      // visible positions [lo, p] sit in the cyclic slot interval starting at
      // lo mod cap (a ring holds the last cap >= W + T - 1 positions)
      const int lo = max(p - a.window + 1, 0);
      const int nvis = real ? p - lo + 1 : 0;
      const int s_lo = lo % a.cap;
      const int e1 = min(s_lo + nvis, a.cap), e2 = s_lo + nvis - a.cap;
      uint32_t vis[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) vis[k] = ring_bits(k, s_lo, e1) | ring_bits(k, 0, e2);
      const uint32_t phc = nv++ & 1u;
      if (!warp_wait(&bars->s_full[w], phc, a.ctl, abort)) break;
      tc_fence_after();
      float m, l_own;
      if (hf == 0) {
        uint32_t s[kRingTcH0];
        red[lane] = ring_load_max<kRingTcH0, 0>(t_s, s, vis);
        tc_fence_before();  // S reads done before the other half writes P
        if (!pair_sync(&bars->pair[w], pph, lane, a, abort)) break;
        tc_fence_after();
        m = fmaxf(red[lane], red[64 + lane]) * a.scale_log2;  // exact max over the ring
        l_own = ring_exp_store<kRingTcH0>(s, t_s, a.scale_log2, m == -INFINITY ? 0.f : m);
      } else {
        uint32_t s[kRingTcH1];
        red[64 + lane] = ring_load_max<kRingTcH1, kRingTcH0>(t_s, s, vis);
        tc_fence_before();  // S reads done before the other half writes P
        if (!pair_sync(&bars->pair[w], pph, lane, a, abort)) break;
        tc_fence_after();
        m = fmaxf(red[lane], red[64 + lane]) * a.scale_log2;
        l_own = ring_exp_store<kRingTcH1>(s, t_s + kRingTcH0 / 2, a.scale_log2,
                                          m == -INFINITY ? 0.f : m);
      }
      red[32 + 64 * hf + lane] = l_own;
      tmem_st_wait();
      if (!warp_wait(&bars->v_full[w], ph, a.ctl, abort)) break;
      if (fuse && e_task < 16 * T) {
        // the new values over their slots' stale rows, in the ring and the cache
        const int slot = (L - T + pl_t) % a.cap;
        *reinterpret_cast<uint4*>(buf + kRingTcOffV + (v_c >> 3) * kRingTcKBox + slot * 128 +
                                  (((v_c & 7) ^ (slot & 7)) << 4)) = vpl;
        static_cast<uint4*>(const_cast<void*>(a.v_cache))[(plane * a.cap + slot) * 16 + v_c] =
            vpl;
        fence_proxy_async_smem();
      }
      const int nslots = min(L, a.cap);  // slots written so far; the rest may hold anything
      if (nslots < a.cap) {
        uint8_t* vs = buf + kRingTcOffV;
        for (int e = 32 * hf + lane; e < (a.cap - nslots) * 16; e += 64) {
          const int rr = nslots + (e >> 4), c16 = e & 15;
          *reinterpret_cast<uint4*>(vs + (c16 >> 3) * kRingTcKBox + rr * 128 + (c16 & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      // both halves' P columns are in TMEM, V is complete
      tc_fence_before();
      if (!pair_sync(&bars->pair[w], pph, lane, a, abort)) break;
      if (issuer) {
        tc_fence_after();
        constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, 0, 1);
        const uint64_t vd = make_sdesc_sw128(sbuf + kRingTcOffV, kRingTcKBox, 1024);
        for (int kk = 0; kk < RR / 16; ++kk)
          umma_ts(d_s + 128, d_s + kk * 8, vd + uint64_t((kk * 2048) >> 4), idesc_o,
                  kk > 0 ? 1u : 0u);
        umma_commit(&bars->pv_done[w]);
      }
      const float l = red[32 + lane] + red[96 + lane];
      if (!warp_wait(&bars->pv_done[w], phc, a.ctl, abort)) break;
      tc_fence_after();
      // ---- epilogue: add the sink, finish this half of the row
      const int h = kvh * G + hh;
      const float sl2 = sink_row * kLog2e;
      const float mt_ = fmaxf(m, sl2);
      const float msub = mt_ == -INFINITY ? 0.f : mt_;
      const float fo = fast_exp2(m - msub);
      const float sw = fast_exp2(sl2 - msub);
      const float sc = fo / (l * fo + sw);
      const uint64_t sc2 = f2_pack(sc, sc);
      const long orow = (long(b) * T + t) * a.hq + h;
      uint4* op = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + orow * 256 + hf * 128);
      uint32_t o[64];
      tmem_ld32_nowait(t_s + 128 + hf * 64, o);
      tmem_ld32_nowait(t_s + 128 + hf * 64 + 32, o + 32);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 64; ++e) tmem_reg_fence(o[e]);
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float2 y = f2_unpack(
            f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), sc2));
        pk[e] = pack_bf16x2(y.x, y.y);
      }
      if (real) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          op[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        if (hf == 0 && a.lse) a.lse[orow] = (msub + log2f(l * fo + sw)) * kLn2;
      }
    }
    // every MMA this worker issued must be complete before TMEM is released
    tc_fence_before();
    __syncwarp();
    if (issuer && issued) {
      umma_commit(&bars->drain[w]);
      mbar_wait_drain(&bars->drain[w], 0, a.ctl);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int G>
cudaError_t launch_ring_tc(const DecodeArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        decode_ring_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingTcSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap mq, mk, mv, mkn, mvn;
  if (!make_map(&mq, a.q, long(a.B) * a.T, a.hq, kDqk, G, a.T) ||
      !make_map(&mk, a.k_cache, long(a.B) * a.hkv, a.cap, kDqk, a.cap, 1) ||
      !make_map(&mv, a.v_cache, long(a.B) * a.hkv, a.cap, kDv, a.cap, 1))
    return cudaErrorInvalidValue;
  // the new tokens' K / V [B, T, hkv, d]: boxes of one KV head's T rows
  if (a.k_new != nullptr) {
    if (!make_map(&mkn, a.k_new, long(a.B) * a.T, a.hkv, kDqk, 1, a.T) ||
        !make_map(&mvn, a.v_new, long(a.B) * a.T, a.hkv, kDv, 1, a.T))
      return cudaErrorInvalidValue;
  } else {
    mkn = mq;  // not read
    mvn = mq;
  }
  // as many CTAs as give each the same number of items (512 items over a
  // 148-SM part: 128 CTAs of 4, two per worker, rather than 148 CTAs of 3 or
  // 4, where the CTAs with 4 set the step's time)
  const long items = long(a.B) * a.hkv;
  const long per = (items + num_sms() - 1) / num_sms();
  const int grid = int((items + per - 1) / per);
  // programmatic dependent launch: the CTAs' setup overlaps the tail of the
  // kernel before them; every global read waits for it (grid_dep_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kRingTcThreads);
  cfg.dynamicSmemBytes = kRingTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_ring_tc_kernel<G>, mq, mk, mv, mkn, mvn, a);
}

cudaError_t launch_decode_kernel(const DecodeArgs& a, cudaStream_t s) {
  const int G = a.hq / a.hkv;
  auto kern = G == 1 ? decode_kernel<1> : G == 2 ? decode_kernel<2> : G == 4 ? decode_kernel<4>
              : G == 8 ? decode_kernel<8> : decode_kernel<16>;
  static bool attr_set[5] = {false, false, false, false, false};
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;
  if (!attr_set[gi]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[gi] = true;
  }
  CUtensorMap mq, mk, mv;
  const bool paged = a.pg.table != nullptr;
  const long planes = paged ? long(a.pg.num_pages) * a.hkv : long(a.B) * a.hkv;
  const int slots = paged ? a.pg.page : a.cap;
  if (!make_map(&mq, a.q, long(a.B) * a.T, a.hq, kDqk, G, a.T) ||
      !make_map(&mk, a.k_cache, planes, slots, kDqk, kBK, 1) ||
      !make_map(&mv, a.v_cache, planes, slots, kDv, kBK, 1))
    return cudaErrorInvalidValue;
  const long nvirt = long(a.nsplit) * a.B * a.hkv;
  const int grid = int(nvirt < num_sms() ? nvirt : num_sms());
  if (a.item_ctr != nullptr) {
    cudaError_t e = cudaMemsetAsync(a.item_ctr, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, a, int(nvirt));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.nsplit == 1) return e;
  const long nrows = long(a.B) * a.T * a.hq;
  decode_merge_kernel<<<dim3(unsigned((nrows + 7) / 8)), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(int max_seqlen_k, int T, int window, int is_ring, int cap, int* chunk) {
  int range;
  if (is_ring)
    range = max_seqlen_k < cap ? max_seqlen_k : cap;
  else if (window > 0)
    // 64-bit: a window near INT_MAX must not wrap around
    range = long(max_seqlen_k) < long(window) + T - 1 ? max_seqlen_k : window + T - 1;
  else
    range = max_seqlen_k;
  if (range <= kSingleChunkMax) {
    *chunk = range > 0 ? range : 1;
    return 1;
  }
  *chunk = range > 16384 ? kChunkLong : kChunkShort;
  return (range + *chunk - 1) / *chunk;
}

size_t decode_workspace_bytes(int B, int T, int hq, int nsplit) {
  if (nsplit <= 1) return 0;
  const size_t rows = size_t(B) * hq * T * nsplit;
  const size_t o_bytes = rows * kDv * sizeof(float);
  const size_t l_bytes = rows * sizeof(float);
  // partial O, partial lse, then the kernel's work counter
  return ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256 + 256;
}

cudaError_t launch_decode(const DecodeArgs& a_in, cudaStream_t s) {
  DecodeArgs a = a_in;
  const int G = a.hq / a.hkv;
  // (its per-worker tables and its share of the append assume T <= 4)
  const bool ring_tc = a.is_ring && a.cap <= kRingTcMaxCap && a.nsplit == 1 && a.T <= 4 &&
                       G * a.T <= 32 && (G == 1 || G == 2 || G == 4 || G == 8);
  if (a.k_new && !ring_tc) {
    // the append as its own launch ahead of the step
    cudaError_t e = launch_kv_append(a.k_new, a.v_new, a.seqlens, const_cast<void*>(a.k_cache),
                                     const_cast<void*>(a.v_cache), a.B, a.T, a.hkv, a.cap,
                                     a.is_ring, a.freqs, a.ctl, s, true, a.pg);
    if (e != cudaSuccess) return e;
    a.k_new = nullptr;
    a.v_new = nullptr;
  }
  // a ring of <= 144 slots with <= 32 query rows: tensor cores, the append fused
  if (ring_tc) {
    switch (G) {
      case 1: return launch_ring_tc<1>(a, s);
      case 2: return launch_ring_tc<2>(a, s);
      case 4: return launch_ring_tc<4>(a, s);
      case 8: return launch_ring_tc<8>(a, s);
      default: break;
    }
  }
  return launch_decode_kernel(a, s);
}

}  // namespace hattn
