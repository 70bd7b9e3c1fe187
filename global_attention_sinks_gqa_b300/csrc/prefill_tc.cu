// prefill_tc.cu -- sliding-window / global causal GQA attention with a
// per-head sink, prefill, on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method (MiMo-V2-Flash paper review, sections 3.1, 3.2 and 4; plmsmile notes
// on the MiMo series, MiMo-V2-Flash "local window" and "Learnable Attention
// Sink"): out = softmax over {visible keys, sink} of scale * q'.k' applied to
// the values (the sink has no value), lse = log of that denominator.  q' and
// k' carry RoPE on dims 0..63.  The keys' rotated dims 0..63 arrive from a
// separate pass (or a cache) and their dims 64..191 straight from k, through
// a second tensor map; Q is rotated here, in shared memory, once per tile.
// The 64 rotated dims are fp16 operands (11 significant bits) and the other
// 128 dims bf16, so QK^T runs as 4 fp16 k-steps plus 8 bf16 k-steps into one
// fp32 accumulator.
//
// Work decomposition (ours).  A tile is 128 query rows = TQ = 128/G
// consecutive tokens x the G query heads that share one KV head, so every K/V
// byte fetched serves all G heads (GQA reuse through the M dimension of the
// MMA).  A unit is two such tiles, A and B (2*TQ consecutive tokens), that
// walk the same key blocks of BN keys: a sliding-window unit walks only the
// band [t0 - W + 1, t0 + 2*TQ - 1], a global unit every block up to its
// diagonal.  The two tiles ping-pong: while the tensor core multiplies one,
// the other's softmax runs.
//
// CTA roles (384 threads, persistent over units):
//   warp 0      TMA producer: Q tiles (3 boxes of 64 dims each) and the key
//               blocks, in slots of one [BN keys][64 dims] box (128-byte
//               swizzle): a K block is 3 consecutive slots, a V block 2.
//               Several blocks per unit: K in KST stages, V in one, loaded
//               K_0, Q_A, Q_B, K_1, V_0, K_2, V_1, ...; K_0 lands on the K_0
//               barrier of its stage, V_j and K_{j+1} on tile A's P barrier
//               of block j (one wait of the MMA issuer covers both); the K
//               stages are released by tile B's rows, the V stage by a
//               commit.  One block per unit: one K and one V stage whose
//               release (and that of the Q tiles) the producer reads from the
//               phases of the S and PV completion barriers; between a unit's
//               K and V blocks it publishes the next unit (the work counter
//               drawn a unit ahead), which the softmax warps take, with its
//               RoPE angles, while their S products run.
//   warp 1      TMEM allocator and single-thread MMA issuer, per key block j:
//                 O_A += P_A,j V_j ; S_A = Q_A K_{j+1}^T ;
//                 O_B += P_B,j V_j ; S_B = Q_B K_{j+1}^T
//               (S: M=128, N=BN, K=192 from shared memory; PV: P from TMEM,
//               V from shared memory).  The tensor core runs them in issue
//               order, so S_t may be rewritten right behind the PV reading P_t.
//               (Two issuers, one per tile, measured slower: their products
//               enter the pipe interleaved, both S complete together and the
//               two softmaxes run while the pipe idles.)
//   warps 2-3   idle (they complete warpgroup 0 for the register split)
//   warps 4-7   tile A, one thread per query row (TMEM lane): RoPE of the Q
//   warps 8-11  tile B  tile, masked online softmax in base 2 (running max
//               exact after the first block, then moved only when it grows
//               by more than 2^8, with O rescaled then), P written back to
//               TMEM as bf16 over the consumed S columns, and the epilogue,
//               which folds in the sink: O 2^m / (2^m l + 2^s).  One-block
//               units with all rows valid stage O in shared memory (64-byte
//               swizzled quarters of the head dim: tile A's in the V stage
//               once PV_B is done, tile B's in the spare slots) and one
//               thread per tile stores it by TMA: a quarter of the L1
//               transactions of row-per-thread stores.
// TMEM: S_A 0.., S_B 128.., O_A 256..383, O_B 384..511 (several key blocks
// per unit), or S_A 0.., O_A 128..255, S_B 256.., O_B 384..511 (one block).
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"

namespace hattn {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Map for TMA stores of O [rows, heads, 128] bf16 in quarters of the head
// dim: a 32-element (64-byte) inner box of box_heads x box_rows, 64-byte
// swizzle.
static bool make_out_map(CUtensorMap* m, void* base, long rows, int heads, int box_heads,
                         int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(kDv), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(kDv) * 2, cuuint64_t(kDv) * 2 * heads};
  cuuint32_t box[3] = {32, cuuint32_t(box_heads), cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past 256x growth
constexpr int kThreads = 384;
// Register split (setmaxnreg): warpgroup 0 (producer, MMA issuer, two idle
// warps) drops to kRegsLow, the two softmax warpgroups rise to kRegsHigh.  The
// sum must not exceed what the launch allocated (kThreads x kRegsLaunch), or
// the increase would wait forever; the host checks the kernel's register
// count against kRegsLaunch before every launch.
constexpr int kRegsLaunch = 168;
constexpr int kRegsLow = 152;
constexpr int kRegsHigh = 176;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");

// ONE: a unit's whole key band is one block of BN <= 256 keys (sliding
// window units); otherwise blocks of BN <= 128 keys with an online softmax.
template <int G, int BN, bool ONE>
struct Cfg {
  static constexpr int TQ = 128 / G;                // tokens per tile
  static constexpr int UT = 2 * TQ;                 // tokens per unit (tiles A and B)
  static constexpr int kQBox = 128 * 128;           // [128 rows][64 dims] bf16
  static constexpr int kQBytes = 3 * kQBox;
  static constexpr int kSlot = BN * 128;            // [BN keys][64 dims] bf16
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = 2 * kQBytes;
  static constexpr int kBarBytes = 2048;
  static constexpr int kMaxSmem = 232448;
  static constexpr int NSLOT = (kMaxSmem - 1024 - kBarBytes - kOffRing) / kSlot;
  static constexpr int kOffBar = kOffRing + NSLOT * kSlot;
  // One block: O leaves by TMA stores, staged in 8 KB quarters (128 rows x
  // 32 dims, 64-byte swizzle).  Tile A's four go to the V stage (free once
  // PV_B of the unit is done; the next V block waits for their reads), tile
  // B's to the spare ring slots and the space past the barrier block -- as
  // many as fit (kBAreas); the rest of its row is stored directly.
  static constexpr int kOArea = 8192;
  static constexpr int kVOff = kOffRing + 3 * kSlot;
  static constexpr int kSpareOff = kOffRing + 5 * kSlot;
  static constexpr int kSpareAreas = NSLOT > 5 ? (NSLOT - 5) * kSlot / kOArea : 0;
  static constexpr int kFreeOff = kOffBar + kBarBytes;
  static constexpr int kFreeAreas = (kMaxSmem - 1024 - kFreeOff) / kOArea;
  static constexpr int kBAreas =
      kSpareAreas + kFreeAreas < 4 ? kSpareAreas + kFreeAreas : 4;
  static constexpr int kFreeUsed = kBAreas > kSpareAreas ? kBAreas - kSpareAreas : 0;
  static constexpr int kSmemBytes =
      (ONE ? kFreeOff + kFreeUsed * kOArea : kOffBar + kBarBytes) + 1024;  // + alignment slack
  __host__ __device__ static constexpr int o_area(int t, int q) {
    return t == 0 ? kVOff + q * kOArea
                  : (q < kSpareAreas ? kSpareOff + q * kOArea : kFreeOff + (q - kSpareAreas) * kOArea);
  }
  static constexpr uint32_t kTmemCols = 512;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= (ONE ? 256 : 128), "BN");
  static_assert(kSlot % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
  static_assert(NSLOT >= (ONE ? 5 : 8), "ring must hold a K and a V block (and room to prefetch)");
  // Several key blocks per unit: the slots form KST stages of one K block
  // (3 boxes each) and one stage of one V block (2 boxes, after them), each
  // stage with its own empty barrier (kv_empty[0..KST-1] for K, kv_empty[KST]
  // for V); the blocks land on k0_full[stage] (K_0) or tile A's p_full (the
  // rest).
  // K_{j+1} can then load as soon as K_{j+1-KST} is released and P_A(j - 1)
  // is done, about a key block ahead of its S product.
  static constexpr int KST = (NSLOT - 2) / 3;
  // One block: the unit's band is TQ keys wider than either tile needs
  // (W - 1 + TQ keys), so tile t multiplies only the NT keys from t * TOFF on
  // when TQ is a whole number of 16-key steps; the band then starts at
  // position t0 - W + 1 even where that is negative (those rows load as
  // zeros and are masked), so that the offset stays TQ.
  static constexpr int TOFF = (ONE && TQ % 16 == 0 && BN - TQ >= 16) ? TQ : 0;
  static constexpr int NT = BN - TOFF;
  static_assert(ONE || KST >= 2, "two K stages");
  static_assert(KST <= 4, "one K_0 barrier per K stage");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory");
  static_assert(!ONE || 2 * kSlot >= 4 * kOArea, "tile A's O quarters fit the V stage");
  static_assert(kSlot % 1024 == 0 && kFreeOff % 1024 == 0, "staging areas 1 KB aligned");
};

// TMEM columns of tile t.  Blocks of <= 128 keys: S_A 0, S_B 128, O_A 256,
// O_B 384.  One block of up to 256 keys: S_t at 256 t and O_t at 256 t + 128,
// over the upper S columns, which are dead once the softmax has read them (P
// takes the first BN / 2 columns); the next S_t is written only after the
// epilogue has read O_t.
template <bool ONE>
__host__ __device__ constexpr uint32_t s_col(int t) { return ONE ? 256u * t : (t ? 128u : 0u); }
template <bool ONE>
__host__ __device__ constexpr uint32_t o_col(int t) {
  return ONE ? 256u * t + 128u : (t ? 384u : 256u);
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

template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

constexpr int kCuCache = 128;  // batches up to 127 sequences keep cu_seqlens in shared memory

constexpr int kUnitQueue = 4;          // units the producer may publish ahead
constexpr int kUnitReaders = 1 + 8;    // the MMA issuer and the eight softmax warps

// t0: index of the unit's first query among its sequence's new tokens; P:
// positions before them (the cached prefix; 0 for a plain prefill); key and
// query positions (kstart, masks, RoPE) count from the sequence's start.
struct UnitInfo {
  int b, g, t0, L, tok0, kstart, nblk, P;
};

template <int NSLOT>
struct Bars {
  uint64_t q_full[2], q_ready[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  uint64_t kv_full[NSLOT], kv_empty[NSLOT];
  // several key blocks per unit: K_0 of each unit, one barrier per K stage
  // (a unit of one block may start loading the next unit's K_0 before its
  // own K_0 has landed; per stage, the stage's previous K_0 was consumed)
  uint64_t k0_full[4];
  // one block per unit: tile t's O quarters are staged (128 rows), and tile
  // A's TMA stores have read theirs out of the V stage
  uint64_t o_staged[2], o_read;
  uint64_t unit_full[kUnitQueue], unit_empty[kUnitQueue];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int unit[kUnitQueue];         // published unit indices, -1: no more
  UnitInfo uinfo[kUnitQueue];  // and what unit_info() gave for them
  int cu[kCuCache];
};

// Unit u of the persistent loop.  Global units run latest (longest) first so
// the tail of the schedule is short; window units run in order.  False for a
// unit past its sequence's end and for every unit of a sequence whose
// device-resident offsets (or prefix) are out of range; `report` records
// the latter as HATTN_ERR_INVALID_ARG (the producer, which sees every unit
// once, reports).
template <int G, int BN, bool WIN, bool UNCLAMPED = false>
__device__ __forceinline__ bool unit_info(int u, const PrefillArgs& a, const int* cu, int nut,
                                          UnitInfo& ui, bool report = false) {
  constexpr int UT = 256 / G;
  const int per = a.batch * a.hkv;
  const int q_ord = u / per;
  const int rem = u - q_ord * per;
  const int qt = WIN ? q_ord : (nut - 1 - q_ord);
  ui.b = rem / a.hkv;
  ui.g = rem - ui.b * a.hkv;
  if (!seq_slice(cu, ui.b, a.total, a.max_seqlen, a.ctl, report, ui.tok0, ui.L)) return false;
  ui.t0 = qt * UT;
  if (ui.t0 >= ui.L) return false;
  ui.P = a.prefix != nullptr ? __ldg(a.prefix + ui.b) : a.lead;
  if (a.prefix != nullptr && (ui.P < 0 || long(ui.P) + ui.L > a.cap)) {
    if (report) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
    return false;
  }
  const int qend = ui.P + min(ui.t0 + UT, ui.L);  // one past the last valid query position
  ui.kstart = WIN ? (UNCLAMPED ? ui.P + ui.t0 - a.window + 1 : max(0, ui.P + ui.t0 - a.window + 1))
                  : 0;
  ui.nblk = (qend - ui.kstart + BN - 1) / BN;
  return true;
}

// Masks of one block: columns past the causal edge (c > c_hi) and / or
// before the window's far edge (c < c_lo) become -inf.  A block only pays for
// the edges that fall inside it.
template <int BN>
__device__ __forceinline__ void mask_block(uint32_t (&s)[BN], bool lower, bool upper, int c_lo,
                                           int c_hi) {
  if (lower && upper) {
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (unsigned(c - c_lo) > unsigned(c_hi - c_lo)) s[c] = __float_as_uint(-INFINITY);
  } else if (lower) {
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (c < c_lo) s[c] = __float_as_uint(-INFINITY);
  } else if (upper) {
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (c > c_hi) s[c] = __float_as_uint(-INFINITY);
  }
}

// Masks of a whole one-block band: columns c < c_lo or c > c_hi of this row
// become -inf, checked only in the 16-column chunks that some row of the tile
// loses a column in (lo_max: the largest c_lo of the tile, hi_min: the
// smallest c_hi).  The chunk tests are the same for every row, so the warps
// do not diverge; a window tile then checks about 32 of its columns.
template <int N>
__device__ __forceinline__ void mask_band(uint32_t (&s)[N], int c_lo, int c_hi, int lo_max,
                                          int hi_min) {
  static_assert(N % 16 == 0, "16-column chunks");
#pragma unroll
  for (int c0 = 0; c0 < N; c0 += 16) {
    const bool lo = c0 < lo_max, hi = c0 + 15 > hi_min;
    if (lo && hi) {
#pragma unroll
      for (int c = c0; c < c0 + 16; ++c)
        if (c < c_lo || c > c_hi) s[c] = __float_as_uint(-INFINITY);
    } else if (lo) {
#pragma unroll
      for (int c = c0; c < c0 + 16; ++c)
        if (c < c_lo) s[c] = __float_as_uint(-INFINITY);
    } else if (hi) {
#pragma unroll
      for (int c = c0; c < c0 + 16; ++c)
        if (c > c_hi) s[c] = __float_as_uint(-INFINITY);
    }
  }
}

// One block of the online softmax for one query row.  s holds the row's BN
// (masked) raw logits.  Writes P (bf16) into the S columns and updates the
// running max m (log2 units, -inf before the first block) and the sum l of
// 2^(x - m).  The first block sets m to its exact maximum, so the dominant
// key's weight is exactly 1 in bf16; later blocks move m only when the max
// grows by more than 2^8 (then O, l are rescaled).
template <int BN>
__device__ __forceinline__ void softmax_block(uint32_t (&s)[BN], float scale_log2, uint32_t t_s,
                                              uint32_t t_o, bool may_rescale, float& m, float& l) {
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int c = 0; c + 3 < BN; c += 4) {
    mx0 = fmax3f(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    mx1 = fmax3f(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
  }
  const float m_new = fmaxf(m, fmaxf(mx0, mx1) * scale_log2);
  const bool resc = m_new > m + kRescaleThreshold;
  float alpha = 1.f;
  if (resc) {
    alpha = fast_exp2(m - m_new);  // 0 when m was -inf
    m = m_new;
    l *= alpha;
  }
  const float msub = (m == -INFINITY) ? 0.f : m;
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
  const uint64_t nm2 = f2_pack(-msub, -msub);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < BN; c += 16) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 x = f2_unpack(
          f2_fma(f2_pack(__uint_as_float(s[c + e]), __uint_as_float(s[c + e + 1])), sc2, nm2));
      const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
      pk[e >> 1] = pack_bf16x2(p0, p1);
      if (e & 2)
        acc1 = f2_add(acc1, f2_pack(p0, p1));
      else
        acc0 = f2_add(acc0, f2_pack(p0, p1));
    }
    tmem_st8(t_s + (c >> 1), pk);  // P (bf16 pairs) over consumed S columns
  }
  const float2 sum = f2_unpack(f2_add(acc0, acc1));
  l += sum.x + sum.y;
  if (may_rescale && __any_sync(0xffffffffu, resc)) {
    // O holds the earlier blocks scaled by 2^-m_old; the PV that wrote them is
    // complete (the S block just waited for was committed after it), and the
    // PV of this block waits for p_full, which follows this rescale.
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
}

// P = 2^(x * scale - msub) of n raw logits, written as bf16 pairs into the
// TMEM columns starting at t_p; returns the sum of the fp32 weights.
template <int N>
__device__ __forceinline__ float exp_pack_store(const uint32_t (&s)[N], float scale_log2, float msub,
                                                uint32_t t_p) {
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
  const uint64_t nm2 = f2_pack(-msub, -msub);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < N; c += 16) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 x = f2_unpack(
          f2_fma(f2_pack(__uint_as_float(s[c + e]), __uint_as_float(s[c + e + 1])), sc2, nm2));
      const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
      pk[e >> 1] = pack_bf16x2(p0, p1);
      if (e & 2)
        acc1 = f2_add(acc1, f2_pack(p0, p1));
      else
        acc0 = f2_add(acc0, f2_pack(p0, p1));
    }
    tmem_st8(t_p + (c >> 1), pk);
  }
  const float2 sum = f2_unpack(f2_add(acc0, acc1));
  return sum.x + sum.y;
}

template <int N>
__device__ __forceinline__ float row_max(const uint32_t (&s)[N]) {
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int c = 0; c + 3 < N; c += 4) {
    mx0 = fmax3f(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    mx1 = fmax3f(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
  }
  return fmaxf(mx0, mx1);
}

template <int BN>
__device__ __forceinline__ void load_s_row(uint32_t t_s, uint32_t (&s)[BN]) {
  int c = 0;
#pragma unroll
  for (; c + 32 <= BN; c += 32) tmem_ld32_nowait(t_s + c, s + c);
#pragma unroll
  for (; c < BN; c += 16) tmem_ld16_nowait(t_s + c, s + c);
  tmem_ld_wait();
#pragma unroll
  for (int e = 0; e < BN; ++e) tmem_reg_fence(s[e]);
}

// The whole key band of a unit as one block of BN columns, in two halves of
// H1 and H2 columns (registers).  Half 1 sets the max m; half 2 is taken
// against m unless its own max exceeds m by more than 2^8, in which case m
// moves and half 1's weights, already in TMEM as bf16 over S, are scaled to
// the new max (rare: the row's weights would otherwise grow past 256 in
// bf16; a weight scaled down by more than 2^8 keeps a relative error of
// 2^-8, i.e. 2^-16 of the row's largest weight).  c_lo / c_hi: this row's visible columns;
// lo_max / hi_min: the largest c_lo and smallest c_hi over the tile, which
// decide which edges a half has to mask.  Returns m (log2 units, -inf if no
// column is visible) and l = sum of 2^(x - m).
template <int BN>
__device__ __forceinline__ void softmax_one(uint32_t t_s, float scale_log2, int c_lo, int c_hi,
                                            int lo_max, int hi_min, float& m, float& l) {
  constexpr int H1 = ((BN / 2 + 15) / 16) * 16;
  constexpr int H2 = BN - H1;
  float l1;
  {
    uint32_t s1[H1];
    load_s_row<H1>(t_s, s1);
    mask_band<H1>(s1, c_lo, c_hi, lo_max, hi_min);
    m = row_max<H1>(s1) * scale_log2;
    l1 = exp_pack_store<H1>(s1, scale_log2, m == -INFINITY ? 0.f : m, t_s);
  }
  bool redo;
  float l2, f1 = 1.f;
  {
    uint32_t s2[H2];
    load_s_row<H2>(t_s + H1, s2);
    mask_band<H2>(s2, c_lo - H1, c_hi - H1, lo_max - H1, hi_min - H1);
    const float m2 = fmaxf(m, row_max<H2>(s2) * scale_log2);
    redo = m2 > m + kRescaleThreshold;
    if (redo) {
      f1 = fast_exp2(m - m2);  // 0 when half 1 saw no key
      m = m2;
    }
    l2 = exp_pack_store<H2>(s2, scale_log2, m == -INFINITY ? 0.f : m, t_s + H1 / 2);
  }
  if (__any_sync(0xffffffffu, redo)) {
    // half 1's P (bf16 pairs in TMEM columns 0 .. H1/2 - 1) times f1
    constexpr int NP = H1 / 2;
    static_assert(NP % 8 == 0, "P columns in pieces of 8");
    uint32_t pv[NP];
    tmem_st_wait();  // half 1's P stores have landed
#pragma unroll
    for (int c = 0; c < NP; c += 8) tmem_ld8_nowait(t_s + c, pv + c);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < NP; c += 8) {
      uint32_t pk[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        tmem_reg_fence(pv[c + e]);
        const float2 x = unpack_bf16x2(pv[c + e]);
        pk[e] = pack_bf16x2(x.x * f1, x.y * f1);
      }
      tmem_st8(t_s + c, pk);
    }
    l1 *= f1;
  }
  l = l1 + l2;
}

template <int G, int BN, bool WIN, bool ONE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap mapQ,
                   const __grid_constant__ CUtensorMap mapK0,
                   const __grid_constant__ CUtensorMap mapK12,
                   const __grid_constant__ CUtensorMap mapV,
                   const __grid_constant__ CUtensorMap mapO, const PrefillArgs a) {
  using C = Cfg<G, BN, ONE>;
  constexpr int TQ = C::TQ;
  constexpr int NSLOT = C::NSLOT;
  static_assert(sizeof(Bars<NSLOT>) <= C::kBarBytes, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars<NSLOT>* bars = reinterpret_cast<Bars<NSLOT>*>(smem + C::kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nut = (a.max_seqlen + C::UT - 1) / C::UT;
  const int nunits = nut * a.batch * a.hkv;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_ready[t], 128);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->s_full[t], 1);
      // several key blocks per unit: tile A's P barrier also takes the
      // producer's V_j and K_{j+1} (or the softmax's stand-in on a unit's
      // last block)
      mbar_init(&bars->p_full[t], (!ONE && t == 0) ? 130 : 128);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_free[t], 128);
    }
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < kUnitQueue; ++i) {
      mbar_init(&bars->unit_full[i], 1);
      mbar_init(&bars->unit_empty[i], kUnitReaders);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars->k0_full[i], 1);
    for (int t = 0; t < 2; ++t) mbar_init(&bars->o_staged[t], 128);
    mbar_init(&bars->o_read, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapQ);
    tma_prefetch_map(&mapK0);
    tma_prefetch_map(&mapK12);
    tma_prefetch_map(&mapV);
    if (ONE && a.o_tma) tma_prefetch_map(&mapO);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  // no offsets (one shard of a sequence): the single sequence holds every row
  const bool cu_cached = a.batch + 1 <= kCuCache || a.cu_seqlens == nullptr;
  if (a.cu_seqlens == nullptr) {
    if (threadIdx.x == 0) {
      bars->cu[0] = 0;
      bars->cu[1] = int(a.total);
    }
  } else if (cu_cached) {
    for (int i = threadIdx.x; i <= a.batch; i += kThreads) bars->cu[i] = __ldg(a.cu_seqlens + i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  uint8_t* ring = smem + C::kOffRing;
  const int* cu = cu_cached ? bars->cu : a.cu_seqlens;
  // Units are handed out by a counter in global memory, so SMs that run
  // faster take more of them; the producer draws each unit and publishes its
  // index and its UnitInfo in a small queue that the MMA issuer and the
  // softmax warps read in the same order (-1: no more units).  n: queue
  // entries read so far; ui (when given): the unit's UnitInfo.
  auto read_unit = [&](uint32_t& n, bool whole_warp, UnitInfo* ui = nullptr) -> int {
    const uint32_t q = n % kUnitQueue, ph = (n / kUnitQueue) & 1u;
    const bool ok = whole_warp ? warp_wait(&bars->unit_full[q], ph, a.ctl, abort)
                               : mbar_wait(&bars->unit_full[q], ph, a.ctl, abort);
    if (!ok) return -1;
    const int u = bars->unit[q];
    if (ui != nullptr) *ui = bars->uinfo[q];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&bars->unit_empty[q]);
    ++n;
    return u;
  };

  if (warp < 4) {
    reg_dealloc<kRegsLow>();  // one instruction for all of warpgroup 0
    if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t qfills0 = 0, qfills1 = 0;  // Q loads issued into the tile A / B buffer
      bool ok = true;
      // K / V box of key position kpos of unit ui: packed keys [total, hkv, d]
      // (coordinates: KV head, token) or a cache [B, hkv, cap, d] (slot, plane)
      auto kv_c1 = [&](const UnitInfo& ui, int kpos) {
        return a.prefix != nullptr ? kpos : ui.g;
      };
      auto kv_c2 = [&](const UnitInfo& ui, int kpos) {
        return a.prefix != nullptr ? ui.b * a.hkv + ui.g : ui.tok0 + kpos;
      };
      // box i of a key block: dims 64 i .. 64 i + 63, the rotated ones (i = 0)
      // through mapK0, the others through mapK12
      auto kmap = [&](int i) { return i == 0 ? &mapK0 : &mapK12; };
      uint32_t un = 0;  // one-block units whose K and V were loaded
      // several key blocks per unit: whole K / V blocks into their stages.
      // K_0 of a unit completes k0_full of its stage.  K_{j+1} and V_j instead complete
      // phase j of tile A's p_full together with the softmax's P_A(j), so
      // that one wait of the MMA issuer covers PV_A(j) and S(j + 1).  Each
      // arrives (with its bytes) only once phase j - 1 is complete: K_{j+1}
      // waits for it here; V_j loads into a stage that PV_B(j - 1) released,
      // and PV_B(j - 1) was issued after that phase.  Phase j cannot complete
      // without these arrivals, so the parity waited on cannot alias.
      uint32_t kq = 0, vq = 0;    // K and V blocks loaded (vq: p_full[0] phases joined)
      uint32_t k0n[C::KST] = {};  // phases of k0_full[stage] (units whose K_0 went there)
      // Launched as a dependent of the key-rotation (or append) kernel, this
      // CTA may start before that kernel ends.  What it writes -- the rotated
      // keys, the caches, the work counter -- is read only after the wait
      // below, which this thread alone passes through; Q, the offsets and
      // the sinks were complete before that kernel started.
      bool dep = false;
      auto dep_wait = [&]() {
        if (!dep) {
          grid_dep_wait();
          dep = true;
        }
      };
      auto load_k = [&](const UnitInfo& ui, int kpos, bool first) -> bool {
        dep_wait();
        const uint32_t st = kq % C::KST, ph = (kq / C::KST) & 1u;
        if (!mbar_wait(&bars->kv_empty[st], ph ^ 1u, a.ctl, abort)) return false;
        if (!first && vq > 0 && !mbar_wait(&bars->p_full[0], (vq - 1) & 1u, a.ctl, abort))
          return false;
        uint64_t* full = first ? &bars->k0_full[st] : &bars->p_full[0];
        mbar_arrive_expect_tx(full, 3 * C::kSlot);
        for (int i = 0; i < 3; ++i)
          tma_load_3d(ring + (st * 3 + i) * C::kSlot, kmap(i), full, 64 * i, kv_c1(ui, kpos),
                      kv_c2(ui, kpos));
        ++kq;
        if (first) ++k0n[st];
        return true;
      };
      auto load_v = [&](const UnitInfo& ui, int vpos) -> bool {
        dep_wait();
        if (!mbar_wait(&bars->kv_empty[C::KST], (vq & 1u) ^ 1u, a.ctl, abort)) return false;
        mbar_arrive_expect_tx(&bars->p_full[0], 2 * C::kSlot);
        for (int i = 0; i < 2; ++i)
          tma_load_3d(ring + (C::KST * 3 + i) * C::kSlot, &mapV, &bars->p_full[0], 64 * i,
                      kv_c1(ui, vpos), kv_c2(ui, vpos));
        ++vq;
        return true;
      };
      uint32_t pn = 0;  // queue entries published
      // The first unit of CTA i is unit i (its Q tiles load before the
      // wait); the counter hands out the rest, from unit gridDim.x on.  One-
      // block units draw the counter one unit ahead: its round trip (over a
      // microsecond while HBM is busy) then overlaps a unit's loads.
      int ahead = -1;  // a counter draw taken ahead, or -1
      auto draw = [&](UnitInfo& ui) -> int {
        int u;
        bool fixed = pn == 0;
        do {
          if (fixed) {
            u = int(blockIdx.x);
            fixed = false;
          } else {
            dep_wait();
            if (ahead >= 0) {
              u = ahead;
              ahead = -1;
            } else {
              u = int(gridDim.x + atomicAdd(a.unit_ctr, 1u));
            }
          }
        } while (u < nunits && !unit_info<G, BN, WIN, (C::TOFF > 0)>(u, a, cu, nut, ui, true));
        return u < nunits ? u : -1;
      };
      // publish a unit that holds a query (or the end, -1) in the queue
      auto publish = [&](int u, const UnitInfo& ui) -> bool {
        const uint32_t q = pn % kUnitQueue;
        if (pn >= uint32_t(kUnitQueue) &&
            !mbar_wait(&bars->unit_empty[q], ((pn / kUnitQueue) & 1u) ^ 1u, a.ctl, abort))
          return false;
        bars->unit[q] = u;
        bars->uinfo[q] = ui;
        mbar_arrive(&bars->unit_full[q]);
        ++pn;
        return true;
      };
      UnitInfo ui;
      int u = draw(ui);
      ok = publish(u, ui);
      while (ok && u >= 0) {
        const int k0pos = ui.kstart;
        // Several blocks: K_0 first (its stage frees while the previous
        // unit finishes), then the two Q tiles, then K_1, V_0, K_2, V_1, ...  One
        // block: the Q tiles first -- a tile's buffer frees with its S MMA of
        // the previous unit and its RoPE heads the tile's next chain -- then
        // K_0, the next unit's queue entry (the softmax warps read it while
        // this unit's S products run), V_0.
        // (The CTA's first unit loads its Q tiles before K_0: they need no
        // wait for the kernel before this one.)
        const bool q_first = pn == 1;
        if (!ONE && !q_first) ok = load_k(ui, k0pos, true);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          uint32_t& qf = t ? qfills1 : qfills0;
          // one-block units: Q_t is free once the previous unit's S_t is
          // done (the phase of s_full[t]; the next phase needs this load, so
          // the parity cannot alias); several blocks: its own barrier
          const bool qfree =
              ONE ? (qf == 0 || mbar_wait(&bars->s_full[t], (qf - 1) & 1u, a.ctl, abort))
                  : mbar_wait(&bars->q_empty[t], (qf & 1u) ^ 1u, a.ctl, abort);
          if (!qfree) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->q_full[t], C::kQBytes);
          uint8_t* qdst = smem + C::kOffQ + t * C::kQBytes;
          for (int i = 0; i < 3; ++i)
            tma_load_3d(qdst + i * C::kQBox, &mapQ, &bars->q_full[t], 64 * i, ui.g * G,
                        ui.tok0 + ui.t0 + t * TQ);
          ++qf;
        }
        if (!ONE && q_first && ok) ok = load_k(ui, k0pos, true);
        UnitInfo nui;
        int nu = -1;
        if constexpr (ONE) {
          // the unit's K block (slots 0-2) once the previous unit's S_B is
          // done, its V block (slots 3-4) once its PV_B is: the phases of
          // s_full[1] and pv_done[1] (products complete in issue order)
          dep_wait();
          if (ok && un > 0)
            ok = mbar_wait(&bars->s_full[1], (un - 1) & 1u, a.ctl, abort);
          if (ok) {
            mbar_arrive_expect_tx(&bars->kv_full[0], 3 * C::kSlot);
            for (int i = 0; i < 3; ++i)
              tma_load_3d(ring + i * C::kSlot, kmap(i), &bars->kv_full[0], 64 * i,
                          kv_c1(ui, k0pos), kv_c2(ui, k0pos));
          }
          if (ok) {
            nu = draw(nui);
            ok = publish(nu, nui);
            if (nu >= 0) ahead = int(gridDim.x + atomicAdd(a.unit_ctr, 1u));
          }
          // (and once tile A's TMA stores of the previous unit's O have read
          // their staging out of the V stage)
          if (ok && un > 0)
            ok = mbar_wait(&bars->pv_done[1], (un - 1) & 1u, a.ctl, abort) &&
                 mbar_wait(&bars->o_read, (un - 1) & 1u, a.ctl, abort);
          if (ok) {
            mbar_arrive_expect_tx(&bars->kv_full[1], 2 * C::kSlot);
            for (int i = 0; i < 2; ++i)
              tma_load_3d(ring + (3 + i) * C::kSlot, &mapV, &bars->kv_full[1], 64 * i,
                          kv_c1(ui, k0pos), kv_c2(ui, k0pos));
            ++un;
          }
        } else {
          // K_{j+1} (its stage frees when S of K_{j+1-KST} completes) before
          // V_j (its stage frees when PV of V_{j-1} completes): the order in
          // which the products release them
          for (int j = 0; j < ui.nblk && ok; ++j) {
            const int vpos = k0pos + j * BN;
            if (j + 1 < ui.nblk) ok = load_k(ui, vpos + BN, false);
            if (ok) ok = load_v(ui, vpos);
          }
          if (ok) {
            nu = draw(nui);
            ok = publish(nu, nui);
          }
        }
        u = nu;
        ui = nui;
      }
      // never leave with copies in flight into this CTA's shared memory
      if (qfills0) mbar_wait_drain(&bars->q_full[0], (qfills0 - 1) & 1u, a.ctl);
      if (qfills1) mbar_wait_drain(&bars->q_full[1], (qfills1 - 1) & 1u, a.ctl);
      if constexpr (ONE) {
        if (un) {
          mbar_wait_drain(&bars->kv_full[0], (un - 1) & 1u, a.ctl);
          mbar_wait_drain(&bars->kv_full[1], (un - 1) & 1u, a.ctl);
        }
      } else {
        for (int st = 0; st < C::KST; ++st)
          if (k0n[st]) mbar_wait_drain(&bars->k0_full[st], (k0n[st] - 1) & 1u, a.ctl);
        if (vq) mbar_wait_drain(&bars->p_full[0], (vq - 1) & 1u, a.ctl);
      }
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_rot = make_idesc_f16(128, C::NT, 0, 0);   // dims 0..63
      constexpr uint32_t idesc_s = make_idesc_bf16(128, C::NT, 0, 0);    // dims 64..191
      constexpr uint32_t idesc_o = make_idesc_bf16(128, 128, 0, 1);
      const uint32_t qbase = smem_u32(smem + C::kOffQ);
      const uint32_t rbase = smem_u32(ring);
      uint32_t blk = 0;   // key blocks completed by both tiles so far
      uint32_t uc = 0;    // units started
      bool ok = true;
      // Shared-memory descriptors are built once; a k-step or slot only adds
      // its byte offset / 16 to the start-address field (addresses stay below
      // 256 KB, so the 14-bit field never carries).
      const uint64_t qdesc0 = make_sdesc_sw128(qbase, 16, 1024);
      const uint64_t kdesc0 = make_sdesc_sw128(rbase, 16, 1024);
      const uint64_t vdesc0 = make_sdesc_sw128(rbase, C::kSlot, 1024);
      // a K block sits in 3 consecutive slots from kslot, a V block in 2 from
      // vslot (dims 0..63 then 64..127: one N=128 MMA per k-step spans both)
      // (tile t's keys start TOFF * t rows into the block: whole 8-row
      // swizzle atoms, 16-key steps)
      auto issue_qk = [&](int t, uint32_t kslot) {
        const uint64_t qd = qdesc0 + uint64_t((t * C::kQBytes) >> 4);
        const uint64_t kd = kdesc0 + uint64_t((kslot * C::kSlot + t * C::TOFF * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < 12; ++kk)
          umma_ss(tmem + s_col<ONE>(t), qd + uint64_t(((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4),
                  kd + uint64_t(((kk >> 2) * C::kSlot + (kk & 3) * 32) >> 4),
                  kk < 4 ? idesc_rot : idesc_s, kk > 0 ? 1u : 0u);
      };
      auto issue_pv = [&](int t, uint32_t vslot, bool acc) {
        const uint64_t vd = vdesc0 + uint64_t((vslot * C::kSlot) >> 4);
        const uint32_t p_tmem = tmem + s_col<ONE>(t);
#pragma unroll
        for (int kk = 0; kk < C::NT / 16; ++kk)
          umma_ts(tmem + o_col<ONE>(t), p_tmem + kk * 8,
                  vd + uint64_t(((t * C::TOFF + 16 * kk) * 128) >> 4), idesc_o,
                  (acc || kk > 0) ? 1u : 0u);
      };
      if constexpr (ONE) {
        // one key block per unit: S_t = Q_t K^T once O_t (over S_t's upper
        // columns) has been read by the previous unit's epilogue, then
        // O_t = P_t V
        // (the producer takes the release of Q_t, K and V from the phases of
        // s_full[t], s_full[1] and pv_done[1]: no commits of their own)
        uint32_t rn = 0;
        while (ok) {
          const int u = read_unit(rn, false);
          if (u < 0) break;
          if (!mbar_wait(&bars->kv_full[0], uc & 1u, a.ctl, abort)) break;
          for (int t = 0; t < 2 && ok; ++t) {
            if (!mbar_wait(&bars->q_ready[t], uc & 1u, a.ctl, abort) ||
                (uc > 0 && !mbar_wait(&bars->o_free[t], (uc - 1) & 1u, a.ctl, abort))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(t, 0);
            umma_commit(&bars->s_full[t]);
          }
          if (!ok) break;
          if (!mbar_wait(&bars->kv_full[1], uc & 1u, a.ctl, abort)) break;
          for (int t = 0; t < 2 && ok; ++t) {
            if (!mbar_wait(&bars->p_full[t], uc & 1u, a.ctl, abort)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, 3, false);
            umma_commit(&bars->pv_done[t]);
          }
          if (!ok) break;
          ++uc;
        }
      } else {
      // K blocks in KST stages (the stage of the c-th K block is c % KST;
      // K stage s holds slots 3s .. 3s + 2), V blocks in one stage (slots
      // 3 KST, 3 KST + 1).  This thread waits on K_0 of a unit (k0_full of
      // its stage) and then, per key block j, only on P_A(j) -- whose barrier also
      // carries V_j and K_{j+1} -- and P_B(j); the softmax of tile B
      // releases each K stage once it has seen S_B of that block.  Every
      // wait and commit costs this thread hundreds of cycles while the
      // products stream operands out of shared memory, so it makes three
      // commits and two waits per block.
      uint32_t kc = 0;
      uint32_t k0c[C::KST] = {};  // K_0 blocks taken from each K stage
      auto next_kslot = [&]() -> uint32_t {
        const uint32_t st = kc % C::KST;
        ++kc;
        return 3 * st;
      };
      constexpr uint32_t kVPos = 3 * C::KST;
      uint32_t rn = 0;
      while (ok) {
        const int u = read_unit(rn, false);
        if (u < 0) break;
        UnitInfo ui;
        unit_info<G, BN, WIN, (C::TOFF > 0)>(u, a, cu, nut, ui);
        const uint32_t k0 = next_kslot();  // slot of stage k0 / 3
        if (!mbar_wait(&bars->k0_full[k0 / 3], k0c[k0 / 3] & 1u, a.ctl, abort)) break;
        ++k0c[k0 / 3];
        for (int t = 0; t < 2 && ok; ++t) {
          if (!mbar_wait(&bars->q_ready[t], uc & 1u, a.ctl, abort)) { ok = false; break; }
          tc_fence_after();
          issue_qk(t, k0);
          umma_commit(&bars->s_full[t]);
          if (ui.nblk == 1) umma_commit(&bars->q_empty[t]);
        }
        if (!ok) break;
        for (int j = 0; j < ui.nblk && ok; ++j, ++blk) {
          const bool more = j + 1 < ui.nblk;
          uint32_t kn = 0;
          for (int t = 0; t < 2; ++t) {
            // t = 0: P_A(j), V_j and (more) K_{j+1} have landed
            if (!mbar_wait(&bars->p_full[t], blk & 1u, a.ctl, abort)) { ok = false; break; }
            if (j == 0 && uc > 0 &&
                !mbar_wait(&bars->o_free[t], (uc - 1) & 1u, a.ctl, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, kVPos, j > 0);
            if (!more) umma_commit(&bars->pv_done[t]);  // the unit's O_t is complete
            if (t == 1) umma_commit(&bars->kv_empty[C::KST]);  // V_j's stage
            if (more) {
              if (t == 0) kn = next_kslot();
              issue_qk(t, kn);
              umma_commit(&bars->s_full[t]);
              if (j + 2 == ui.nblk) umma_commit(&bars->q_empty[t]);
            }
          }
        }
        ++uc;
      }
      }
      // every MMA issued must be complete before TMEM is released
      umma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, a.ctl);
    }
    }  // warps 2 and 3: idle
  } else {
    // ------------------------------------------------------------ softmax rows
    reg_alloc<kRegsHigh>();
    const int t = (warp - 4) >> 2;             // tile: warps 4-7 -> A, 8-11 -> B
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;            // query row of the tile
    const int hl = r % G;
    const int tl = r / G;
    const uint32_t lane_addr = uint32_t(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + s_col<ONE>(t);
    const uint32_t t_o = tmem + lane_addr + o_col<ONE>(t);
    uint32_t blk = 0, uc = 0;
    // the previous unit's row, finished after the next unit's Q is rotated
    bool have_prev = false;
    float pm = 0.f, pl = 0.f, psink = 0.f;
    bool pvalid = false;
    long porow = 0;
    // one block per unit: the tile's first token row and head, and whether
    // all its rows are valid (then O leaves by TMA)
    int ptok = 0, pgh = 0;
    bool pfull = false;
    uint32_t nstaged = 0;  // epilogues of this tile that staged O (phases of o_staged[t])
    uint32_t puc = 0;  // index of the unit the epilogue finishes

    const bool out32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
    auto epilogue = [&]() -> bool {
      if (!warp_wait(&bars->pv_done[t], puc & 1u, a.ctl, abort)) return false;
      tc_fence_after();
      // fold in the sink: denominator 2^m l + 2^s, taken relative to max(m, s)
      const float mt = fmaxf(pm, psink);
      const float msub = (mt == -INFINITY) ? 0.f : mt;
      const float fo = exp2f(pm - msub);
      const float l_tot = pl * fo + exp2f(psink - msub);
      const float inv = fo / l_tot;
      const uint64_t inv2 = f2_pack(inv, inv);
      // O leaves TMEM first (scaled, packed to bf16 in registers), so O_t's
      // columns go back to the MMA before the stores, whose drain then
      // overlaps the next unit's QK^T
      uint32_t pk[64];
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // 64 columns in flight per wait
        uint32_t v[64];
        tmem_ld32_nowait(t_o + half * 64, v);
        tmem_ld32_nowait(t_o + half * 64 + 32, v + 32);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 64; ++e) tmem_reg_fence(v[e]);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 y = f2_unpack(
              f2_mul(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), inv2));
          pk[32 * half + e] = pack_bf16x2(y.x, y.y);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
      if constexpr (ONE) {
        if (a.o_tma && pfull) {
          // Tile A stages into the V stage, which PV_B of the unit must
          // have finished reading.  16-byte chunk c of row r's quarter sits
          // at c ^ (r / 2 % 4) (64-byte swizzle: conflict-free).
          if (t == 0 && !warp_wait(&bars->pv_done[1], puc & 1u, a.ctl, abort)) return false;
          const int nq = t == 0 ? 4 : C::kBAreas;
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            if (qd < nq) {
              uint8_t* row = smem + C::o_area(t, qd) + r * 64;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(row + ((c ^ ((r >> 1) & 3)) << 4)) =
                    make_uint4(pk[16 * qd + 4 * c], pk[16 * qd + 4 * c + 1],
                               pk[16 * qd + 4 * c + 2], pk[16 * qd + 4 * c + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&bars->o_staged[t]);
          // the quarters that found no staging area: stored directly
          uint8_t* dst = static_cast<uint8_t*>(a.out) + porow * 256;
#pragma unroll
          for (int qd = 0; qd < 4; ++qd)
            if (qd >= nq) {
              if (out32) {
                st_global_v8(dst + 64 * qd, pk + 16 * qd);
                st_global_v8(dst + 64 * qd + 32, pk + 16 * qd + 8);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  reinterpret_cast<uint4*>(dst + 64 * qd)[e] =
                      make_uint4(pk[16 * qd + 4 * e], pk[16 * qd + 4 * e + 1],
                                 pk[16 * qd + 4 * e + 2], pk[16 * qd + 4 * e + 3]);
              }
            }
          // one thread of the tile stores the staged boxes once all 128
          // rows are in, and (tile A) reports when they have been read
          bool good = true;
          if (r == 0) {
            good = mbar_wait(&bars->o_staged[t], nstaged & 1u, a.ctl, abort);
            if (good) {
              for (int qd = 0; qd < nq; ++qd)
                tma_store_3d(&mapO, smem + C::o_area(t, qd), 32 * qd, pgh, ptok);
              bulk_commit();
              bulk_wait_read();
              if (t == 0) mbar_arrive(&bars->o_read);
            }
          }
          ++nstaged;
          if (!__shfl_sync(0xffffffffu, good, 0)) return false;
          if (a.lse != nullptr) a.lse[porow] = (msub + log2f(l_tot)) * kLn2;
          return true;
        }
        if (t == 0 && r == 0) mbar_arrive(&bars->o_read);  // nothing staged
      }
      if (pvalid) {
        uint8_t* dst = static_cast<uint8_t*>(a.out) + porow * 256;
        if (out32) {  // 32-byte stores: one full sector each
#pragma unroll
          for (int e = 0; e < 8; ++e) st_global_v8(dst + 32 * e, pk + 8 * e);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            reinterpret_cast<uint4*>(dst)[e] =
                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
        if (a.lse != nullptr) a.lse[porow] = (msub + log2f(l_tot)) * kLn2;
      }
      return true;
    };

    // RoPE angles of this row's token in unit x: the G lanes holding one
    // token's heads each evaluate 32/G of the 32 and exchange them by
    // shuffles when rotating.
    auto angles = [&](const UnitInfo& x, float2 (&cs)[32 / G]) {
      const int pos = x.P + x.t0 + t * TQ + tl + a.rope_off;
#pragma unroll
      for (int k2 = 0; k2 < 32 / G; ++k2)
        cs[k2] = rope_cos_sin(pos, a.freqs.hi[hl + G * k2], a.freqs.lo[hl + G * k2]);
    };
    bool ok = true;
    uint32_t rn = 0;
    // One-block units take the next unit and its angles from the queue while
    // their own S product runs (the epilogue's TMA stores leave that time
    // free), so that the next Q tile's RoPE follows the softmax directly.
    UnitInfo ui;
    int u = ONE ? read_unit(rn, true, &ui) : 0;
    float2 cs_own[32 / G];
    if (ONE && u >= 0) angles(ui, cs_own);
    while (true) {
      if constexpr (!ONE) u = read_unit(rn, true);
      if (u < 0) {
        ok = !*abort;
        break;
      }
      if constexpr (!ONE) {
        unit_info<G, BN, WIN, (C::TOFF > 0)>(u, a, cu, nut, ui);
        angles(ui, cs_own);
      }
      const int qmin = ui.P + ui.t0 + t * TQ;    // position of the tile's first token
      const int qpos = qmin + tl;
      const int qidx = qpos - ui.P;              // this row's index among the new tokens
      // RoPE of this row's dims 0..63 (box 0, 128-byte row, 16-byte chunks
      // swizzled by row % 8): pairs (i, i + 32) live in chunks c and c + 4.
      {
        if (!warp_wait(&bars->q_full[t], uc & 1u, a.ctl, abort)) { ok = false; break; }
        uint8_t* qrow = smem + C::kOffQ + t * C::kQBytes + r * 128;
        uint4 ch[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) ch[c] = *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4));
        uint32_t big = 0u;  // |rotated| of every pair, as fp16 (inf once out of range)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t* x = reinterpret_cast<uint32_t*>(&ch[c]);
          uint32_t* y = reinterpret_cast<uint32_t*>(&ch[c + 4]);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int i = 8 * c + 2 * w;
            const float2 xv = unpack_bf16x2(x[w]);
            const float2 yv = unpack_bf16x2(y[w]);
            const float2 c0 = shared_cos_sin<G>(cs_own, i, lane);
            const float2 c1 = shared_cos_sin<G>(cs_own, i + 1, lane);
            const float a0 = xv.x * c0.x - yv.x * c0.y, a1 = xv.y * c1.x - yv.y * c1.y;
            const float b0 = yv.x * c0.x + xv.x * c0.y, b1 = yv.y * c1.x + xv.y * c1.y;
            x[w] = pack_f16x2(a0, a1);  // rotated dims are fp16 operands
            y[w] = pack_f16x2(b0, b1);
            big = f16x2_absmax3(big, x[w], y[w]);
          }
        }
        if (f16x2_any_inf(big)) record_status(a.ctl, HATTN_ERR_INVALID_ARG);
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(qrow + ((c ^ (r & 7)) << 4)) = ch[c];
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_ready[t]);
      }
      if (have_prev && !epilogue()) { ok = false; break; }
      const int h = ui.g * G + hl;
      const float sink_l2 = __ldg(a.sink + h) * kLog2e;
      float m = -INFINITY;  // running max (log2 units); the sink joins at the end
      float l = 0.f;
      const int qmax = qmin + TQ - 1;
      UnitInfo nui;
      int nu = -1;
      float2 ncs[32 / G];
      if constexpr (ONE) {
        nu = read_unit(rn, true, &nui);
        if (nu >= 0) angles(nui, ncs);
        if (!warp_wait(&bars->s_full[t], blk & 1u, a.ctl, abort)) { ok = false; break; }
        tc_fence_after();
        const int kb = ui.kstart + t * C::TOFF;  // position of column 0 (may be < 0)
        // the window's far edge, and position 0 where the band starts before it
        const int lo = max(qpos - a.window + 1, 0), lo_max = max(qmax - a.window + 1, 0);
        softmax_one<C::NT>(t_s, a.scale_log2, lo - kb, qpos - kb, lo_max - kb, qmin - kb, m, l);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
        ++blk;
      } else
      for (int j = 0; j < ui.nblk; ++j, ++blk) {
        if (!warp_wait(&bars->s_full[t], blk & 1u, a.ctl, abort)) { ok = false; break; }
        // S_B of this block is done, and S_A before it: K_j's stage is free
        // (the blk-th K block of this CTA)
        if (t == 1 && r == 0) mbar_arrive(&bars->kv_empty[blk % C::KST]);
        tc_fence_after();
        const int kb = ui.kstart + j * BN;  // position of column 0
        uint32_t s[BN];
        load_s_row<BN>(t_s, s);
        // masks where a row of the tile loses columns to the causal edge
        // (upper) or, with a window, to the window's far edge (lower)
        const bool upper = kb + BN - 1 > qmin;
        const bool lower = WIN && kb < qmax - a.window + 1;
        mask_block<BN>(s, lower, upper, qpos - a.window + 1 - kb, qpos - kb);
        softmax_block<BN>(s, a.scale_log2, t_s, t_o, j > 0, m, l);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
        // a unit's last block has no K_{j+1}: one softmax thread arrives in
        // its place
        if (t == 0 && r == 0 && j + 1 == ui.nblk) mbar_arrive(&bars->p_full[0]);
      }
      if (!ok) break;
      have_prev = true;
      pm = m;
      pl = l;
      psink = sink_l2;
      pvalid = qidx < ui.L;
      porow = long(ui.tok0 + qidx) * a.hq + h;
      ptok = ui.tok0 + ui.t0 + t * TQ;
      pgh = ui.g * G;
      pfull = ui.t0 + (t + 1) * TQ <= ui.L;
      puc = uc;
      ++uc;
      if constexpr (ONE) {
        u = nu;
        ui = nui;
#pragma unroll
        for (int k2 = 0; k2 < 32 / G; ++k2) cs_own[k2] = ncs[k2];
      }
    }
    if (ok && have_prev) epilogue();
    // the TMA stores of O complete before the CTA's shared memory goes
    if (ONE && r == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int G, int BN, bool WIN, bool ONE>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  using C = Cfg<G, BN, ONE>;
  CUtensorMap mq, mk0, mk12, mv, mo;
  const bool cached = a.prefix != nullptr;
  // packed: rotated dims [total_k, hkv, 64] and raw keys [total_k, hkv, 192];
  // cached: both from the cache [batch * hkv, cap, 192]
  const long kr = a.total_k > 0 ? a.total_k : a.total;
  if (!make_map(&mq, a.q, a.total, a.hq, kDqk, G, C::TQ) ||
      !(cached ? make_map(&mk0, a.k_rot, long(a.batch) * a.hkv, a.cap, kDqk, BN, 1)
               : make_map(&mk0, a.k_rot, kr, a.hkv, kRopeDim, 1, BN)) ||
      !(cached ? make_map(&mk12, a.k_raw, long(a.batch) * a.hkv, a.cap, kDqk, BN, 1)
               : make_map(&mk12, a.k_raw, kr, a.hkv, kDqk, 1, BN)) ||
      !(cached ? make_map(&mv, a.v, long(a.batch) * a.hkv, a.cap, kDv, BN, 1)
               : make_map(&mv, a.v, kr, a.hkv, kDv, 1, BN)))
    return cudaErrorInvalidValue;
  PrefillArgs a2 = a;
  // O by TMA stores where the output's layout allows a map (16-byte base)
  a2.o_tma = ONE && make_out_map(&mo, a.out, a.total, a.hq, G, C::TQ);
  if (!a2.o_tma) mo = mq;  // unused
  auto kern = prefill_kernel<G, BN, WIN, ONE>;
  static bool attr_set = false;
  if (!attr_set) {
    // The register split inside the kernel needs the launch to allocate
    // kRegsLaunch registers per thread; anything less would stall it.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long nut = (a.max_seqlen + C::UT - 1) / C::UT;
  const long nunits = nut * a.batch * a.hkv;
  if (nunits == 0) return cudaSuccess;
  const int grid = int(nunits < num_sms() ? nunits : num_sms());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = a.after_pass ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk0, mk12, mv, mo, a2);
}

// Key blocks: a window unit whose band (W - 1 + 2*TQ keys) fits one block
// of 144 (G = 16) or 160 (G = 8) keys runs as one block; other window units
// use blocks of 80 when the band fits two of them, else 128; global units
// use 128.
template <int G>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t s) {
  const int band = a.window - 1 + 256 / G;
  if (a.window == 0) return launch_t<G, 128, false, false>(a, s);
  if constexpr (G == 16) {
    if (band <= 144) return launch_t<G, 144, true, true>(a, s);
  }
  if constexpr (G == 8) {
    if (band <= 160) return launch_t<G, 160, true, true>(a, s);
  }
  if (band <= 160) return launch_t<G, 80, true, false>(a, s);
  return launch_t<G, 128, true, false>(a, s);
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
