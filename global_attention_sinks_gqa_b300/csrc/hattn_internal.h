// hattn_internal.h -- declarations shared between the C-ABI layer and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hattn.h"

namespace hattn {

constexpr int kDqk = 192;
constexpr int kDv = 128;
constexpr int kRopeDim = 64;
constexpr int kRopeHalf = 32;

// Where kernels report failures, and how long a device-side wait may last.
struct DeviceCtl {
  unsigned int* status;          // device address of the status word
  unsigned long long wait_limit_ns;
};

// theta_i / (2 pi) for the 32 RoPE frequencies as double-float pairs.
struct RopeFreqs {
  float hi[kRopeHalf];
  float lo[kRopeHalf];
};

void make_rope_freqs(float base, RopeFreqs* f);

// ---- host helpers (prefill_tc.cu) -------------------------------------------
// 3-D TMA map over a [rows, heads, dim] bf16 tensor: 64-element (128-byte)
// inner box of box_heads x box_rows, 128-byte swizzle, out-of-range rows read
// as zero.  False if the driver entry point is missing or encoding fails.
bool make_map(CUtensorMap* m, const void* base, long rows, int heads, int dim, int box_heads,
              int box_rows);
// Number of SMs of the current device.
int num_sms();

// ---- rope / append (rope_append.cu) --------------------------------------
// The rotated dims 0..63 of every key row, as fp16, into k_rot [total, hkv,
// 64].  Also zeroes *unit_ctr (the prefill kernel's work counter) when non-null.
// cu_seqlens == nullptr: one sequence whose row n sits at position n + pos_off.
cudaError_t launch_rope_keys_packed(const void* k, void* k_rot, const int* cu_seqlens, int batch,
                                    long total, int hkv, const RopeFreqs& f, const DeviceCtl& ctl,
                                    cudaStream_t s, unsigned int* unit_ctr = nullptr,
                                    int pos_off = 0);
// A paged cache: position p of sequence b lives in page
// table[b * stride + p / page], slot p % page; pages are [num_pages, hkv,
// page, d].  table == nullptr: a contiguous cache [B, hkv, cap, d].
struct Paging {
  const int* table = nullptr;
  int stride = 0, page = 0, num_pages = 0;
};

// Token t of sequence b goes to position start_pos[b] + t, or, with
// from_len, to seqlens[b] - T + t (start_pos then holds seqlens).
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int* start_pos,
                             void* k_cache, void* v_cache, int B, int T, int hkv, int cap,
                             int is_ring, const RopeFreqs& f, const DeviceCtl& ctl,
                             cudaStream_t s, bool from_len = false, Paging pg = Paging());

// Packed new tokens of sequence b to slots prefix[b] + t of a linear cache;
// also zeroes V slots [end, end + 256) past each sequence's new end and
// *unit_ctr (see rope_append.cu).
cudaError_t launch_kv_append_packed(const void* k_new, const void* v_new, const int* cu_seqlens,
                                    const int* prefix, void* k_cache, void* v_cache, int batch,
                                    long total, int hkv, int cap, const RopeFreqs& f,
                                    const DeviceCtl& ctl, unsigned int* unit_ctr, cudaStream_t s);

// ---- prefill (prefill_tc.cu) ------------------------------------------------
struct PrefillArgs {
  const void* q;
  const void* k_rot;   // rotated dims 0..63: [total, hkv, 64] fp16, or the K cache
  const void* k_raw;   // dims 64..191: the un-rotated keys [total, hkv, 192], or the K cache
  unsigned int* unit_ctr;  // work counter (zeroed by the key rotation pass)
  const void* v;
  const float* sink;
  void* out;
  float* lse;
  const int* cu_seqlens;
  int batch;
  long total;
  int max_seqlen;
  int hq, hkv;
  int window;
  float scale_log2;  // softmax_scale * log2(e)
  RopeFreqs freqs;
  DeviceCtl ctl;
  // Prefill over a cached prefix (hattn_prefill_cached): sequence b's new
  // tokens sit at positions prefix[b]..; keys and values are read from the
  // caches [batch, hkv, cap, d] (k_rot, v point at them), slot = position.
  const int* prefix = nullptr;
  int cap = 0;
  // One shard of a sequence (hattn_prefill_shard; batch 1, cu_seqlens null):
  // the packed K/V hold total_k = lead + total rows, the `lead` rows of keys
  // before the shard's first query followed by the shard's own; RoPE
  // positions are the rows' indices plus rope_off.
  long total_k = 0;  // 0: total
  int lead = 0;
  int rope_off = 0;
  // The kernel just before on the stream is this call's key-rotation pass
  // or append (itself launched in stream order), which writes only the
  // rotated keys / caches, the work counter and the status word: the
  // attention kernel may then start before it ends (programmatic dependent
  // launch) and waits for it only before reading those.
  bool after_pass = false;
  bool o_tma = false;  // set by the launcher: O may leave by TMA stores
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

// ---- decode (decode.cu) -----------------------------------------------------
struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* seqlens;
  const float* sink;
  void* out;
  float* lse;
  int B, T, hq, hkv, cap, is_ring, window, max_seqlen_k;
  float scale_log2;
  RopeFreqs freqs;
  float* part_o;    // [B, hq, T, nsplit, dv] fp32 (nsplit > 1 only)
  float* part_lse;  // [B, hq, T, nsplit] fp32, log2 domain
  int nsplit;
  int chunk;        // keys per split
  // Append fused into the step (hattn_decode_append): the T new tokens' K
  // (un-rotated) and V, written into the caches before they are read.
  // nullptr: the caches already hold them.
  unsigned int* item_ctr = nullptr;  // work counter in the workspace (nsplit > 1)
  Paging pg;                         // paged caches (linear positions, cap = stride * page)
  const void* k_new = nullptr;  // bf16 [B, T, hkv, dqk]
  const void* v_new = nullptr;  // bf16 [B, T, hkv, dv]
  DeviceCtl ctl;
};
int decode_num_splits(int max_seqlen_k, int T, int window, int is_ring, int cap, int* chunk);
// The argument checks of hattn_decode() / hattn_decode_append() (all but the
// workspace; hattn_api.cu).  *empty: nothing to launch (B == 0).
hattn_status_t decode_check_args(const void* q, const void* k_new, const void* v_new,
                                 const void* k_cache, const void* v_cache, const int* seqlens_k,
                                 const float* sink, const void* out, const float* lse, int B,
                                 int T, int hq, int hkv, int dqk, int dv, int cap, int is_ring,
                                 int window, int max_seqlen_k, int rope_dim, float rope_base,
                                 float softmax_scale, bool* empty);
size_t decode_workspace_bytes(int B, int T, int hq, int nsplit);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// ---- backward of the prefill (backward.cu) ---------------------------------
struct BackwardArgs {
  const void* q;      // bf16 [total, hq, dqk], un-rotated
  const void* k;      // bf16 [total, hkv, dqk], un-rotated
  const void* v;      // bf16 [total, hkv, dv]
  const float* sink;  // [hq]
  const void* out;    // bf16 [total, hq, dv], the forward's output
  const float* lse;   // [total, hq], the forward's lse (natural log, sink included)
  const void* dout;   // bf16 [total, hq, dv]
  void* dq;           // bf16 [total, hq, dqk]
  void* dk;           // bf16 [total, hkv, dqk]
  void* dv;           // bf16 [total, hkv, dv]
  float* dsink;       // [hq]
  const int* cu_seqlens;
  int batch;
  long total;
  int max_seqlen;
  int hq, hkv, window;
  float scale, scale_log2;
  RopeFreqs freqs;
  DeviceCtl ctl;
  // workspace
  void* q_rot;       // bf16 [total, hq, 64]: rotated dims of q
  void* k_rot;       // bf16 [total, hkv, 64]
  float* delta;      // [total, hq]: dout . out
  float* sink_part;  // [nprep, hq]: sink-gradient partial sums of the prep blocks
  long nprep;
};
long backward_prep_blocks(long total);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);

// ---- status ------------------------------------------------------------------
cudaError_t launch_lost_arrival_selftest(const DeviceCtl& ctl, cudaStream_t s);

}  // namespace hattn
