/*
 * hattn.h -- C ABI of the hybrid sliding-window / global sink-attention
 * library (libhattn.so, NVIDIA B300, sm_103a).
 *
 * What the library computes (one attention layer's forward pass):
 *
 *   MiMo-V2-Flash Technical Report paper review (xllm-io), section 3.1
 *   "overall structure": causal GQA attention, 64 query heads over 8 KV heads
 *   in sliding-window (SWA) layers and over 4 KV heads in global (GA)
 *   layers, Q/K head dim 192, V head dim 128, RoPE on the first 64 dims,
 *   window W = 128, SWA and GA layers interleaved 5:1.
 *   Same page, section 4: RoPE base 10K for SWA layers, 5M for GA layers.
 *   Same page, section 3.2, and the plmsmile notes on the MiMo series,
 *   MiMo-V2-Flash "Learnable Attention Sink": each query head h has a
 *   learnable logit s_h whose exp(s_h) joins the softmax denominator:
 *
 *     out[p,h] = sum_{j in J(p)} exp(z_pj - m) v_j / Z,
 *     Z = sum_{j in J(p)} exp(z_pj - m) + exp(s_h - m),
 *     lse[p,h] = m + ln Z   (natural log; the sink is included),
 *     z_pj = scale * <RoPE(q_p, p), RoPE(k_j, j)>,
 *     J(p) = { j : j <= p and (window == 0 or p - j < window) }.
 *
 *   plmsmile notes, MiMo-V2-Flash "local window": SWA layers keep a KV cache
 *   that does not grow with the history (here a ring buffer); GA layers keep
 *   a growing cache.  Same notes, MTP: drafted tokens are verified by the
 *   main model in one parallel pass (here: 1 to 4 query tokens per sequence).
 *
 * Readings (the pages leave these open): the window holds W keys including
 * the query itself; the sink is a raw logit, one fp32 per query head; query
 * head h reads KV head h / (hq / hkv); RoPE turns the pairs (i, i + 32),
 * i < 32, by pos * base^(-i / 32) ("rotate-half").
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous, 16-byte aligned.  bf16 is IEEE bfloat16 (uint16 bits).
 *   - `stream` is a cudaStream_t (passed as void*); NULL = legacy default
 *     stream.  Calls are asynchronous on that stream; the library does not
 *     synchronise except in hattn_check_device_status().
 *   - The library allocates no device memory.  Scratch space is a caller
 *     buffer ("workspace") whose size the *_workspace_size() functions give.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-HATTN_OK status means nothing was launched (except HATTN_ERR_CUDA,
 *     reported when a launch itself fails).  Nothing throws across the ABI.
 *   - Supported shapes: dqk = 192, dv = 128, rope_dim = 64, hq % hkv == 0 and
 *     G = hq / hkv in {1, 2, 4, 8, 16}.  Others return HATTN_ERR_UNSUPPORTED.
 *   - Kernels never trap.  Device-side failures (a bounded wait that ran out)
 *     are recorded in a device status word read by
 *     hattn_check_device_status().
 */
#ifndef HATTN_H_
#define HATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HATTN_OK = 0,
  HATTN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment */
  HATTN_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shape set */
  HATTN_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed */
  HATTN_ERR_RING_TOO_SMALL = 4,/* ring cache cap < window + T - 1 */
  HATTN_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out */
  HATTN_ERR_WORKSPACE = 6      /* workspace missing or smaller than required */
} hattn_status_t;

/* Library version (major * 10000 + minor * 100 + patch). */
int hattn_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* hattn_status_string(hattn_status_t status);

/*
 * Bytes of workspace hattn_prefill() needs: the keys' rotated dims 0..63,
 * total_tokens * hkv * 64 fp16 values, rounded up to 256 bytes, then 256
 * bytes for the attention kernel's work counter (both rewritten by every
 * call: a workspace serves one call at a time).  dqk must be 192.
 */
size_t hattn_prefill_workspace_size(long total_tokens, int hkv, int dqk);

/*
 * Prefill: one attention layer over packed variable-length sequences (a
 * hybrid block is five window layers and one global layer, called in turn).
 *
 *   q          bf16 [total_tokens, hq, dqk]   un-rotated queries
 *   k          bf16 [total_tokens, hkv, dqk]  un-rotated keys
 *   v          bf16 [total_tokens, hkv, dv]
 *   sink       fp32 [hq]                      sink logits s_h
 *   out        bf16 [total_tokens, hq, dv]    written
 *   lse        fp32 [total_tokens, hq]        written (may be NULL)
 *   batch      number of sequences (>= 1)
 *   cu_seqlens int32 [batch + 1] DEVICE; cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[batch] = total_tokens.  RoPE positions restart at 0
 *              in every sequence.  The offsets are device memory the host
 *              cannot read: the kernels check them, and a sequence whose rows
 *              [cu_seqlens[b], cu_seqlens[b+1]) are not inside
 *              [0, total_tokens) or number more than max_seqlen is skipped --
 *              none of its out / lse rows is written -- and
 *              HATTN_ERR_INVALID_ARG is recorded in the device status.
 *   max_seqlen an upper bound of every sequence length (sizes the grid)
 *   window     > 0: sliding window of `window` keys including the query;
 *              0: global causal attention
 *   rope_base  RoPE base (1e4 for SWA layers, 5e6 for GA layers)
 *   softmax_scale  logit scale (1/sqrt(192) for this model)
 *   workspace  DEVICE scratch of >= hattn_prefill_workspace_size() bytes,
 *              overwritten with the keys' rotated dims 0..63 as fp16
 *              [total_tokens, hkv, 64] (dims 64..191 are read from k);
 *              out and lse must not overlap q, k, v or it.
 * Queries and keys are rotated before the tensor-core products; the rotated
 * dims are carried as fp16 (see hattn_rope_kv_append), so |RoPE(x)| must stay
 * below 65504 on dims 0..63 (recorded as HATTN_ERR_INVALID_ARG otherwise).
 */
hattn_status_t hattn_prefill(const void* q, const void* k, const void* v, const float* sink,
                             void* out, float* lse, int batch, const int* cu_seqlens,
                             long total_tokens, int max_seqlen, int hq, int hkv, int dqk, int dv,
                             int rope_dim, float rope_base, int window, float softmax_scale,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * One shard of a layer's prefill under context parallelism: a sequence is cut
 * into consecutive shards, one per GPU, and shard r holds its tokens
 * [pos0, pos0 + shard_tokens).  A query at position p of a window layer sees
 * keys p - window + 1 .. p, so besides its own keys a shard needs only the
 * last min(window - 1, pos0) keys before it -- the halo -- which an exchange
 * step brings from the GPUs that hold them (plmsmile notes on the MiMo
 * series, MiMo-V2.6, "DFlash and long-context system optimisation", training
 * memory: SWA context parallelism exchanges only the window-reachable KV).
 * A global layer (window 0) needs the whole history as its halo.  Same
 * results as rows [pos0, pos0 + shard_tokens) of hattn_prefill() over the
 * whole sequence.
 *
 *   q      bf16 [shard_tokens, hq, dqk]   the shard's queries, un-rotated
 *   k      bf16 [halo + shard_tokens, hkv, dqk]: the halo's keys (positions
 *          pos0 - halo .. pos0 - 1) followed by the shard's own, un-rotated
 *   v      bf16 [halo + shard_tokens, hkv, dv], the same rows
 *   out    bf16 [shard_tokens, hq, dv], lse fp32 [shard_tokens, hq] (or NULL)
 *   halo   rows of k and v before the shard's own: at least
 *          min(window - 1, pos0) for window > 0, exactly pos0 for window = 0,
 *          and at most pos0 (else HATTN_ERR_INVALID_ARG)
 *   pos0   absolute position of the shard's first token (RoPE positions are
 *          absolute: the halo's keys rotate at pos0 - halo ..)
 *   workspace  DEVICE scratch of >= hattn_prefill_workspace_size(halo +
 *          shard_tokens, hkv, dqk) bytes
 *   other arguments as for hattn_prefill().
 */
hattn_status_t hattn_prefill_shard(const void* q, const void* k, const void* v,
                                   const float* sink, void* out, float* lse, long shard_tokens,
                                   int halo, long pos0, int hq, int hkv, int dqk, int dv,
                                   int rope_dim, float rope_base, int window, float softmax_scale,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace hattn_prefill_backward() needs: the rotated dims 0..63 of
 * q and k (total_tokens * (hq + hkv) * 64 bf16 values), delta = dout . out
 * (total_tokens * hq floats) and the sink-gradient partials of the prep pass
 * (ceil(total_tokens / 32) * hq floats), each rounded up to 256 bytes.  All of
 * it is rewritten by every call: a workspace serves one call at a time.
 */
size_t hattn_prefill_backward_workspace_size(long total_tokens, int hq, int hkv);

/*
 * Backward of hattn_prefill(): the gradients of sum(dout * out) with respect
 * to q, k, v and the sink logits (the sink is a learnable per-head parameter:
 * MiMo-V2-Flash paper review, section 3.2).  With p_j = exp(z_j - lse), the
 * forward's weights, and delta = dout . out per row:
 *   dv_j = sum over rows of p_j dout;   dz_j = p_j (dout . v_j - delta);
 *   dq = R^T scale sum_j dz_j k'_j;     dk_j = R^T scale sum over rows of dz_j q';
 *   dsink_h = -sum over rows of head h of exp(sink_h - lse) delta,
 * R the row's RoPE rotation (dims 0..63), q', k' the rotated vectors.
 *
 *   q, k, v, sink  the forward's inputs (same layouts as hattn_prefill())
 *   out        bf16 [total_tokens, hq, dv]  the forward's output
 *   lse        fp32 [total_tokens, hq]      the forward's lse (required)
 *   dout       bf16 [total_tokens, hq, dv]  gradient of the loss w.r.t. out
 *   grad_q     bf16 [total_tokens, hq, dqk]  written
 *   grad_k     bf16 [total_tokens, hkv, dqk] written (summed over the G query
 *              heads of each KV head)
 *   grad_v     bf16 [total_tokens, hkv, dv]  written
 *   grad_sink  fp32 [hq] DEVICE, written (summed over every row of the head)
 *   workspace  DEVICE scratch of >= hattn_prefill_backward_workspace_size()
 *   other arguments as for hattn_prefill() (a sequence whose offsets fail the
 *   device-side check is skipped: none of its gradient rows is written).
 *   Outputs must not overlap inputs or the workspace.  Every gradient row is written by one thread and no
 *   atomics are used: the results are the same on every run.  The products
 *   take bf16 operands (P, dS and the rotated dims rounded to bf16) with fp32
 *   accumulation.
 */
hattn_status_t hattn_prefill_backward(const void* q, const void* k, const void* v,
                                      const float* sink, const void* out, const float* lse,
                                      const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                      float* grad_sink, int batch, const int* cu_seqlens,
                                      long total_tokens, int max_seqlen, int hq, int hkv, int dqk,
                                      int dv, int rope_dim, float rope_base, int window,
                                      float softmax_scale, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Rotate new keys and write them and their values into the KV cache.
 *
 *   k_new     bf16 [B, T, hkv, dqk]   un-rotated keys of the T new tokens
 *   v_new     bf16 [B, T, hkv, dv]
 *   start_pos int32 [B] DEVICE: position of token 0 of sequence b (>= 0)
 *   k_cache   [B, hkv, cap, dqk] rotated keys, updated in place: dims 0..63
 *             (the rotated ones) as IEEE fp16, dims 64..191 as bf16.  fp16
 *             keeps 11 significant bits of the rotated values (bf16 keeps 8),
 *             which holds the log-sum-exp error near 3e-4; a rotated value
 *             beyond +-65504 is recorded as HATTN_ERR_INVALID_ARG in the
 *             device status.
 *   v_cache   bf16 [B, hkv, cap, dv]  updated in place
 *   is_ring   1: slot = pos % cap (fixed-size SWA cache);
 *             0: slot = pos (growing GA cache); a position >= cap is skipped
 *             and recorded as HATTN_ERR_INVALID_ARG in the device status.
 *   T         1..cap tokens per sequence
 */
hattn_status_t hattn_rope_kv_append(const void* k_new, const void* v_new, const int* start_pos,
                                    void* k_cache, void* v_cache, int B, int T, int hkv, int dqk,
                                    int dv, int cap, int is_ring, int rope_dim, float rope_base,
                                    void* stream);

/*
 * Prefill over a cached prefix (prefix-cache reuse, chunked prefill): the new
 * tokens of each sequence continue a history already held in a linear cache.
 * Their keys (rotated) and values are appended to the caches, then each new
 * token attends causally (within the window, if any) over the whole cache.
 * Same results as hattn_rope_kv_append() of the new tokens at positions
 * prefix_lens[b] + t followed by attention over all prefix_lens[b] + L_b
 * keys.  MiMo-V2-Flash paper review, section 5.6 (prefix cache and rollout);
 * plmsmile notes, MiMo-V2-Flash (partial rollouts re-prefilled).
 *
 *   q           bf16 [total_tokens, hq, dqk]  the new tokens' queries, un-rotated, packed
 *   k_new, v_new  bf16 [total_tokens, hkv, dqk] / [total_tokens, hkv, dv], packed
 *   k_cache, v_cache  [batch, hkv, cap, dqk|dv] linear (slot = position): slots
 *               [0, prefix_lens[b]) hold the prefix as hattn_rope_kv_append()
 *               writes it; the new tokens are written at [prefix, prefix + L_b),
 *               and V slots [prefix + L_b, prefix + L_b + 256) are zeroed (they
 *               hold no token yet)
 *   cu_seqlens  int32 [batch + 1] DEVICE, as for hattn_prefill(): the new tokens
 *   prefix_lens int32 [batch] DEVICE: tokens already in the caches, >= 0
 *   out, lse    as for hattn_prefill(), one row per new token
 *   max_seqlen  upper bound of the new tokens per sequence; max_prefix upper
 *               bound of prefix_lens; prefix_lens[b] + L_b <= cap
 *   workspace   DEVICE scratch of >= 256 bytes (the kernel's work counter)
 *   other arguments as for hattn_prefill().
 * A position outside [0, cap) is skipped and recorded as HATTN_ERR_INVALID_ARG;
 * the attention skips a sequence whose offsets fail hattn_prefill()'s check or
 * whose prefix_lens[b] + L_b leaves [0, cap] (its out / lse rows are not written).
 */
hattn_status_t hattn_prefill_cached(const void* q, const void* k_new, const void* v_new,
                                    void* k_cache, void* v_cache, const int* cu_seqlens,
                                    const int* prefix_lens, const float* sink, void* out,
                                    float* lse, int batch, long total_tokens, int max_seqlen,
                                    int max_prefix, int cap, int hq, int hkv, int dqk, int dv,
                                    int rope_dim, float rope_base, int window,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * Bytes of workspace hattn_decode() needs for a batch whose longest
 * sequence holds max_seqlen_k tokens, with the same cap, is_ring and window
 * as the hattn_decode() call (0 when one pass per KV head suffices: a
 * window or ring of at most 1024 keys).  A linear cache is cut into chunks
 * of 2048 keys (4096 beyond 16K keys); a ring into chunks of its cap slots.
 * The workspace holds the chunks' partial O and lse and 256 bytes for the
 * kernel's work counter (zeroed by every call: a workspace serves one call
 * at a time).
 */
size_t hattn_decode_workspace_size(int B, int T, int hq, int hkv, int dv, int max_seqlen_k,
                                   int window, int cap, int is_ring);

/*
 * Decode / MTP-verify step: the last T tokens of
 * every sequence (positions seqlens_k[b] - T + t) attend over the cache,
 * which must already hold them (call hattn_rope_kv_append() first).
 *
 *   q          bf16 [B, T, hq, dqk]    un-rotated queries
 *   k_cache    [B, hkv, cap, dqk] rotated keys as written by
 *              hattn_rope_kv_append() (dims 0..63 fp16, 64..191 bf16)
 *   v_cache    bf16 [B, hkv, cap, dv]
 *   seqlens_k  int32 [B] DEVICE: tokens of sequence b including the T new
 *              ones; T <= seqlens_k[b] <= max_seqlen_k, and for a linear
 *              cache seqlens_k[b] <= cap.
 *   sink       fp32 [hq]
 *   out        bf16 [B, T, hq, dv]     written
 *   lse        fp32 [B, T, hq]         written (may be NULL)
 *   T          1..8 query tokens per sequence, with (hq / hkv) * T <= 128
 *              (else HATTN_ERR_UNSUPPORTED)
 *   is_ring    1: key j lives in slot j % cap and cap >= window + T - 1 is
 *              required (else HATTN_ERR_RING_TOO_SMALL); needs window > 0.
 *              0: key j lives in slot j.
 *   workspace  DEVICE scratch of >= hattn_decode_workspace_size() bytes
 *              (may be NULL when that size is 0).
 */
hattn_status_t hattn_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int* seqlens_k, const float* sink, void* out, float* lse, int B,
                            int T, int hq, int hkv, int dqk, int dv, int cap, int is_ring,
                            int window, int max_seqlen_k, int rope_dim, float rope_base,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Size of the fixed device array hattn_decode_static_scratch() uses as its
 * scratch (32 MiB): enough for B * hq * T * chunks <= 65,000 partial rows of
 * 516 bytes, chunks = ceil(keys / 2048) up to 16K keys, ceil(keys / 4096)
 * beyond -- e.g. batch 8 x 64 heads x 4 tokens over up to 64K keys (32,768
 * rows).  A window layer whose ring fits in one chunk needs no scratch at all.
 */
#define HATTN_DECODE_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * One whole decode / MTP-verify step of a layer: the append of the T new
 * tokens (hattn_rope_kv_append() at positions seqlens_k[b] - T + t) and the
 * attention of hattn_decode() over the cache that then holds them, with the
 * same results as those two calls in that order (cache contents included).
 * MiMo-V2-Flash paper review, section 3.1 (hybrid layers, fixed window
 * cache); plmsmile notes, MiMo-V2-Flash "local window" (the window layer's
 * cache is a fixed ring).
 *
 *   k_new, v_new  bf16 [B, T, hkv, dqk] / [B, T, hkv, dv]: the new tokens'
 *                 un-rotated keys and their values
 *   k_cache, v_cache  written in the T new tokens' slots, then read
 *   every other argument as for hattn_decode()
 *
 * For a ring of at most 144 slots with at most 32 query rows per KV head
 * (T <= 4, G * T <= 32, G in {1, 2, 4, 8}) the append runs inside the attention
 * kernel: one launch per step.  Otherwise the append kernel runs first, on
 * the same stream.  Errors as for the two calls; a sequence whose length
 * fails the checks is neither appended nor attended (its output rows are
 * not written) and HATTN_ERR_INVALID_ARG is recorded.
 */
hattn_status_t hattn_decode_append(const void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, const int* seqlens_k,
                                   const float* sink, void* out, float* lse, int B, int T, int hq,
                                   int hkv, int dqk, int dv, int cap, int is_ring, int window,
                                   int max_seqlen_k, int rope_dim, float rope_base,
                                   float softmax_scale, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * hattn_decode_append() over paged caches: position p of sequence b lives in
 * page block_table[b * table_stride + p / page], slot p % page.
 *
 *   k_pages, v_pages  [num_pages, hkv, page, dqk|dv]: K stored as
 *               hattn_rope_kv_append() writes it (dims 0..63 fp16, rest bf16),
 *               V bf16; the new tokens are written into their pages
 *   block_table int32 [B, table_stride] DEVICE: page of each run of `page`
 *               positions; entries past a sequence's last position are not read
 *   page        positions per page, a multiple of 64
 *   every other argument as for hattn_decode_append() with is_ring = 0 and
 *   cap = table_stride * page (so max_seqlen_k <= table_stride * page).
 * A page index outside [0, num_pages) is recorded as HATTN_ERR_INVALID_ARG and
 * reads as zeros (it is never written).  The workspace is that of
 * hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window,
 * table_stride * page, 0).
 */
hattn_status_t hattn_decode_append_paged(const void* q, const void* k_new, const void* v_new,
                                         void* k_pages, void* v_pages, const int* block_table,
                                         int table_stride, int num_pages, int page,
                                         const int* seqlens_k, const float* sink, void* out,
                                         float* lse, int B, int T, int hq, int hkv, int dqk,
                                         int dv, int window, int max_seqlen_k, int rope_dim,
                                         float rope_base, float softmax_scale, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * hattn_decode() for callers that cannot allocate device memory.  The paper
 * has no counterpart to this entry point; it exists for callers that cannot
 * call cudaMalloc -- code running inside a host framework that owns all
 * device memory through its own pool and forbids side allocations, or a
 * serving loop whose memory budget is fixed at start-up -- and so cannot
 * provide hattn_decode()'s workspace.
 *
 * Same arguments and results as hattn_decode() minus the workspace; the
 * scratch is a fixed array of HATTN_DECODE_STATIC_SCRATCH_BYTES inside the
 * library, held on every GPU that loads the library until the process exits.
 *   - Allocates nothing: no cudaMalloc / cudaFree, no allocating library call.
 *   - A step whose scratch need (hattn_decode_workspace_size()) exceeds that
 *     size returns HATTN_ERR_WORKSPACE and launches nothing.
 *   - Arguments are checked as hattn_decode() checks them (same status
 *     codes) before the scratch need is compared with the array's size.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  A failed lookup returns HATTN_ERR_CUDA.
 *     The address is kept until the process exits; it belongs to the
 *     device's context, so after cudaDeviceReset() on that device this entry
 *     point must not be called there again (the same holds for every entry
 *     point: the device status word's address is cached the same way).
 *   - Every call shares the one array per device and it keeps the last
 *     call's contents.  Nothing in it needs to start at zero: every partial
 *     result is written before it is read.  Calls that overlap on the GPU
 *     (on different streams, or from several host threads) race on it and
 *     must be serialised by the caller.
 */
hattn_status_t hattn_decode_static_scratch(const void* q, const void* k_cache,
                                           const void* v_cache, const int* seqlens_k,
                                           const float* sink, void* out, float* lse, int B,
                                           int T, int hq, int hkv, int dqk, int dv, int cap,
                                           int is_ring, int window, int max_seqlen_k,
                                           int rope_dim, float rope_base, float softmax_scale,
                                           void* stream);

/*
 * Synchronise `stream`, then report (and clear) the device status word:
 * HATTN_OK, HATTN_ERR_TIMEOUT (a bounded wait inside a kernel ran out) or
 * HATTN_ERR_INVALID_ARG (a device-side index check skipped an access), or
 * HATTN_ERR_CUDA if the synchronisation itself failed.
 */
hattn_status_t hattn_check_device_status(void* stream);

/*
 * Set how long (nanoseconds) any single device-side wait may last before the
 * kernel gives up with HATTN_ERR_TIMEOUT (default 2e9 = 2 s; 0 restores the
 * default).  Applies to launches made after the call on the current device.
 */
hattn_status_t hattn_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Self-test of the failure path: launches one CTA that waits on an mbarrier
 * nothing ever arrives at, bounded by the current wait limit.  The kernel
 * returns normally; hattn_check_device_status() then reports
 * HATTN_ERR_TIMEOUT.  Nothing faults, traps or hangs.
 */
hattn_status_t hattn_selftest_lost_arrival(void* stream);

/*
 * Test hook, host-side fault injection: the next n calls that would launch
 * kernels (after their argument checks pass) return HATTN_ERR_CUDA without
 * touching the device, as a failed launch would, so a caller's error handling
 * can be exercised without faulting a GPU.  n <= 0 clears it.  Returns the
 * number of injected failures that were still pending.  Process-wide,
 * thread-safe; calls rejected by their argument checks do not consume one.
 */
int hattn_test_fail_next_launches(int n);

#ifdef __cplusplus
}
#endif

#endif /* HATTN_H_ */
