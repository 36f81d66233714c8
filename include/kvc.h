/*
 * kvc.h — C ABI of libkvc: attention-score-driven KV-cache compression on GB300 (sm_103a).
 *
 * The library scores cached tokens by the softmax attention of an observation window of
 * recent queries, selects per KV head the tokens to keep (or evict), gather-compacts the
 * kept K/V rows, and runs the two variants defined on the same score pipeline: the
 * Scissorhands low-attention history and ThinK key-channel pruning.
 *
 * Conventions (every call):
 *  - Pointers named K, V, q_*, scores, idx, ... are DEVICE pointers owned by the caller.
 *    The library never allocates or frees device memory: callers size scratch buffers with
 *    kvc_workspace_size() and pass them as (ws, ws_bytes).  A workspace needs no initial
 *    content (some calls keep bookkeeping words in it that accept any prior bytes); calls
 *    that may run at the same time on the GPU must not share one.
 *  - bf16 tensors are passed as kvc_bf16 (the raw 16-bit pattern).  Scores are float32,
 *    indices int32.  Unless stated otherwise tensors are dense row-major with the shape in
 *    the comment; K/V caches are described by kvc_kv_desc and may be strided.
 *  - All compute is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *    Inputs must stay alive and unmodified until the stream reaches the call.
 *  - Arguments are validated on the host before anything is launched; on failure nothing is
 *    enqueued and an error status is returned (details: kvc_last_error_message()).
 *    No C++ exception crosses the ABI.  Device code never traps: an out-of-range index found
 *    on the device sets a sticky device status read by kvc_get_device_status().
 *  - Alignment: every device pointer must be 16-byte aligned; K/V strides must be multiples
 *    of 8 elements; the innermost (head_dim) stride is 1.
 *  - Outputs never alias inputs unless a call says so.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvc_bf16;                 /* bf16 bit pattern */
typedef struct CUstream_st* kvc_stream_t;  /* same type as cudaStream_t */

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment, aliasing or state */
  KVC_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim not 64/128) */
  KVC_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  KVC_ERR_TIMEOUT = 4,       /* a bounded device wait gave up */
  KVC_ERR_DEVICE_BOUNDS = 5, /* a kernel met an out-of-range index and skipped it */
  KVC_ERR_WORKSPACE = 6      /* ws is NULL or smaller than kvc_workspace_size() */
} kvc_status;

typedef enum {
  KVC_REDUCE_GQA_GROUP = 0, /* score[b,kvh,j] = sum_i mean_{h in group(kvh)} p[b,h,i,j] */
  KVC_REDUCE_ALL_HEADS = 1  /* score[b,*,j]   = sum_i mean_{all h} p[b,h,i,j], same for every kvh */
} kvc_head_reduce;

/* A K or V cache: element (b, kvh, s, d) lives at base + b*stride_b + kvh*stride_h + s*stride_s + d. */
typedef struct {
  int32_t B;        /* batch */
  int32_t H;        /* query heads (H % KVH == 0; the group of KV head kvh is h / (H/KVH) == kvh) */
  int32_t KVH;      /* key/value heads */
  int32_t D;        /* head_dim: 64 or 128 */
  int64_t S;        /* rows (tokens or slots) per (b, kvh) */
  int64_t stride_b; /* element strides */
  int64_t stride_h;
  int64_t stride_s;
} kvc_kv_desc;

typedef enum {
  KVC_OP_WINDOW_SCORES = 0,
  KVC_OP_TOPK_SELECT = 1,
  KVC_OP_COMPRESS_PREFILL = 2,
  KVC_OP_TOVA_DECODE_STEP = 3,
  KVC_OP_SCISSORHANDS_UPDATE = 4,
  KVC_OP_SCISSORHANDS_EVICT = 5,
  KVC_OP_CHANNEL_SCORE = 6,
  KVC_OP_DECODE_ATTENTION = 7,
  KVC_OP_VALUE_CHANNEL_SCORE = 8,
  KVC_OP_COMPRESS_PREFILL_CHANNELS = 9,
  KVC_OP_TOPK_COMPACT_CHANNELS = 10
} kvc_op;

/* Bytes of scratch the call `op` needs for these shapes on the current device (w: window
 * rows; k: kept tokens; unused arguments may be 0).  Returns 0 for ops that need none and
 * (size_t)-1 for invalid shapes.  The value depends on the device's SM count. */
size_t kvc_workspace_size(kvc_op op, const kvc_kv_desc* kv, int32_t w, int32_t k);

/* ---------------------------------------------------------------------------------------
 * kvc_window_scores — token scores from window attention.
 * Defined by "Add TOVA press" (kvpress PR 12, SimJeg's shape walk-through): only the last w
 * rows of the attention matrix are formed; scores are the mean over query heads (repeated
 * over KV heads), and by cold-compress PR 11 (attention mean-pooled over each KV head's
 * grouped queries; SnapKV's observation window votes for prefix tokens).
 *
 *   s[b,h,i,j] = scale * q_win[b,h,i,:] . K[b,kvh(h),j,:]
 *   p = softmax over the visible j (row max / sum taken over the whole sequence)
 *   scores[b,kvh,j] = sum_i mean_{h} p[b,h,i,j]   (mean over the group, or over all heads)
 *
 *   q_win  [B,H,w,D] bf16, the last w query rows; window row i sits at position S-w+i.
 *   K      cache described by kv (S rows).
 *   causal 1: row i sees j <= S-w+i (prefill); 0: every row sees every slot (decode).
 *   live_mask [B,KVH,ceil(S/32)] uint32 (bit j%32 of word j/32 = slot j live) or NULL = all.
 *   scores [B,KVH,S] float32 out; 0 for dead, invisible, or fully-masked slots.
 *   The [H,w,S] probabilities are never written to memory.
 *   1 <= w <= S, w*H/KVH <= 512.  ws: kvc_workspace_size(KVC_OP_WINDOW_SCORES, kv, w, 0).
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_window_scores(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_kv_desc* kv,
                             int32_t w, float scale, int32_t causal, const uint32_t* live_mask,
                             kvc_head_reduce reduce, float* scores, void* ws, size_t ws_bytes,
                             kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_window_scores_noalloc — kvc_window_scores without a caller workspace and without any
 * device allocation.  The pages have no counterpart: this is a calling convenience.
 *
 * Some callers cannot call cudaMalloc or hand over scratch memory: a plugin run inside
 * another runtime's step whose memory planner owns every device buffer and passes the
 * plugin only its inputs and outputs, or a latency-critical loop where an allocation (and
 * the device synchronisation it can imply) is not allowed.  This entry point serves them:
 * its scratch is one fixed array of KVC_NOALLOC_SCRATCH_BYTES (4 MiB) compiled into the
 * library as device memory, which every GPU that loads the library holds until the process
 * exits.  Inputs and outputs are still the caller's, exactly as for kvc_window_scores.
 *
 *  - Shapes whose scratch (kvc_workspace_size(KVC_OP_WINDOW_SCORES, ...) for this reduce
 *    mode) exceeds the fixed size are rejected with KVC_ERR_UNSUPPORTED; nothing is launched.
 *  - The first call on a device looks up the array's device address (once, with that device
 *    current); make that first call before any stream capture on the device.  The address is
 *    kept per device ordinal for the life of the process: it belongs to the device's primary
 *    context, so do not call this after cudaDeviceReset on that device, or with another
 *    context made current through the driver API.
 *  - All calls on a device share the one array, and it keeps the last call's contents.
 *    Nothing has to be cleared between calls: the (max, sum) partials a call reads are
 *    written earlier in the same call, and the cross-CTA bookkeeping words of the fused
 *    tensor-core launch accept any prior content (each launch advances an epoch word and
 *    tags every arrival with a hash of that epoch, so words left by an earlier call, of any
 *    shape, are never mistaken for this call's arrivals).  But two calls that overlap on the
 *    GPU (different streams, or different host threads without ordering) race on the array
 *    and corrupt each other's results.  Serialise them on one stream.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 * ------------------------------------------------------------------------------------- */
#define KVC_NOALLOC_SCRATCH_BYTES (4u << 20)
kvc_status kvc_window_scores_noalloc(const kvc_bf16* q_win, const kvc_bf16* K,
                                     const kvc_kv_desc* kv, int32_t w, float scale, int32_t causal,
                                     const uint32_t* live_mask, kvc_head_reduce reduce,
                                     float* scores, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_topk_select —per (b,kvh) row of `scores`, the k chosen token indices, ascending.
 * Keeping (largest=1) takes the k highest-ranked eligible tokens; evicting (largest=0) takes
 * the k lowest-ranked.  Ranking: a outranks b iff score_a > score_b, or equal and a < b.
 * protect_tail = w forces the last w positions in (SnapKV keeps the observation window and
 * compresses only the prefix, cold-compress PR 11); it requires largest=1 and w <= k.
 * Eligible = live (live_mask as above, NULL = all).  If fewer than k are eligible (e.g.
 * k >= S: SnapKV compresses only on overflow), all are returned and the rest of the row is -1.
 *   scores [B,KVH,S] float32 (finite), S <= 327680; idx [B,KVH,k] int32 out.  ws: none needed
 *   (pass NULL, 0).
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_topk_select(const float* scores, int32_t B, int32_t KVH, int64_t S, int32_t k,
                           int32_t protect_tail, const uint32_t* live_mask, int32_t largest,
                           int32_t* idx, void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_compact_kv — gather the kept rows into a dense cache.  "Add TOVA press" (SimJeg's
 * reply): the press runs after the layer's forward pass and only rewrites its KV cache, which
 * then stays compressed (hassidm's reply); cold-compress PR 11 (SnapKV paragraph): the cache
 * receives the kept tokens only.  The compressed cache is therefore the kept rows, in order:
 *   K_out[b,kvh,t,:] = K[b,kvh,idx[b,kvh,t],:], same for V; idx -1 writes a zero row.
 *   idx [B,KVH,k] int32 in [-1, S); K_out, V_out [B,KVH,k,D] dense bf16 out.
 *   V and V_out may both be NULL (keys only).  Outputs must not overlap inputs.  V may be
 *   the device address of page-locked host memory (kvc_host_device_pointer): only the kept
 *   rows are read.
 *   An index >= S is skipped and reported as KVC_ERR_DEVICE_BOUNDS by kvc_get_device_status.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_compact_kv(const kvc_bf16* K, const kvc_bf16* V, const kvc_kv_desc* kv,
                          const int32_t* idx, int32_t k, kvc_bf16* K_out, kvc_bf16* V_out,
                          kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_topk_compact — kvc_topk_select followed by kvc_compact_kv of the chosen rows, in one
 * call (two kernels; the gather starts as the selection ends): choosing the tokens a press
 * keeps per KV head and rewriting the cache to them ("Add TOVA press": the scores are repeated
 * over the KV heads and each head's cache keeps its best tokens; cold-compress PR 11: SnapKV
 * keeps the observation window and compresses the prefix).
 *   Arguments as in those two calls: scores [B,KVH,S] float32; K/V described by kv (V may be
 *   NULL, then V_out too); idx [B,KVH,k] int32 out; K_out/V_out [B,KVH,k,D] dense bf16 out,
 *   zero rows where idx is -1.  No output may overlap scores, K, V or another output.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_topk_compact(const float* scores, const kvc_bf16* K, const kvc_bf16* V,
                            const kvc_kv_desc* kv, int32_t k, int32_t protect_tail,
                            const uint32_t* live_mask, int32_t largest, int32_t* idx,
                            kvc_bf16* K_out, kvc_bf16* V_out, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_topk_compact_channels — kvc_topk_compact, and ThinK's key-channel scores of the kept
 * keys ("Add ThinK_Press", kvpress PR 18: the group's window queries' squared norm per channel,
 * averaged over the group's heads, times the kept keys' squared norm per channel; as
 * kvc_channel_score with idx = the kept rows).  The compaction sums the kept keys' squares as
 * it reads them, so K_out is not read again; one small kernel then forms the scores.
 *   Arguments as kvc_topk_compact, plus q_win [B,H,w,D] bf16 (the window queries, kv.H heads)
 *   and channel_scores [B,KVH,D] float32 out (16-byte aligned, overlapping no other argument).
 *   ws: kvc_workspace_size(KVC_OP_TOPK_COMPACT_CHANNELS, kv, 0, k) bytes, any content.  Rows
 *   whose index is -1 add nothing to the key norms.  B * KVH <= 65535 (else
 *   KVC_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_topk_compact_channels(const float* scores, const kvc_bf16* K, const kvc_bf16* V,
                                     const kvc_kv_desc* kv, int32_t k, int32_t protect_tail,
                                     const uint32_t* live_mask, int32_t largest, int32_t* idx, kvc_bf16* K_out,
                                     kvc_bf16* V_out, const kvc_bf16* q_win, int32_t w, float* channel_scores,
                                     void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_compress_prefill — window scores, top-k and compaction in one call: the press applied
 * after the prefill attention of one layer.  "Add TOVA press" (kvpress PR 12): score the
 * cached tokens by the last query rows' attention averaged over heads and keep the best;
 * cold-compress PR 11 (SnapKV paragraph): keep every token of the observation window and
 * compress the prefix by the window's attention.
 *   q_win [B,H,w,D] bf16; K/V described by kv (V may be NULL with V_out NULL: keys only; V
 *   may be mapped page-locked host memory, see kvc_host_device_pointer).
 *   scores [B,KVH,S] float32 out, or NULL (not written).  idx [B,KVH,k] int32 out, ascending,
 *   -1 padded when fewer than k tokens exist.  K_out/V_out [B,KVH,k,D] dense bf16 out, zero
 *   rows where idx is -1.  Causal window; protect_tail as in kvc_topk_select (<= min(k, w)).
 *   No output may overlap an input or another output.
 *   Short rows (G*w <= 16, S <= 1024 at D = 64 or S <= 512 at D = 128, k <= S rounded up to a
 *   multiple of 64; all-heads mode also KVH <= 8) run as one kernel that reads K once and
 *   needs no workspace.  Otherwise ws: kvc_workspace_size(KVC_OP_COMPRESS_PREFILL, kv, w, k)
 *   bytes (k must be the call's k), which include room for the scores when scores is NULL.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_compress_prefill(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_bf16* V,
                                const kvc_kv_desc* kv, int32_t w, float scale,
                                kvc_head_reduce reduce, int32_t k, int32_t protect_tail,
                                float* scores, int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out,
                                void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_compress_prefill_channels — kvc_compress_prefill, and ThinK's key-channel scores of the
 * kept keys ("Add ThinK_Press", kvpress PR 18: the channel score is the window queries'
 * squared norm per channel, averaged over the group's heads, times the kept keys' squared
 * norm per channel, as in kvc_channel_score with idx = the kept rows).  The key norms are
 * summed by the compaction while it reads the kept K rows (kvc_topk_compact_channels), so
 * K_out is not read again.
 *   Arguments as kvc_compress_prefill, plus channel_scores [B,KVH,D] float32 out (16-byte
 *   aligned, not NULL, overlapping no other argument).  Always takes the multi-kernel path
 *   (window scores, top-k, compaction with the channel sums, one small final kernel).
 *   ws: kvc_workspace_size(KVC_OP_COMPRESS_PREFILL_CHANNELS, kv, w, k) bytes (k must be the
 *   call's k), including room for the scores when scores is NULL.  Rows whose index is -1
 *   (fewer than k tokens) add nothing to the key norms.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_compress_prefill_channels(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_bf16* V,
                                         const kvc_kv_desc* kv, int32_t w, float scale,
                                         kvc_head_reduce reduce, int32_t k, int32_t protect_tail,
                                         float* scores, int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out,
                                         float* channel_scores, void* ws, size_t ws_bytes,
                                         kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_write_slots — the decode-step insertion into a fixed-size cache: the new token's key and
 * value rows go into the slot an eviction freed (cold-compress PR 11 description: the eviction
 * queue evicts one token at each step, so every new token takes an evicted token's slot and no
 * slot stays empty; a TOVA decode step evicts the lowest-scoring token the same way).
 *   K[b,kvh,slot[b,kvh],:] = k_new[b,kvh,:] (same for V; V pair may be NULL).
 *   k_new, v_new [B,KVH,D] bf16; slot [B,KVH] int32 in [0, S).  K/V are updated in place.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_write_slots(const kvc_bf16* k_new, const kvc_bf16* v_new, const int32_t* slot,
                           kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_tova_decode_step — one TOVA generation step on a cache of S = budget+1 slots
 * ("Add TOVA press": the score is the last query's attention averaged over heads).
 * Writes the new token into slot free_slot[b,kvh], scores every slot with the new query
 * (mean over all heads, no causal mask), and evicts the lowest-ranked slot: on return
 * free_slot[b,kvh] holds the evicted slot (identical for every kvh of a batch row).
 *   q_new [B,H,D], k_new/v_new [B,KVH,D] bf16; K/V updated in place; free_slot [B,KVH]
 *   int32 in/out; scores [B,KVH,S] float32 out.  ws: KVC_OP_TOVA_DECODE_STEP.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_tova_decode_step(const kvc_bf16* q_new, const kvc_bf16* k_new,
                                const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V,
                                const kvc_kv_desc* kv, float scale, int32_t* free_slot,
                                float* scores, void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Scissorhands (cold-compress PR 11): per (b,kvh,slot) a circular history of
 * "attention < 1/keys" flags over the last `history` steps (default 400), and bulk eviction
 * of the tokens with the highest fraction of low flags.
 *
 * State: caller-owned device buffers (zeroed by kvc_scissorhands_init) plus host counters.
 *   hist        [history][B][KVH][cap/32] uint32 — bit plane (t % history) = step t's flags
 *   low_count   [B][KVH][cap] uint16 — low flags of the current token over its last
 *               n_obs = min(history, t - insert_step + 1) observations
 *   insert_step [B][KVH][cap] int32 — step at which the slot's token entered (prefill: 0)
 *   live        [B][KVH][cap/32] uint32 — occupied slots
 *   slot        [B][KVH] int32 — slot filled by the last insertion
 *   t           host: index of the next recorded step (advanced by each update)
 *   n_free      host: free slots per (b,kvh) (identical for all heads)
 * cap must be a multiple of 32 and <= 40960, history in [1, 4096], B * KVH <= 65535.
 * ------------------------------------------------------------------------------------- */
typedef struct {
  int32_t B, KVH, cap, history;
  uint32_t* hist;
  uint16_t* low_count;
  int32_t* insert_step;
  uint32_t* live;
  int32_t* slot;
  int64_t t;
  int32_t n_free;
} kvc_sh_state;

/* Zero the state; mark slots [0, n_live) live with insert_step 0; t = 0. */
kvc_status kvc_scissorhands_init(kvc_sh_state* st, int32_t n_live, kvc_stream_t stream);

/* Record step t from GQA-mean probabilities p [B,KVH,cap] float32 (dead slots ignored):
 * flag = live && p < float32(1)/float32(keys), keys = live slots of the (b,kvh) row; the
 * flag replaces bit plane t % history; low_count gains the new flag and loses the flag it
 * overwrites when that one belongs to the current token (age >= history).  Then t += 1. */
kvc_status kvc_scissorhands_update_from_probs(kvc_sh_state* st, const float* p,
                                              kvc_stream_t stream);

/* One decode step: insert the new token (k_new/v_new [B,KVH,D]) into the lowest free slot of
 * every (b,kvh) (written to K/V, live, insert_step = t, low_count = 0, st->slot), score the
 * new query q_new [B,H,D] over the live slots (GQA-mean probability, written to probs
 * [B,KVH,cap] float32), and record the flags as kvc_scissorhands_update_from_probs.
 * kv describes K/V with S == cap.  Requires st->n_free > 0.  ws: KVC_OP_SCISSORHANDS_UPDATE. */
kvc_status kvc_scissorhands_update(kvc_sh_state* st, const kvc_bf16* q_new, const kvc_bf16* k_new,
                                   const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V,
                                   const kvc_kv_desc* kv, float scale, float* probs, void* ws,
                                   size_t ws_bytes, kvc_stream_t stream);

/* Evict, per (b,kvh), the m live slots with the highest fraction low_count / n_obs of the
 * last recorded step (compared exactly; ties: lower slot first; a token not yet observed,
 * n_obs = 0, counts as fraction 0).  evicted [B,KVH,m] int32
 * out, ascending (-1 padded when fewer are live); their live bits are cleared. */
kvc_status kvc_scissorhands_evict(kvc_sh_state* st, int32_t m, int32_t* evicted,
                                  kvc_stream_t stream);

/* Eviction-queue variant (cold-compress PR 11 description: instead of evicting in bulk every
 * m steps, refill an eviction queue every m steps and evict one token per step, so no slot is
 * left empty).  Fill queue [B,KVH,m] int32 with the m live slots that kvc_scissorhands_evict
 * would take, listed most evictable first (highest fraction low_count / n_obs, compared
 * exactly; ties: lower slot first), -1 padded when fewer are live.  Nothing is evicted: live
 * bits are not touched.  1 <= m <= min(cap, 2048); requires st->t >= 1. */
kvc_status kvc_scissorhands_refill_queue(kvc_sh_state* st, int32_t m, int32_t* queue,
                                         kvc_stream_t stream);

/* One decode step of the queue variant: as kvc_scissorhands_update, except that the new token
 * replaces the token in slot queue[b,kvh,pos] (which must be live; otherwise the row is
 * skipped and KVC_ERR_DEVICE_BOUNDS is recorded for kvc_get_device_status).  n_free is
 * unchanged.  0 <= pos < m. */
kvc_status kvc_scissorhands_update_queued(kvc_sh_state* st, const int32_t* queue, int32_t m,
                                          int32_t pos, const kvc_bf16* q_new,
                                          const kvc_bf16* k_new, const kvc_bf16* v_new,
                                          kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv,
                                          float scale, float* probs, void* ws, size_t ws_bytes,
                                          kvc_stream_t stream);

/* Insert the new token without recording: the steps between two observations under sparse
 * recording (the PR review thread's suggestion: look at attention only every M steps; t and
 * n_obs then count recordings).  queue == NULL: the lowest free slot (requires n_free > 0;
 * n_free -= 1).  Otherwise the token replaces slot queue[b,kvh,pos] as in
 * kvc_scissorhands_update_queued.  The slot gets insert_step = t (its first observation is
 * the next recording) and low_count = 0; the new rows are written to K/V (S == cap). */
kvc_status kvc_scissorhands_insert(kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos,
                                   const kvc_bf16* k_new, const kvc_bf16* v_new, kvc_bf16* K,
                                   kvc_bf16* V, const kvc_kv_desc* kv, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_channel_score — ThinK key-channel score ("Add ThinK_Press", kvpress PR 18: the
 * defining sum_{i,j} (q_id k_jd)^2 factorises into query_norm * key_norm):
 *   cs[b,kvh,d] = (mean_{h in group} sum_i q_win[b,h,i,d]^2) * sum_{j} K[b,kvh,j,d]^2
 * with raw (unscaled) window queries.  idx == NULL: j runs over all S rows of K (e.g. the
 * already compacted cache); otherwise over the rows idx[b,kvh,0..k) of K (-1 skipped).
 *   q_win [B,H,w,D] bf16; cs [B,KVH,D] float32 out.  ws: KVC_OP_CHANNEL_SCORE (w, k).
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_channel_score(const kvc_bf16* q_win, int32_t w, const kvc_bf16* K,
                             const kvc_kv_desc* kv, const int32_t* idx, int32_t k, float* cs,
                             void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_channel_prune — keep the C highest-scoring key channels per (b,kvh) (ties: lower
 * channel first); ch_idx [B,KVH,C] int32 out, ascending.
 *   zero_mode 0: K_out [B,KVH,S,C] dense = K[..., ch_idx] (the smaller key cache; "Add
 *                ThinK_Press" options 3b/3c).
 *   zero_mode 1: K_out [B,KVH,S,D] dense = K with the other channels zeroed (option 3a);
 *                K_out may equal K when K is dense (in place).
 *   cs [B,KVH,D] float32.  ch_idx shares no bytes with cs, K or K_out (KVC_ERR_INVALID_ARG).
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_channel_prune(const float* cs, const kvc_bf16* K, const kvc_kv_desc* kv,
                             int32_t C, int32_t zero_mode, int32_t* ch_idx, kvc_bf16* K_out,
                             kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_value_channel_score — ThinK value-channel score ("Add ThinK_Press" names value-cache
 * pruning without defining it; this carries the key score's definition over to values):
 *   cs[b,kvh,d] = mean_{h in group} sum_i sum_j (p[b,h,i,j] * Vc[b,kvh,j,d])^2
 * with p the window's attention over the compressed cache: softmax_j(scale * q_win . Kc_j),
 * causal with the w window rows as the LAST w tokens of the cache (as kvc_compress_prefill
 * with protect_tail = w leaves them).  Computed as sum_j wt_j Vc_jd^2 with
 * wt_j = mean_h sum_i p_hij^2 (the window scores with p squared).
 *   q_win [B,H,w,D] bf16; Kc, Vc: the compressed cache, both described by kv (S = kept
 *   tokens); cs [B,KVH,D] float32 out; ws: kvc_workspace_size(KVC_OP_VALUE_CHANNEL_SCORE,
 *   kv, w, 0).  kvc_channel_prune(cs, Vc, ...) then prunes the value channels.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_value_channel_score(const kvc_bf16* q_win, int32_t w, const kvc_bf16* Kc,
                                   const kvc_bf16* Vc, const kvc_kv_desc* kv, float scale,
                                   float* cs, void* ws, size_t ws_bytes, kvc_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kvc_decode_attention — attention of one new query per head over a (compressed) cache, the
 * decoding step that uses ThinK's smaller key cache ("Add ThinK_Press": option 3c prunes the
 * query to the kept channels, as the author's reply proposes; with ch == NULL it is plain
 * decoding attention, which option 3b runs after kvc_zero_add_back).  For each (b, h) with
 * kvh = h / (H / KVH):
 *   s_j = scale * sum_c q[b,h,ch[b,kvh,c]] * K[b,kvh,j,c]   over live slots j,
 *   out[b,h,:] = sum_j softmax(s)_j * V[b,kvh,j,:]          (zeros when no slot is live).
 *   q [B,H,D] bf16, D = vd->D (the full head); scale: the full head's 1/sqrt(D).
 *   kd: K [B,KVH,S,Ck] bf16 with Ck = kd->D kept channels (64 or 128, <= D), rows dense
 *       (stride_s == Ck); ch [B,KVH,Ck] int32 kept channel list, or NULL when Ck == D.
 *   vd: V [B,KVH,S,D] bf16, rows dense; kd and vd agree on B, H, KVH, S.
 *   live_mask [B,KVH,ceil(S/32)] or NULL; out [B,H,D] float32.
 *   ws: kvc_workspace_size(KVC_OP_DECODE_ATTENTION, vd, 0, 0).
 * An entry of ch outside [0, D) counts as a zero query channel and records
 * KVC_ERR_DEVICE_BOUNDS for kvc_get_device_status.  B * KVH <= 65535.
 * ------------------------------------------------------------------------------------- */
kvc_status kvc_decode_attention(const kvc_bf16* q, const int32_t* ch, const kvc_bf16* K,
                                const kvc_kv_desc* kd, const kvc_bf16* V, const kvc_kv_desc* vd,
                                const uint32_t* live_mask, float scale, float* out, void* ws,
                                size_t ws_bytes, kvc_stream_t stream);

/* kvc_zero_add_back — option 3b of "Add ThinK_Press": rebuild the full-width key cache from
 * the pruned one, K_out[b,kvh,j,ch[b,kvh,c]] = Kp[b,kvh,j,c] and every other channel 0.
 *   pd: Kp [B,KVH,S,C] (C = pd->D); od: K_out [B,KVH,S,D] (D = od->D >= C); ch [B,KVH,C]
 *   int32 (as written by kvc_channel_prune).  K_out must not overlap Kp.  Entries of ch
 *   outside [0, D) are skipped and record KVC_ERR_DEVICE_BOUNDS. */
kvc_status kvc_zero_add_back(const kvc_bf16* Kp, const kvc_kv_desc* pd, const int32_t* ch,
                             kvc_bf16* K_out, const kvc_kv_desc* od, kvc_stream_t stream);

/* Device address of page-locked (pinned) host memory, for the inputs that may stay on the
 * host: V of kvc_compact_kv, kvc_topk_compact and kvc_compress_prefill is read only by the
 * compaction kernel, with plain loads, row by row, so passing this address moves just the
 * kept rows over the host link instead of uploading all of V.  KVC_ERR_INVALID_ARG when
 * host_ptr is not page-locked host memory mapped for the current device.  No other pointer
 * argument of this library may be host memory. */
kvc_status kvc_host_device_pointer(const void* host_ptr, void** dev_ptr);

/* Synchronize `stream`, then return (and clear) the sticky device status: KVC_OK,
 * KVC_ERR_DEVICE_BOUNDS or KVC_ERR_TIMEOUT.  KVC_ERR_CUDA if the sync itself failed. */
kvc_status kvc_get_device_status(kvc_stream_t stream);

/* Static description of a status code. */
const char* kvc_status_string(kvc_status s);

/* Detail of the most recent failed call on this host thread ("" if none). */
const char* kvc_last_error_message(void);

/* Library version: major*10000 + minor*100 + patch. */
int32_t kvc_version(void);

/* Diagnostics: number of kernels this library has enqueued since it was loaded (all host
 * threads, all devices).  The difference over a region counts the region's launches. */
int64_t kvc_launch_count(void);

/* Diagnostics: a test of the bounded-wait path.  armed = 1: the next fused tensor-core window
 * scoring launch in this process (kvc_window_scores and the calls built on it, for shapes
 * with more than 32 query rows per KV head whose CTAs are all resident at once) bounds each
 * wait by 1 ms instead of 2 s and leaves out the key-range arrival of its first CTA.  The
 * other CTAs of that (b, kvh) give up their wait, the launch still returns (its scores for
 * that (b, kvh) are then undefined), and kvc_get_device_status reports KVC_ERR_TIMEOUT.  The
 * device stays usable: the next call computes normally.  armed = 0 disarms it if no such
 * launch came.  Never needed outside tests. */
kvc_status kvc_debug_inject_timeout(int32_t armed);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
