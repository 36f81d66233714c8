// libkvc C ABI: argument validation, workspace planning and dispatch onto the caller's
// stream.  Every entry point validates on the host before enqueuing anything and reports
// failures as kvc_status codes; no exception crosses the boundary.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "kvc_decode.cuh"
#include "kvc_internal.cuh"

namespace kvc {

namespace {
thread_local char t_err[512] = {0};

// An NVTX range named after the entry point around each call, so that a timeline tool shows
// which library call enqueued which kernels.  Without a tool attached a push/pop is a call
// through an empty function pointer.
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
};
#define KVC_RANGE() NvtxScope kvc_nvtx_scope_(__func__)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvc_status fail(kvc_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return s;
}

kvc_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVC_OK;
  return fail(KVC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

kvc_status check_desc(const kvc_kv_desc* kv, const char* name) {
  if (!kv) return fail(KVC_ERR_INVALID_ARG, "%s: descriptor is NULL", name);
  if (kv->B < 1 || kv->H < 1 || kv->KVH < 1 || kv->S < 1)
    return fail(KVC_ERR_INVALID_ARG, "%s: B, H, KVH and S must be >= 1", name);
  if (kv->H % kv->KVH != 0) return fail(KVC_ERR_INVALID_ARG, "%s: H %% KVH != 0", name);
  if (kv->D != 64 && kv->D != 128) return fail(KVC_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128", name);
  if (kv->S > (int64_t)INT32_MAX - 64) return fail(KVC_ERR_UNSUPPORTED, "%s: S too large", name);
  if (kv->stride_b % 8 || kv->stride_h % 8 || kv->stride_s % 8)
    return fail(KVC_ERR_INVALID_ARG, "%s: strides must be multiples of 8 elements", name);
  if (kv->stride_s < kv->D) return fail(KVC_ERR_INVALID_ARG, "%s: stride_s < D", name);
  if (kv->stride_b < 0 || kv->stride_h < 0) return fail(KVC_ERR_INVALID_ARG, "%s: negative stride", name);
  return KVC_OK;
}

// byte range [lo, hi) touched by a strided cache
void cache_range(const void* base, const kvc_kv_desc& kv, uintptr_t* lo, uintptr_t* hi) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  const int64_t last = (kv.B - 1) * kv.stride_b + (kv.KVH - 1) * kv.stride_h + (kv.S - 1) * kv.stride_s + kv.D;
  *lo = b;
  *hi = b + (uintptr_t)last * 2;
}
bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

kvc_status check_ptr(const void* p, const char* what) {
  if (!p) return fail(KVC_ERR_INVALID_ARG, "%s is NULL", what);
  if (!aligned16(p)) return fail(KVC_ERR_INVALID_ARG, "%s is not 16-byte aligned", what);
  return KVC_OK;
}

// An output [out, out + out_bytes) may share no byte with any of the n input ranges [lo, hi)
// (a range with lo == hi is absent).
kvc_status check_out_apart(const void* out, size_t out_bytes, const uintptr_t (*in)[2], int n, const char* what) {
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + out_bytes;
  for (int i = 0; i < n; ++i)
    if (in[i][0] != in[i][1] && overlaps(o0, o1, in[i][0], in[i][1]))
      return fail(KVC_ERR_INVALID_ARG, "%s overlaps an input or the workspace", what);
  return KVC_OK;
}

kvc_status check_ws(void* ws, size_t have, size_t need, const char* what) {
  if (need == 0) return KVC_OK;
  if (!ws || have < need)
    return fail(KVC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed (%zu given)", what, need, ws ? have : 0);
  if (!aligned16(ws)) return fail(KVC_ERR_INVALID_ARG, "%s: workspace not 16-byte aligned", what);
  return KVC_OK;
}

#define KVC_TRY(x)                  \
  do {                              \
    const kvc_status _s = (x);      \
    if (_s != KVC_OK) return _s;    \
  } while (0)

// scratch of kvc_value_channel_score, 16-byte aligned pieces: the window-score workspace,
// one weight per token (at *wts_off), the channel partials (at *part_off)
size_t value_score_workspace(const kvc_kv_desc& kv, int w, size_t* wts_off = nullptr, size_t* part_off = nullptr) {
  const size_t a = (scores_workspace(kv, w, KVC_REDUCE_GQA_GROUP) + 15) / 16 * 16;
  const size_t b = ((size_t)kv.B * kv.KVH * kv.S * sizeof(float) + 15) / 16 * 16;
  if (wts_off) *wts_off = a;
  if (part_off) *part_off = a + b;
  return a + b + channel_score_workspace(kv, 0, false);
}

kvc_status check_window(const kvc_kv_desc* kv, int32_t w, const char* name) {
  if (w < 1 || (int64_t)w > kv->S) return fail(KVC_ERR_INVALID_ARG, "%s: need 1 <= w <= S", name);
  if ((int64_t)w * (kv->H / kv->KVH) > 512)
    return fail(KVC_ERR_UNSUPPORTED, "%s: w * H / KVH must be <= 512", name);
  return KVC_OK;
}

kvc_status check_sh(const kvc_sh_state* st) {
  if (!st) return fail(KVC_ERR_INVALID_ARG, "scissorhands state is NULL");
  if (st->B < 1 || st->KVH < 1 || st->cap < 32 || st->cap % 32)
    return fail(KVC_ERR_INVALID_ARG, "scissorhands: B, KVH >= 1 and cap a positive multiple of 32");
  if (st->history < 1 || st->history > 4096) return fail(KVC_ERR_INVALID_ARG, "scissorhands: history in [1, 4096]");
  if (st->cap > 40960) return fail(KVC_ERR_UNSUPPORTED, "scissorhands: cap must be <= 40960");
  if ((int64_t)st->B * st->KVH > 65535) return fail(KVC_ERR_UNSUPPORTED, "scissorhands: B * KVH must be <= 65535");
  if (!st->hist || !st->low_count || !st->insert_step || !st->live || !st->slot)
    return fail(KVC_ERR_INVALID_ARG, "scissorhands: a state buffer is NULL");
  if (st->t < 0 || st->t > INT32_MAX) return fail(KVC_ERR_INVALID_ARG, "scissorhands: step counter out of range");
  return KVC_OK;
}

}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
}

static std::atomic<long long> g_launches{0};

cudaError_t launched(int n) {
  g_launches.fetch_add(n, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t func_attrs_once(const void* fn, int max_dynamic_smem) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({fn, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && max_dynamic_smem > 48 * 1024)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
  if (e == cudaSuccess) done.insert({fn, dev});
  return e;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

}  // namespace kvc

using namespace kvc;

extern "C" {

int32_t kvc_version(void) { return 10000; }

int64_t kvc_launch_count(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }

kvc_status kvc_debug_inject_timeout(int32_t armed) {
  KVC_RANGE();
  inject_scores_timeout(armed);
  return KVC_OK;
}

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVC_ERR_CUDA: return "CUDA error";
    case KVC_ERR_TIMEOUT: return "device wait timed out";
    case KVC_ERR_DEVICE_BOUNDS: return "device index out of range";
    case KVC_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* kvc_last_error_message(void) { return t_err; }

size_t kvc_workspace_size(kvc_op op, const kvc_kv_desc* kv, int32_t w, int32_t k) {
  if (op == KVC_OP_TOPK_SELECT || op == KVC_OP_SCISSORHANDS_EVICT) return 0;
  if (!kv || check_desc(kv, "kvc_workspace_size") != KVC_OK) return (size_t)-1;
  switch (op) {
    case KVC_OP_WINDOW_SCORES:
      if (check_window(kv, w, "kvc_workspace_size") != KVC_OK) return (size_t)-1;
      return scores_workspace(*kv, w, KVC_REDUCE_ALL_HEADS);
    case KVC_OP_TOPK_COMPACT_CHANNELS:
      if (check_desc(kv, "kvc_workspace_size") != KVC_OK || k < 1) return (size_t)-1;
      return compact_channels_workspace(*kv, k);
    case KVC_OP_COMPRESS_PREFILL_CHANNELS:
      if (check_window(kv, w, "kvc_workspace_size") != KVC_OK) return (size_t)-1;
      return (scores_workspace(*kv, w, KVC_REDUCE_ALL_HEADS) + 255) / 256 * 256 +
             ((size_t)kv->B * kv->KVH * kv->S * sizeof(float) + 255) / 256 * 256 + compact_channels_workspace(*kv, k);
    case KVC_OP_COMPRESS_PREFILL:
      if (check_window(kv, w, "kvc_workspace_size") != KVC_OK) return (size_t)-1;
      // the fused short-row kernel needs none; otherwise the window-score scratch plus room
      // for the scores when the caller passes none
      if (prefill_fused_supported(*kv, w, k, KVC_REDUCE_GQA_GROUP) &&
          prefill_fused_supported(*kv, w, k, KVC_REDUCE_ALL_HEADS))
        return 0;
      return (scores_workspace(*kv, w, KVC_REDUCE_ALL_HEADS) + 255) / 256 * 256 +
             (size_t)kv->B * kv->KVH * kv->S * sizeof(float);
    case KVC_OP_TOVA_DECODE_STEP:
    case KVC_OP_SCISSORHANDS_UPDATE:
      return scores_workspace(*kv, 1, KVC_REDUCE_ALL_HEADS);
    case KVC_OP_CHANNEL_SCORE:
      return channel_score_workspace(*kv, k, k > 0);
    case KVC_OP_DECODE_ATTENTION:
      return plan_decode(*kv).part_bytes;
    case KVC_OP_VALUE_CHANNEL_SCORE:
      if (check_window(kv, w, "kvc_workspace_size") != KVC_OK) return (size_t)-1;
      return value_score_workspace(*kv, w);
    default:
      return (size_t)-1;
  }
}

kvc_status kvc_window_scores(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_kv_desc* kv,
                             int32_t w, float scale, int32_t causal, const uint32_t* live_mask,
                             kvc_head_reduce reduce, float* scores, void* ws, size_t ws_bytes,
                             kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_window_scores"));
  KVC_TRY(check_window(kv, w, "kvc_window_scores"));
  KVC_TRY(check_ptr(q_win, "q_win"));
  KVC_TRY(check_ptr(K, "K"));
  KVC_TRY(check_ptr(scores, "scores"));
  if (live_mask && !aligned16(live_mask)) return fail(KVC_ERR_INVALID_ARG, "live_mask not 16-byte aligned");
  if (reduce != KVC_REDUCE_GQA_GROUP && reduce != KVC_REDUCE_ALL_HEADS)
    return fail(KVC_ERR_INVALID_ARG, "unknown head reduction");
  if (!(scale > 0.f) || scale != scale) return fail(KVC_ERR_INVALID_ARG, "scale must be > 0");
  const size_t need = scores_workspace(*kv, w, reduce);
  KVC_TRY(check_ws(ws, ws_bytes, need, "kvc_window_scores"));
  {
    uintptr_t in[3][2];
    cache_range(K, *kv, &in[0][0], &in[0][1]);
    in[1][0] = reinterpret_cast<uintptr_t>(q_win);
    in[1][1] = in[1][0] + (uintptr_t)kv->B * kv->H * w * kv->D * 2;
    in[2][0] = reinterpret_cast<uintptr_t>(ws);
    in[2][1] = need ? in[2][0] + need : in[2][0];
    KVC_TRY(check_out_apart(scores, (size_t)kv->B * kv->KVH * kv->S * 4, in, 3, "kvc_window_scores: scores"));
  }
  return cuda_status(launch_window_scores(q_win, K, *kv, w, scale, causal ? 1 : 0, live_mask, reduce,
                                          scores, ws, (cudaStream_t)stream),
                     "kvc_window_scores launch");
}

kvc_status kvc_window_scores_noalloc(const kvc_bf16* q_win, const kvc_bf16* K,
                                     const kvc_kv_desc* kv, int32_t w, float scale, int32_t causal,
                                     const uint32_t* live_mask, kvc_head_reduce reduce,
                                     float* scores, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_window_scores_noalloc"));
  KVC_TRY(check_window(kv, w, "kvc_window_scores_noalloc"));
  KVC_TRY(check_ptr(q_win, "q_win"));
  KVC_TRY(check_ptr(K, "K"));
  KVC_TRY(check_ptr(scores, "scores"));
  if (live_mask && !aligned16(live_mask)) return fail(KVC_ERR_INVALID_ARG, "live_mask not 16-byte aligned");
  if (reduce != KVC_REDUCE_GQA_GROUP && reduce != KVC_REDUCE_ALL_HEADS)
    return fail(KVC_ERR_INVALID_ARG, "unknown head reduction");
  if (!(scale > 0.f) || scale != scale) return fail(KVC_ERR_INVALID_ARG, "scale must be > 0");
  const size_t need = scores_workspace(*kv, w, reduce);
  if (need > (size_t)KVC_NOALLOC_SCRATCH_BYTES)
    return fail(KVC_ERR_UNSUPPORTED,
                "kvc_window_scores_noalloc: these shapes need %zu bytes of scratch; the fixed array holds %zu",
                need, (size_t)KVC_NOALLOC_SCRATCH_BYTES);
  {
    uintptr_t in[2][2];
    cache_range(K, *kv, &in[0][0], &in[0][1]);
    in[1][0] = reinterpret_cast<uintptr_t>(q_win);
    in[1][1] = in[1][0] + (uintptr_t)kv->B * kv->H * w * kv->D * 2;
    KVC_TRY(check_out_apart(scores, (size_t)kv->B * kv->KVH * kv->S * 4, in, 2,
                            "kvc_window_scores_noalloc: scores"));
  }
  void* scratch = nullptr;
  KVC_TRY(cuda_status(noalloc_scratch(&scratch), "kvc_window_scores_noalloc scratch address"));
  return cuda_status(launch_window_scores(q_win, K, *kv, w, scale, causal ? 1 : 0, live_mask, reduce,
                                          scores, scratch, (cudaStream_t)stream),
                     "kvc_window_scores_noalloc launch");
}

kvc_status kvc_topk_select(const float* scores, int32_t B, int32_t KVH, int64_t S, int32_t k,
                           int32_t protect_tail, const uint32_t* live_mask, int32_t largest,
                           int32_t* idx, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  (void)ws;
  (void)ws_bytes;
  if (B < 1 || KVH < 1 || S < 1 || k < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select: B, KVH, S, k must be >= 1");
  if (S > topk_max_len()) return fail(KVC_ERR_UNSUPPORTED, "kvc_topk_select: S > %lld", (long long)topk_max_len());
  if ((int64_t)B * KVH > 2147483647LL) return fail(KVC_ERR_UNSUPPORTED, "kvc_topk_select: too many rows");
  if (protect_tail < 0 || protect_tail > k || (int64_t)protect_tail > S)
    return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select: need 0 <= protect_tail <= min(k, S)");
  if (protect_tail && !largest) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_select: protect_tail needs largest=1");
  KVC_TRY(check_ptr(scores, "scores"));
  if (!idx) return fail(KVC_ERR_INVALID_ARG, "idx is NULL");
  if (live_mask && !aligned16(live_mask)) return fail(KVC_ERR_INVALID_ARG, "live_mask not 16-byte aligned");
  return cuda_status(launch_topk(scores, B, KVH, S, k, protect_tail, live_mask, largest ? 1 : 0, idx,
                                 (cudaStream_t)stream),
                     "kvc_topk_select launch");
}

namespace {
// K/V, the dense outputs K_out/V_out [B,KVH,k,D] and their overlaps, for the gathers
kvc_status check_gather(const kvc_bf16* K, const kvc_bf16* V, const kvc_kv_desc* kv, int32_t k,
                        const kvc_bf16* K_out, const kvc_bf16* V_out, const char* who) {
  KVC_TRY(check_desc(kv, who));
  if (k < 1) return fail(KVC_ERR_INVALID_ARG, "%s: k must be >= 1", who);
  KVC_TRY(check_ptr(K, "K"));
  KVC_TRY(check_ptr(K_out, "K_out"));
  if ((V == nullptr) != (V_out == nullptr)) return fail(KVC_ERR_INVALID_ARG, "V and V_out must both be given or both NULL");
  if (V) {
    KVC_TRY(check_ptr(V, "V"));
    KVC_TRY(check_ptr(V_out, "V_out"));
  }
  uintptr_t k0, k1, v0 = 0, v1 = 0;
  cache_range(K, *kv, &k0, &k1);
  if (V) cache_range(V, *kv, &v0, &v1);
  const uintptr_t osz = (uintptr_t)kv->B * kv->KVH * (uintptr_t)k * kv->D * 2;
  const uintptr_t ko = reinterpret_cast<uintptr_t>(K_out), vo = reinterpret_cast<uintptr_t>(V_out);
  if (overlaps(ko, ko + osz, k0, k1) || (V && (overlaps(ko, ko + osz, v0, v1) || overlaps(vo, vo + osz, k0, k1) ||
                                               overlaps(vo, vo + osz, v0, v1) || overlaps(ko, ko + osz, vo, vo + osz))))
    return fail(KVC_ERR_INVALID_ARG, "%s: outputs overlap inputs", who);
  return KVC_OK;
}
}  // namespace

kvc_status kvc_compact_kv(const kvc_bf16* K, const kvc_bf16* V, const kvc_kv_desc* kv,
                          const int32_t* idx, int32_t k, kvc_bf16* K_out, kvc_bf16* V_out,
                          kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_gather(K, V, kv, k, K_out, V_out, "kvc_compact_kv"));
  if (!idx) return fail(KVC_ERR_INVALID_ARG, "idx is NULL");
  return cuda_status(launch_compact(K, V, *kv, idx, k, K_out, V_out, (cudaStream_t)stream), "kvc_compact_kv launch");
}

// kvc_topk_compact, and with channel_scores also ThinK's key-channel scores of the kept keys
// (kvc_topk_compact_channels)
static kvc_status topk_compact_impl(const char* who, const float* scores, const kvc_bf16* K, const kvc_bf16* V,
                                    const kvc_kv_desc* kv, int32_t k, int32_t protect_tail,
                                    const uint32_t* live_mask, int32_t largest, int32_t* idx, kvc_bf16* K_out,
                                    kvc_bf16* V_out, const kvc_bf16* q_win, int32_t w, float* channel_scores,
                                    void* ws, size_t ws_bytes, kvc_stream_t stream) {
  if (channel_scores && (int64_t)kv->B * kv->KVH > 65535)  // (kv checked by the caller)
    return fail(KVC_ERR_UNSUPPORTED, "%s: B * KVH > 65535 with channel scores", who);
  KVC_TRY(check_gather(K, V, kv, k, K_out, V_out, who));
  if (kv->S > topk_max_len()) return fail(KVC_ERR_UNSUPPORTED, "%s: S > %lld", who, (long long)topk_max_len());
  if ((int64_t)kv->B * kv->KVH > 2147483647LL) return fail(KVC_ERR_UNSUPPORTED, "%s: too many rows", who);
  if (protect_tail < 0 || protect_tail > k || (int64_t)protect_tail > kv->S)
    return fail(KVC_ERR_INVALID_ARG, "%s: need 0 <= protect_tail <= min(k, S)", who);
  if (protect_tail && !largest) return fail(KVC_ERR_INVALID_ARG, "%s: protect_tail needs largest=1", who);
  if (channel_scores) {
    if (w < 1) return fail(KVC_ERR_INVALID_ARG, "%s: w must be >= 1", who);
    KVC_TRY(check_ptr(q_win, "q_win"));
    if (!aligned16(channel_scores)) return fail(KVC_ERR_INVALID_ARG, "channel_scores is not 16-byte aligned");
    KVC_TRY(check_ws(ws, ws_bytes, compact_channels_workspace(*kv, k), who));
  }
  KVC_TRY(check_ptr(scores, "scores"));
  if (!idx) return fail(KVC_ERR_INVALID_ARG, "idx is NULL");
  if (live_mask && !aligned16(live_mask)) return fail(KVC_ERR_INVALID_ARG, "live_mask not 16-byte aligned");
  // the kernel writes K_out/V_out while other rows are still being selected: no output may
  // overlap the scores
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(scores), s1 = s0 + (uintptr_t)kv->B * kv->KVH * kv->S * 4;
  const uintptr_t osz = (uintptr_t)kv->B * kv->KVH * (uintptr_t)k * kv->D * 2;
  const uintptr_t ko = reinterpret_cast<uintptr_t>(K_out), vo = reinterpret_cast<uintptr_t>(V_out);
  const uintptr_t i0 = reinterpret_cast<uintptr_t>(idx), i1 = i0 + (uintptr_t)kv->B * kv->KVH * k * 4;
  if (overlaps(ko, ko + osz, s0, s1) || (V_out && overlaps(vo, vo + osz, s0, s1)) || overlaps(i0, i1, s0, s1) ||
      overlaps(i0, i1, ko, ko + osz) || (V_out && overlaps(i0, i1, vo, vo + osz)))
    return fail(KVC_ERR_INVALID_ARG, "%s: outputs overlap inputs or each other", who);
  if (channel_scores) {
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(channel_scores), c1 = c0 + (uintptr_t)kv->B * kv->KVH * kv->D * 4;
    uintptr_t k0, k1;
    cache_range(K, *kv, &k0, &k1);
    if (overlaps(c0, c1, s0, s1) || overlaps(c0, c1, ko, ko + osz) || (V_out && overlaps(c0, c1, vo, vo + osz)) ||
        overlaps(c0, c1, i0, i1) || overlaps(c0, c1, k0, k1))
      return fail(KVC_ERR_INVALID_ARG, "%s: channel_scores overlaps another argument", who);
  }
  // two launches chained by programmatic dependent launch: the gather then runs on every SM
  // (a gather inside the selection grid, on its B*KVH*8 CTAs, measured slower)
  KVC_TRY(cuda_status(launch_topk(scores, kv->B, kv->KVH, kv->S, k, protect_tail, live_mask, largest ? 1 : 0, idx,
                                  (cudaStream_t)stream),
                      "selection launch"));
  if (channel_scores)
    return cuda_status(launch_compact_channels(K, V, *kv, idx, k, K_out, V_out, q_win, w, channel_scores, ws,
                                               (cudaStream_t)stream),
                       "gather launch");
  return cuda_status(launch_compact(K, V, *kv, idx, k, K_out, V_out, (cudaStream_t)stream), "gather launch");
}

kvc_status kvc_topk_compact(const float* scores, const kvc_bf16* K, const kvc_bf16* V, const kvc_kv_desc* kv,
                            int32_t k, int32_t protect_tail, const uint32_t* live_mask, int32_t largest,
                            int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out, kvc_stream_t stream) {
  KVC_RANGE();
  return topk_compact_impl("kvc_topk_compact", scores, K, V, kv, k, protect_tail, live_mask, largest, idx, K_out,
                           V_out, nullptr, 0, nullptr, nullptr, 0, stream);
}

kvc_status kvc_topk_compact_channels(const float* scores, const kvc_bf16* K, const kvc_bf16* V,
                                     const kvc_kv_desc* kv, int32_t k, int32_t protect_tail,
                                     const uint32_t* live_mask, int32_t largest, int32_t* idx, kvc_bf16* K_out,
                                     kvc_bf16* V_out, const kvc_bf16* q_win, int32_t w, float* channel_scores,
                                     void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  if (!channel_scores) return fail(KVC_ERR_INVALID_ARG, "kvc_topk_compact_channels: channel_scores is NULL");
  KVC_TRY(check_desc(kv, "kvc_topk_compact_channels"));
  return topk_compact_impl("kvc_topk_compact_channels", scores, K, V, kv, k, protect_tail, live_mask, largest, idx,
                           K_out, V_out, q_win, w, channel_scores, ws, ws_bytes, stream);
}

// kvc_compress_prefill, and with channel_scores also ThinK's key-channel scores of the kept
// keys, summed by the compaction as it reads them (kvc_compress_prefill_channels)
static kvc_status compress_prefill_impl(const char* who, const kvc_bf16* q_win, const kvc_bf16* K,
                                        const kvc_bf16* V, const kvc_kv_desc* kv, int32_t w, float scale,
                                        kvc_head_reduce reduce, int32_t k, int32_t protect_tail, float* scores,
                                        int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out, float* channel_scores,
                                        void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_TRY(check_desc(kv, who));
  if (k < 1) return fail(KVC_ERR_INVALID_ARG, "%s: k must be >= 1", who);
  KVC_TRY(check_window(kv, w, who));
  if (protect_tail < 0 || protect_tail > k || protect_tail > w)
    return fail(KVC_ERR_INVALID_ARG, "%s: need 0 <= protect_tail <= min(k, w)", who);
  if (reduce != KVC_REDUCE_GQA_GROUP && reduce != KVC_REDUCE_ALL_HEADS)
    return fail(KVC_ERR_INVALID_ARG, "unknown head reduction");
  if (!(scale > 0.f) || scale != scale) return fail(KVC_ERR_INVALID_ARG, "scale must be > 0");
  KVC_TRY(check_ptr(q_win, "q_win"));
  KVC_TRY(check_gather(K, V, kv, k, K_out, V_out, who));
  if (kv->S > topk_max_len()) return fail(KVC_ERR_UNSUPPORTED, "%s: S > %lld", who, (long long)topk_max_len());
  KVC_TRY(check_ptr(idx, "idx"));
  if (scores && !aligned16(scores)) return fail(KVC_ERR_INVALID_ARG, "scores is not 16-byte aligned");
  if (channel_scores && !aligned16(channel_scores))
    return fail(KVC_ERR_INVALID_ARG, "channel_scores is not 16-byte aligned");
  {  // no output may overlap another output or an input
    const uintptr_t osz = (uintptr_t)kv->B * kv->KVH * (uintptr_t)k * kv->D * 2;
    const uintptr_t ko = reinterpret_cast<uintptr_t>(K_out), vo = reinterpret_cast<uintptr_t>(V_out);
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(idx), i1 = i0 + (uintptr_t)kv->B * kv->KVH * k * 4;
    uintptr_t k0, k1, v0 = 0, v1 = 0;
    cache_range(K, *kv, &k0, &k1);
    if (V) cache_range(V, *kv, &v0, &v1);
    if (overlaps(i0, i1, ko, ko + osz) || (V_out && overlaps(i0, i1, vo, vo + osz)) || overlaps(i0, i1, k0, k1) ||
        (V && overlaps(i0, i1, v0, v1)))
      return fail(KVC_ERR_INVALID_ARG, "%s: idx overlaps another argument", who);
    if (scores) {
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(scores), s1 = s0 + (uintptr_t)kv->B * kv->KVH * kv->S * 4;
      if (overlaps(s0, s1, ko, ko + osz) || (V_out && overlaps(s0, s1, vo, vo + osz)) || overlaps(s0, s1, i0, i1) ||
          overlaps(s0, s1, k0, k1) || (V && overlaps(s0, s1, v0, v1)))
        return fail(KVC_ERR_INVALID_ARG, "%s: scores overlaps another argument", who);
    }
    if (channel_scores) {
      const uintptr_t c0 = reinterpret_cast<uintptr_t>(channel_scores),
                      c1 = c0 + (uintptr_t)kv->B * kv->KVH * kv->D * 4;
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(scores), s1 = s0 + (uintptr_t)kv->B * kv->KVH * kv->S * 4;
      if (overlaps(c0, c1, ko, ko + osz) || (V_out && overlaps(c0, c1, vo, vo + osz)) || overlaps(c0, c1, i0, i1) ||
          overlaps(c0, c1, k0, k1) || (V && overlaps(c0, c1, v0, v1)) || (scores && overlaps(c0, c1, s0, s1)))
        return fail(KVC_ERR_INVALID_ARG, "%s: channel_scores overlaps another argument", who);
    }
  }
  // short rows: one fused kernel (scores, selection and compaction per (b, kvh); no workspace)
  if (!channel_scores && prefill_fused_supported(*kv, w, k, reduce))
    return cuda_status(launch_prefill_fused(q_win, K, V, *kv, w, scale, reduce, k, protect_tail, scores, idx, K_out,
                                            V_out, (cudaStream_t)stream),
                       "kvc_compress_prefill launch");
  // otherwise: window scores (into `scores`, or into the workspace when scores is NULL), then
  // selection and compaction; the channel partials follow the scores in the workspace
  const size_t sc_need = (scores_workspace(*kv, w, reduce) + 255) / 256 * 256;
  const size_t sc_room = ((size_t)kv->B * kv->KVH * kv->S * sizeof(float) + 255) / 256 * 256;
  const size_t need = sc_need + (scores ? 0 : sc_room) + (channel_scores ? compact_channels_workspace(*kv, k) : 0);
  KVC_TRY(check_ws(ws, ws_bytes, need, who));
  float* sc = scores ? scores : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sc_need);
  KVC_TRY(kvc_window_scores(q_win, K, kv, w, scale, 1, nullptr, reduce, sc, ws, sc_need, stream));
  if (!channel_scores) return kvc_topk_compact(sc, K, V, kv, k, protect_tail, nullptr, 1, idx, K_out, V_out, stream);
  const size_t used = sc_need + (scores ? 0 : sc_room);
  return topk_compact_impl(who, sc, K, V, kv, k, protect_tail, nullptr, 1, idx, K_out, V_out, q_win, w,
                           channel_scores, static_cast<uint8_t*>(ws) + used, ws_bytes - used, stream);
}

kvc_status kvc_compress_prefill(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_bf16* V,
                                const kvc_kv_desc* kv, int32_t w, float scale,
                                kvc_head_reduce reduce, int32_t k, int32_t protect_tail,
                                float* scores, int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out,
                                void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  return compress_prefill_impl("kvc_compress_prefill", q_win, K, V, kv, w, scale, reduce, k, protect_tail, scores,
                               idx, K_out, V_out, nullptr, ws, ws_bytes, stream);
}

kvc_status kvc_compress_prefill_channels(const kvc_bf16* q_win, const kvc_bf16* K, const kvc_bf16* V,
                                         const kvc_kv_desc* kv, int32_t w, float scale,
                                         kvc_head_reduce reduce, int32_t k, int32_t protect_tail,
                                         float* scores, int32_t* idx, kvc_bf16* K_out, kvc_bf16* V_out,
                                         float* channel_scores, void* ws, size_t ws_bytes,
                                         kvc_stream_t stream) {
  KVC_RANGE();
  if (!channel_scores) return fail(KVC_ERR_INVALID_ARG, "kvc_compress_prefill_channels: channel_scores is NULL");
  return compress_prefill_impl("kvc_compress_prefill_channels", q_win, K, V, kv, w, scale, reduce, k, protect_tail,
                               scores, idx, K_out, V_out, channel_scores, ws, ws_bytes, stream);
}

kvc_status kvc_write_slots(const kvc_bf16* k_new, const kvc_bf16* v_new, const int32_t* slot,
                           kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_write_slots"));
  KVC_TRY(check_ptr(k_new, "k_new"));
  KVC_TRY(check_ptr(K, "K"));
  if (!slot) return fail(KVC_ERR_INVALID_ARG, "slot is NULL");
  if ((v_new == nullptr) != (V == nullptr)) return fail(KVC_ERR_INVALID_ARG, "v_new and V must both be given or both NULL");
  if (V) {
    KVC_TRY(check_ptr(v_new, "v_new"));
    KVC_TRY(check_ptr(V, "V"));
  }
  return cuda_status(launch_write_slots(k_new, v_new, slot, K, V, *kv, (cudaStream_t)stream), "kvc_write_slots launch");
}

kvc_status kvc_tova_decode_step(const kvc_bf16* q_new, const kvc_bf16* k_new,
                                const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V,
                                const kvc_kv_desc* kv, float scale, int32_t* free_slot,
                                float* scores, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_tova_decode_step"));
  if (!free_slot) return fail(KVC_ERR_INVALID_ARG, "free_slot is NULL");
  KVC_TRY(check_ptr(scores, "scores"));
  KVC_TRY(check_ws(ws, ws_bytes, scores_workspace(*kv, 1, KVC_REDUCE_ALL_HEADS), "kvc_tova_decode_step"));
  KVC_TRY(check_ptr(q_new, "q_new"));
  KVC_TRY(check_ptr(k_new, "k_new"));
  KVC_TRY(check_ptr(K, "K"));
  if ((v_new == nullptr) != (V == nullptr)) return fail(KVC_ERR_INVALID_ARG, "v_new and V must both be given or both NULL");
  if (V) KVC_TRY(check_ptr(v_new, "v_new"));
  {
    const cudaError_t e = launch_tova_decode(q_new, k_new, v_new, K, V, *kv, scale, free_slot, scores, ws,
                                             (cudaStream_t)stream);
    if (e != cudaErrorNotSupported) return cuda_status(e, "kvc_tova_decode_step launch");
    // (returned by the planner, not by the runtime: the shapes take the general kernels below)
  }
  KVC_TRY(kvc_write_slots(k_new, v_new, free_slot, K, V, kv, stream));
  KVC_TRY(kvc_window_scores(q_new, K, kv, 1, scale, 0, nullptr, KVC_REDUCE_ALL_HEADS, scores, ws, ws_bytes, stream));
  return kvc_topk_select(scores, kv->B, kv->KVH, kv->S, 1, 0, nullptr, 0, free_slot, nullptr, 0, stream);
}

kvc_status kvc_scissorhands_init(kvc_sh_state* st, int32_t n_live, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_sh(st));
  if (n_live < 0 || n_live > st->cap) return fail(KVC_ERR_INVALID_ARG, "scissorhands_init: n_live in [0, cap]");
  st->t = 0;
  st->n_free = st->cap - n_live;
  return cuda_status(launch_sh_init(*st, n_live, (cudaStream_t)stream), "kvc_scissorhands_init launch");
}

kvc_status kvc_scissorhands_update_from_probs(kvc_sh_state* st, const float* p, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_sh(st));
  KVC_TRY(check_ptr(p, "p"));
  const kvc_status s = cuda_status(launch_sh_record(*st, p, (cudaStream_t)stream), "scissorhands record launch");
  if (s == KVC_OK) st->t += 1;
  return s;
}

namespace {
// Validation shared by the insertion entry points; `queue` (nullable) with m and pos.
kvc_status check_sh_insert(const kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos,
                           const kvc_bf16* k_new, const kvc_bf16* v_new, const kvc_bf16* K, const kvc_bf16* V,
                           const kvc_kv_desc* kv, const char* name) {
  KVC_TRY(check_sh(st));
  KVC_TRY(check_desc(kv, name));
  if (kv->B != st->B || kv->KVH != st->KVH || kv->S != st->cap)
    return fail(KVC_ERR_INVALID_ARG, "%s: cache shape does not match the state", name);
  if (queue) {
    if (m < 1 || m > st->cap) return fail(KVC_ERR_INVALID_ARG, "%s: queue length m in [1, cap]", name);
    if (pos < 0 || pos >= m) return fail(KVC_ERR_INVALID_ARG, "%s: queue position in [0, m)", name);
  } else if (st->n_free <= 0) {
    return fail(KVC_ERR_INVALID_ARG, "%s: no free slot (evict first, or give a queue)", name);
  }
  KVC_TRY(check_ptr(k_new, "k_new"));
  KVC_TRY(check_ptr(K, "K"));
  if ((v_new == nullptr) != (V == nullptr)) return fail(KVC_ERR_INVALID_ARG, "v_new and V must both be given or both NULL");
  return KVC_OK;
}

kvc_status sh_insert(kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos, const kvc_bf16* k_new,
                     const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv, kvc_stream_t stream) {
  KVC_TRY(cuda_status(launch_sh_insert(*st, queue, m, pos, k_new, v_new, K, V, *kv, (cudaStream_t)stream),
                      "scissorhands insert launch"));
  if (!queue) st->n_free -= 1;  // a queued slot is replaced, not filled
  return KVC_OK;
}

kvc_status sh_update(kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos, const kvc_bf16* q_new,
                     const kvc_bf16* k_new, const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv,
                     float scale, float* probs, void* ws, size_t ws_bytes, kvc_stream_t stream, const char* name) {
  KVC_TRY(check_sh_insert(st, queue, m, pos, k_new, v_new, K, V, kv, name));
  KVC_TRY(check_ptr(q_new, "q_new"));
  KVC_TRY(check_ptr(probs, "probs"));
  KVC_TRY(check_ws(ws, ws_bytes, scores_workspace(*kv, 1, KVC_REDUCE_GQA_GROUP), name));
  {  // insert, score and record in one launch where the small-row scoring kernel applies
    const cudaError_t e = launch_sh_update_fused(*st, queue, m, pos, q_new, k_new, v_new, K, V, *kv, scale, probs, ws,
                                                 (cudaStream_t)stream);
    if (e != cudaErrorNotSupported) {
      KVC_TRY(cuda_status(e, "scissorhands update launch"));
      if (!queue) st->n_free -= 1;
      st->t += 1;
      return KVC_OK;
    }
  }
  KVC_TRY(sh_insert(st, queue, m, pos, k_new, v_new, K, V, kv, stream));
  KVC_TRY(kvc_window_scores(q_new, K, kv, 1, scale, 0, st->live, KVC_REDUCE_GQA_GROUP, probs, ws, ws_bytes, stream));
  return kvc_scissorhands_update_from_probs(st, probs, stream);
}
}  // namespace

kvc_status kvc_scissorhands_update(kvc_sh_state* st, const kvc_bf16* q_new, const kvc_bf16* k_new,
                                   const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V,
                                   const kvc_kv_desc* kv, float scale, float* probs, void* ws,
                                   size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  return sh_update(st, nullptr, 0, 0, q_new, k_new, v_new, K, V, kv, scale, probs, ws, ws_bytes, stream,
                   "kvc_scissorhands_update");
}

kvc_status kvc_scissorhands_update_queued(kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos,
                                          const kvc_bf16* q_new, const kvc_bf16* k_new, const kvc_bf16* v_new,
                                          kvc_bf16* K, kvc_bf16* V, const kvc_kv_desc* kv, float scale,
                                          float* probs, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  if (!queue) return fail(KVC_ERR_INVALID_ARG, "kvc_scissorhands_update_queued: queue is NULL");
  return sh_update(st, queue, m, pos, q_new, k_new, v_new, K, V, kv, scale, probs, ws, ws_bytes, stream,
                   "kvc_scissorhands_update_queued");
}

kvc_status kvc_scissorhands_insert(kvc_sh_state* st, const int32_t* queue, int32_t m, int32_t pos,
                                   const kvc_bf16* k_new, const kvc_bf16* v_new, kvc_bf16* K, kvc_bf16* V,
                                   const kvc_kv_desc* kv, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_sh_insert(st, queue, m, pos, k_new, v_new, K, V, kv, "kvc_scissorhands_insert"));
  return sh_insert(st, queue, m, pos, k_new, v_new, K, V, kv, stream);
}

kvc_status kvc_scissorhands_refill_queue(kvc_sh_state* st, int32_t m, int32_t* queue, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_sh(st));
  if (m < 1 || m > st->cap || m > SH_QUEUE_MAX)
    return fail(KVC_ERR_INVALID_ARG, "scissorhands_refill_queue: m in [1, min(cap, %d)]", SH_QUEUE_MAX);
  if (st->t < 1) return fail(KVC_ERR_INVALID_ARG, "scissorhands_refill_queue: no step recorded yet");
  if (!queue) return fail(KVC_ERR_INVALID_ARG, "queue is NULL");
  return cuda_status(launch_sh_queue(*st, m, queue, (cudaStream_t)stream), "scissorhands queue launch");
}

kvc_status kvc_scissorhands_evict(kvc_sh_state* st, int32_t m, int32_t* evicted, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_sh(st));
  if (m < 1 || m > st->cap) return fail(KVC_ERR_INVALID_ARG, "scissorhands_evict: m in [1, cap]");
  if (st->t < 1) return fail(KVC_ERR_INVALID_ARG, "scissorhands_evict: no step recorded yet");
  if (!evicted) return fail(KVC_ERR_INVALID_ARG, "evicted is NULL");
  const kvc_status s = cuda_status(launch_sh_evict(*st, m, evicted, (cudaStream_t)stream), "scissorhands evict launch");
  if (s == KVC_OK) st->n_free = std::min(st->cap, st->n_free + m);
  return s;
}

kvc_status kvc_channel_score(const kvc_bf16* q_win, int32_t w, const kvc_bf16* K,
                             const kvc_kv_desc* kv, const int32_t* idx, int32_t k, float* cs,
                             void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_channel_score"));
  if (w < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_score: w must be >= 1");
  if (idx && k < 1) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_score: k must be >= 1 with idx");
  KVC_TRY(check_ptr(q_win, "q_win"));
  KVC_TRY(check_ptr(K, "K"));
  if (!cs) return fail(KVC_ERR_INVALID_ARG, "cs is NULL");
  const size_t need = channel_score_workspace(*kv, idx ? k : 0, idx != nullptr);
  KVC_TRY(check_ws(ws, ws_bytes, need, "kvc_channel_score"));
  {
    uintptr_t in[4][2];
    cache_range(K, *kv, &in[0][0], &in[0][1]);
    in[1][0] = reinterpret_cast<uintptr_t>(q_win);
    in[1][1] = in[1][0] + (uintptr_t)kv->B * kv->H * w * kv->D * 2;
    in[2][0] = reinterpret_cast<uintptr_t>(ws);
    in[2][1] = in[2][0] + need;
    in[3][0] = reinterpret_cast<uintptr_t>(idx);
    in[3][1] = idx ? in[3][0] + (uintptr_t)kv->B * kv->KVH * k * 4 : in[3][0];
    KVC_TRY(check_out_apart(cs, (size_t)kv->B * kv->KVH * kv->D * 4, in, 4, "kvc_channel_score: cs"));
  }
  return cuda_status(launch_channel_score(q_win, w, K, *kv, idx, idx ? k : 0, cs, ws, (cudaStream_t)stream),
                     "kvc_channel_score launch");
}

kvc_status kvc_channel_prune(const float* cs, const kvc_bf16* K, const kvc_kv_desc* kv,
                             int32_t C, int32_t zero_mode, int32_t* ch_idx, kvc_bf16* K_out,
                             kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_channel_prune"));
  if (C < 1 || C > kv->D) return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: need 1 <= C <= D");
  if (!zero_mode && C % 8) return fail(KVC_ERR_UNSUPPORTED, "kvc_channel_prune: compact mode needs C %% 8 == 0");
  if (!cs || !ch_idx) return fail(KVC_ERR_INVALID_ARG, "cs and ch_idx must be given");
  KVC_TRY(check_ptr(K, "K"));
  KVC_TRY(check_ptr(K_out, "K_out"));
  uintptr_t k0, k1;
  cache_range(K, *kv, &k0, &k1);
  const uintptr_t ko = reinterpret_cast<uintptr_t>(K_out);
  const uintptr_t osz = (uintptr_t)kv->B * kv->KVH * (uintptr_t)kv->S * (zero_mode ? kv->D : C) * 2;
  if (zero_mode) {
    const bool dense = kv->stride_s == kv->D && kv->stride_h == kv->S * kv->D && kv->stride_b == kv->KVH * kv->S * kv->D;
    if (!(ko == k0 && dense) && overlaps(ko, ko + osz, k0, k1))
      return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: K_out overlaps K (in place needs K_out == K, dense)");
  } else if (overlaps(ko, ko + osz, k0, k1)) {
    return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: K_out overlaps K");
  }
  // every CTA of a row reads the row's scores and its keys while the row's first CTA writes
  // the channel list, so the list may share no bytes with cs, K or K_out
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(ch_idx), c1 = c0 + (uintptr_t)kv->B * kv->KVH * C * 4;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(cs), s1 = s0 + (uintptr_t)kv->B * kv->KVH * kv->D * 4;
  if (overlaps(c0, c1, s0, s1) || overlaps(c0, c1, k0, k1) || overlaps(c0, c1, ko, ko + osz))
    return fail(KVC_ERR_INVALID_ARG, "kvc_channel_prune: ch_idx overlaps cs, K or K_out");
  return cuda_status(launch_channel_prune(cs, K, *kv, C, zero_mode ? 1 : 0, ch_idx, K_out, (cudaStream_t)stream),
                     "kvc_channel_prune launch");
}

kvc_status kvc_value_channel_score(const kvc_bf16* q_win, int32_t w, const kvc_bf16* Kc, const kvc_bf16* Vc,
                                   const kvc_kv_desc* kv, float scale, float* cs, void* ws, size_t ws_bytes,
                                   kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kv, "kvc_value_channel_score"));
  KVC_TRY(check_window(kv, w, "kvc_value_channel_score"));
  KVC_TRY(check_ptr(q_win, "q_win"));
  KVC_TRY(check_ptr(Kc, "Kc"));
  KVC_TRY(check_ptr(Vc, "Vc"));
  if (!cs) return fail(KVC_ERR_INVALID_ARG, "cs is NULL");
  if (!(scale > 0.f) || scale != scale) return fail(KVC_ERR_INVALID_ARG, "scale must be > 0");
  KVC_TRY(check_ws(ws, ws_bytes, value_score_workspace(*kv, w), "kvc_value_channel_score"));
  {  // cs is written while the partials in ws are read, and must leave the caches intact
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(cs), c1 = c0 + (uintptr_t)kv->B * kv->KVH * kv->D * 4;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(ws), w1 = w0 + value_score_workspace(*kv, w);
    uintptr_t k0, k1, v0, v1;
    cache_range(Kc, *kv, &k0, &k1);
    cache_range(Vc, *kv, &v0, &v1);
    if (overlaps(c0, c1, w0, w1) || overlaps(c0, c1, k0, k1) || overlaps(c0, c1, v0, v1))
      return fail(KVC_ERR_INVALID_ARG, "kvc_value_channel_score: cs overlaps ws, Kc or Vc");
  }
  // the window's attention over the compressed cache, squared and summed over the window
  // rows (mean over the group): one weight per kept token, then the weighted sums of V^2
  uint8_t* base = static_cast<uint8_t*>(ws);
  size_t wts_off = 0, part_off = 0;
  value_score_workspace(*kv, w, &wts_off, &part_off);
  float* wts = reinterpret_cast<float*>(base + wts_off);
  void* part = base + part_off;
  KVC_TRY(cuda_status(launch_window_scores(q_win, Kc, *kv, w, scale, 1, nullptr, KVC_REDUCE_GQA_GROUP, wts, base,
                                           (cudaStream_t)stream, 2),
                      "kvc_value_channel_score weights launch"));
  return cuda_status(launch_weighted_channel_norm(wts, Vc, *kv, cs, part, (cudaStream_t)stream),
                     "kvc_value_channel_score launch");
}

kvc_status kvc_decode_attention(const kvc_bf16* q, const int32_t* ch, const kvc_bf16* K, const kvc_kv_desc* kd,
                                const kvc_bf16* V, const kvc_kv_desc* vd, const uint32_t* live_mask, float scale,
                                float* out, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(kd, "kvc_decode_attention (K)"));
  KVC_TRY(check_desc(vd, "kvc_decode_attention (V)"));
  if (kd->B != vd->B || kd->H != vd->H || kd->KVH != vd->KVH || kd->S != vd->S)
    return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attention: K and V descriptors differ in B, H, KVH or S");
  if (!decode_shape_supported(kd->D, vd->D))
    return fail(KVC_ERR_UNSUPPORTED, "kvc_decode_attention: kept key channels must be 64 or 128 and <= D");
  if (!ch && kd->D != vd->D)
    return fail(KVC_ERR_INVALID_ARG, "kvc_decode_attention: without a channel list K must keep all D channels");
  if (kd->stride_s != kd->D || vd->stride_s != vd->D)
    return fail(KVC_ERR_UNSUPPORTED, "kvc_decode_attention: K and V rows must be dense (stride_s == channels)");
  if ((int64_t)kd->B * kd->KVH > 65535) return fail(KVC_ERR_UNSUPPORTED, "kvc_decode_attention: B * KVH must be <= 65535");
  KVC_TRY(check_ptr(q, "q"));
  KVC_TRY(check_ptr(K, "K"));
  KVC_TRY(check_ptr(V, "V"));
  KVC_TRY(check_ptr(out, "out"));
  if (ch && !aligned16(ch)) return fail(KVC_ERR_INVALID_ARG, "ch not 16-byte aligned");
  if (live_mask && !aligned16(live_mask)) return fail(KVC_ERR_INVALID_ARG, "live_mask not 16-byte aligned");
  if (!(scale > 0.f) || scale != scale) return fail(KVC_ERR_INVALID_ARG, "scale must be > 0");
  const size_t need = plan_decode(*vd).part_bytes;
  KVC_TRY(check_ws(ws, ws_bytes, need, "kvc_decode_attention"));
  {
    uintptr_t in[5][2];
    cache_range(K, *kd, &in[0][0], &in[0][1]);
    cache_range(V, *vd, &in[1][0], &in[1][1]);
    in[2][0] = reinterpret_cast<uintptr_t>(q);
    in[2][1] = in[2][0] + (uintptr_t)vd->B * vd->H * vd->D * 2;
    in[3][0] = reinterpret_cast<uintptr_t>(ws);
    in[3][1] = in[3][0] + need;
    in[4][0] = reinterpret_cast<uintptr_t>(ch);
    in[4][1] = ch ? in[4][0] + (uintptr_t)kd->B * kd->KVH * kd->D * 4 : in[4][0];
    KVC_TRY(check_out_apart(out, (size_t)vd->B * vd->H * vd->D * 4, in, 5, "kvc_decode_attention: out"));
  }
  return cuda_status(launch_decode_attention(q, ch, K, *kd, V, *vd, live_mask, scale, out, ws, (cudaStream_t)stream),
                     "kvc_decode_attention launch");
}

kvc_status kvc_zero_add_back(const kvc_bf16* Kp, const kvc_kv_desc* pd, const int32_t* ch, kvc_bf16* K_out,
                             const kvc_kv_desc* od, kvc_stream_t stream) {
  KVC_RANGE();
  KVC_TRY(check_desc(pd, "kvc_zero_add_back (Kp)"));
  KVC_TRY(check_desc(od, "kvc_zero_add_back (K_out)"));
  if (pd->B != od->B || pd->KVH != od->KVH || pd->S != od->S)
    return fail(KVC_ERR_INVALID_ARG, "kvc_zero_add_back: Kp and K_out descriptors differ in B, KVH or S");
  if (pd->D > od->D) return fail(KVC_ERR_INVALID_ARG, "kvc_zero_add_back: more kept channels than D");
  if ((int64_t)od->B * od->KVH > 65535) return fail(KVC_ERR_UNSUPPORTED, "kvc_zero_add_back: B * KVH must be <= 65535");
  KVC_TRY(check_ptr(Kp, "Kp"));
  KVC_TRY(check_ptr(K_out, "K_out"));
  KVC_TRY(check_ptr(ch, "ch"));
  uintptr_t p0, p1, o0, o1;
  cache_range(Kp, *pd, &p0, &p1);
  cache_range(K_out, *od, &o0, &o1);
  if (overlaps(p0, p1, o0, o1)) return fail(KVC_ERR_INVALID_ARG, "kvc_zero_add_back: K_out overlaps Kp");
  return cuda_status(launch_zero_add_back(Kp, *pd, ch, K_out, *od, (cudaStream_t)stream), "kvc_zero_add_back launch");
}

kvc_status kvc_host_device_pointer(const void* host_ptr, void** dev_ptr) {
  KVC_RANGE();
  if (!host_ptr || !dev_ptr) return fail(KVC_ERR_INVALID_ARG, "kvc_host_device_pointer: NULL argument");
  *dev_ptr = nullptr;
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, host_ptr);
  if (e != cudaSuccess || at.type != cudaMemoryTypeHost) {
    cudaGetLastError();  // the query's own error, if any: not a failure of earlier work
    return fail(KVC_ERR_INVALID_ARG, "kvc_host_device_pointer: not page-locked host memory");
  }
  e = cudaHostGetDevicePointer(dev_ptr, const_cast<void*>(host_ptr), 0);
  if (e != cudaSuccess || *dev_ptr == nullptr) {
    cudaGetLastError();
    *dev_ptr = nullptr;
    return fail(KVC_ERR_INVALID_ARG, "kvc_host_device_pointer: host memory not mapped for the device");
  }
  return KVC_OK;
}

kvc_status kvc_get_device_status(kvc_stream_t stream) {
  KVC_RANGE();
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "kvc_get_device_status sync");
  cudaError_t (*takers[])(unsigned int*) = {take_status_scores,       take_status_scores_tc, take_status_select,
                                            take_status_gather,       take_status_scissorhands, take_status_decode,
                                            take_status_prefill,      take_status_scores_stream};
  unsigned int first = 0u;
  for (auto fn : takers) {
    unsigned int v = 0u;
    e = fn(&v);
    if (e != cudaSuccess) return cuda_status(e, "kvc_get_device_status read");
    if (first == 0u) first = v;
  }
  if (first != 0u) return fail((kvc_status)first, "device status: %s", kvc_status_string((kvc_status)first));
  return KVC_OK;
}

}  // extern "C"
