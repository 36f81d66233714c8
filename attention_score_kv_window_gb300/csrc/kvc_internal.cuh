// Internal declarations shared by the libkvc translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvc.h"

namespace kvc {

// Sticky device status: the first kernel that meets a bad index or gives up a bounded wait
// records its code here; kvc_get_device_status() reads and clears it.  Each translation
// unit has its own word (no relocatable device code needed); KVC_TU_STATUS(name) defines
// the host function take_status_<name>() that reads and clears it.
namespace {
__device__ unsigned int g_device_status = 0u;
__device__ __forceinline__ void set_device_status(unsigned int code) {
  atomicCAS(&g_device_status, 0u, code);
}
inline cudaError_t take_tu_status(unsigned int* v) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess || *v == 0u) return e;
  const unsigned int z = 0u;
  return cudaMemcpyToSymbol(g_device_status, &z, sizeof(unsigned int));
}
}  // namespace
#define KVC_TU_STATUS(name) \
  cudaError_t take_status_##name(unsigned int* v) { return take_tu_status(v); }
cudaError_t take_status_scores(unsigned int* v);
cudaError_t take_status_select(unsigned int* v);
cudaError_t take_status_gather(unsigned int* v);
cudaError_t take_status_scissorhands(unsigned int* v);
cudaError_t take_status_scores_tc(unsigned int* v);
cudaError_t take_status_prefill(unsigned int* v);
cudaError_t take_status_scores_stream(unsigned int* v);

// Programmatic dependent launch.  Kernels launched with pdl_config() may start before the
// previous kernel on the stream has finished; each such kernel calls pdl_wait() before its
// first global-memory access (it returns once the previous kernel has completed and its
// writes are visible; it returns at once when there is nothing to wait for).  pdl_trigger()
// lets the next kernel's launch begin once every CTA of this grid has called it or exited;
// kernels that do not call it release the next one when they exit.  Early triggers pay where
// the next kernel's CTAs start on SMs this grid leaves free (top-k after scoring, compaction
// after top-k); in chains of small kernels they only crowd the running grid.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Launch configuration with programmatic stream serialisation and, when cluster_x > 1, a
// cluster shape.  `attrs` must outlive the launch call.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t st, cudaLaunchAttribute* attrs,
                                     int cluster_x = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cfg;
}

// Launch `kern` with programmatic stream serialisation (see pdl_config).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(grid, block, smem, st, attrs);
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Once per kernel and device: prefer the largest shared-memory carveout (consecutive kernels
// of a call then do not make the SM change its L1 / shared split) and, above 48 KB, allow
// `max_dynamic_smem` bytes of dynamic shared memory.  `fn` is the kernel's address.
cudaError_t func_attrs_once(const void* fn, int max_dynamic_smem);

// Host-side helpers
int num_sms();                      // SM count of the current device (cached per device)
// Count n kernels just enqueued (reported by kvc_launch_count) and return the launch status.
cudaError_t launched(int n);
void set_error(const char* fmt, ...);  // records the thread's last error message

// ----------------------------------------------------------------------------------------
// window scores (kvc_scores.cu)
// ----------------------------------------------------------------------------------------
struct ScoresArgs {
  const uint16_t* q;
  const uint16_t* K;
  int64_t sb, sh, ss;
  int B, H, KVH, w, G, R, Rpad;
  int64_t S;
  int causal;
  const uint32_t* live;
  int64_t live_words;
  float sl2;  // scale * log2(e)
  float pw;   // pass 2 sums p^pw over the query rows (1: scores; 2: value-channel weights)
  int nsplit;    // key ranges per (b, kvh)
  int64_t units; // 128-key units per (b, kvh); range s covers units [s*units/nsplit, (s+1)*units/nsplit)
  float* part;   // [B*KVH][nsplit][Rpad]  log2-domain log-sum-exp of a key range per query row (-inf: no key)
  float* mrow;   // [B*KVH][Rpad]          M2 + log2(L)  (+inf: no visible key)
  float* out;    // [B*KVH][S]
  float out_mul; // 1/G
  unsigned long long* sync;  // fused tensor-core kernel: epoch word + one tag per CTA (may be null)
  unsigned long long wait_ns;  // tensor-core kernel: bound on any single wait (2 s)
  int64_t withhold;            // fused tensor-core kernel: CTA whose key-range arrival a test leaves out (-1)
  // Decode step with the new token written on the fly (small-row kernel only; wslot null
  // otherwise): slot wslot[b*KVH+kvh] holds the new key knew[b*KVH+kvh] (its stale cache row
  // is never read), and the CTA whose slice holds it stores knew / vnew into Kw / Vw there.
  const int32_t* wslot;
  const uint16_t* knew;
  const uint16_t* vnew;
  uint16_t* Kw;
  uint16_t* Vw;
  // Scissorhands step fused into the small-row kernel (shs.B > 0): the new token takes the
  // lowest free slot, or slot queue[(b*KVH+kvh)*qm + qpos] when queue is given, and the
  // step's low-attention flags are recorded into the state as kvc_scissorhands.cu does.
  kvc_sh_state shs;
  const int32_t* queue;
  int qm, qpos;
};

// Partial of query row r from key range `split` (m + log2 l over the range's keys): one
// range's rows are contiguous (a range writes them coalesced; the merge reads whole sectors)
__host__ __device__ __forceinline__ int64_t part_index(const ScoresArgs& a, int bk, int r, int split) {
  return ((int64_t)bk * a.nsplit + split) * a.Rpad + r;
}
#ifdef __CUDACC__
// log2-domain log-sum-exp of a key range for one query row, from its running (max, sum)
__device__ __forceinline__ float range_lse(float m, float l) { return l > 0.f ? m + log2f(l) : -__int_as_float(0x7f800000); }
// Row r's normaliser over all key ranges, log2 domain: log2 of the sum of 2^lse over the
// ranges; +inf when the row sees no key.  Loads are issued eight at a time and bypass L1
// (other CTAs of the same launch may have written the partials).
__device__ __forceinline__ float merge_row(const ScoresArgs& a, int bk, int r) {
  float M = -__int_as_float(0x7f800000), Ls = 0.f;
  for (int s0 = 0; s0 < a.nsplit; s0 += 8) {
    float o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      o[q] = (s0 + q < a.nsplit) ? __ldcg(a.part + part_index(a, bk, r, s0 + q)) : -__int_as_float(0x7f800000);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (o[q] != -__int_as_float(0x7f800000)) {
        if (o[q] > M) {
          Ls = Ls * exp2f(M - o[q]) + 1.f;
          M = o[q];
        } else {
          Ls += exp2f(o[q] - M);
        }
      }
    }
  }
  return Ls > 0.f ? M + log2f(Ls) : __int_as_float(0x7f800000);
}
#endif

constexpr int KEY_UNIT = 128;
// keys [*kbeg, *kend) of key range `split` (balanced: ranges differ by at most one unit)
__host__ __device__ __forceinline__ void key_range(const ScoresArgs& a, int split, int64_t* kbeg, int64_t* kend) {
  const int64_t u0 = (int64_t)split * a.units / a.nsplit;
  const int64_t u1 = (int64_t)(split + 1) * a.units / a.nsplit;
  *kbeg = u0 * KEY_UNIT;
  const int64_t e = u1 * KEY_UNIT;
  *kend = e < a.S ? e : a.S;
}

// tcgen05 (TMEM/TMA) scoring (kvc_scores_tc.cu).  tc_supported() tells whether the shapes
// fit it; launch_scores_tc() runs both passes, fused in one cooperative launch when a.sync is
// set and the grid fits on the GPU at once, else as two launches.
bool tc_supported(const ScoresArgs& a, int D);
// kvc_debug_inject_timeout: arm (1) or disarm (0) the timeout test of the next fused launch
void inject_scores_timeout(int armed);
// TMA map of a [B, KVH, S, D] bf16 cache: boxes of 64 channels x box_rows rows (<= 256),
// 128-byte swizzle (row r's 16-byte chunk c of a 64-channel panel lands at chunk c ^ (r & 7));
// false when the strides cannot be described
bool make_cache_tensor_map(const uint16_t* K, const kvc_kv_desc& kv, CUtensorMap* tm, int box_rows);
cudaError_t launch_scores_tc(const ScoresArgs& a, int D, cudaStream_t st);

struct ScoresPlan {
  int R;         // query rows per (b,kvh): G*w
  int Rpad;      // padded to the kernel's row tile
  int nsplit;    // key ranges per (b,kvh)
  int64_t units; // 128-key units per (b,kvh)
  size_t part_bytes;   // (m,l) partials
  size_t sync_bytes;   // fused tensor-core kernel: epoch word + one tag per CTA
  size_t group_bytes;  // per-group scores for the all-heads reduction
};
ScoresPlan plan_scores(const kvc_kv_desc& kv, int w, int reduce);
size_t scores_workspace(const kvc_kv_desc& kv, int w, int reduce);
// device address of the fixed scratch array behind kvc_window_scores_noalloc (per device)
cudaError_t noalloc_scratch(void** out);
cudaError_t launch_window_scores(const uint16_t* q, const uint16_t* K, const kvc_kv_desc& kv, int w,
                                 float scale, int causal, const uint32_t* live, int reduce,
                                 float* scores, void* ws, cudaStream_t st, int power = 1);
// One TOVA decode step as three kernels: the new token written into slot free_slot[b,kvh]
// while the small-row kernel scores all slots with it, then the all-heads mean of the group
// scores fused with the eviction (argmin) that overwrites free_slot.  cudaErrorNotSupported
// when the shapes need another scoring kernel.
cudaError_t launch_tova_decode(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                               const kvc_kv_desc& kv, float scale, int32_t* free_slot, float* scores, void* ws,
                               cudaStream_t st);
// TMA-streamed decode-step scoring (kvc_scores_stream.cu), one launch each; the new token's
// rows are written into its slot (free_slot / the Scissorhands slot search) on the way.
// cudaErrorNotSupported when the shapes do not fit (more than 8 query rows per KV head,
// head_dim not 64/128, a slice's logits beyond shared memory, strides a tensor map cannot
// describe).  group_scores: [B*KVH][S] group-mean probabilities.
cudaError_t launch_decode_scores_stream(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K,
                                        uint16_t* V, const kvc_kv_desc& kv, float scale, const int32_t* free_slot,
                                        float* group_scores, cudaStream_t st);
// A whole TOVA decode step in one streamed kernel (scores, all-heads mean, eviction) when the
// head clusters fit; cudaErrorNotSupported otherwise.
cudaError_t launch_tova_step_stream(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K,
                                    uint16_t* V, const kvc_kv_desc& kv, float scale, int32_t* free_slot, float* scores,
                                    cudaStream_t st);
cudaError_t launch_sh_update_stream(const kvc_sh_state& sh, const int32_t* queue, int qm, int qpos, const uint16_t* q,
                                    const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                                    const kvc_kv_desc& kv, float scale, float* probs, cudaStream_t st);
// One Scissorhands decode step (insert, score, record) as one small-row kernel launch;
// cudaErrorNotSupported when the shapes need another scoring kernel.
cudaError_t launch_sh_update_fused(const kvc_sh_state& s, const int32_t* queue, int qm, int qpos, const uint16_t* q,
                                   const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                                   const kvc_kv_desc& kv, float scale, float* probs, void* ws, cudaStream_t st);
// value-channel score: cs[b,kvh,d] = sum_j wts[b,kvh,j] * V[b,kvh,j,d]^2 (kvc_gather.cu); ws holds
// channel_score_workspace(kv, 0, false) bytes of partials
cudaError_t launch_weighted_channel_norm(const float* wts, const uint16_t* V, const kvc_kv_desc& kv, float* cs,
                                         void* ws, cudaStream_t st);

// ----------------------------------------------------------------------------------------
// fused prefill compression for short rows (kvc_prefill.cu): scores, top-k and compaction of
// one (b, kvh) per CTA, K read once into shared memory.  Supported when G*w <= 16, the key
// block fits shared memory (S <= 1024 at 64 channels, 512 at 128), k <= S rounded up to 64
// and, in all-heads mode, KVH <= 8.  cudaErrorNotSupported otherwise.
// ----------------------------------------------------------------------------------------
bool prefill_fused_supported(const kvc_kv_desc& kv, int w, int k, int reduce);
cudaError_t launch_prefill_fused(const uint16_t* q, const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv, int w,
                                 float scale, int reduce, int k, int protect, float* scores, int32_t* idx,
                                 uint16_t* Ko, uint16_t* Vo, cudaStream_t st);

// ----------------------------------------------------------------------------------------
// selection (kvc_select.cu)
// ----------------------------------------------------------------------------------------
int64_t topk_max_len();  // longest row kvc_topk_select accepts
cudaError_t launch_topk(const float* scores, int B, int KVH, int64_t S, int k, int protect_tail,
                        const uint32_t* live, int largest, int32_t* idx, cudaStream_t st);
cudaError_t launch_sh_evict(const kvc_sh_state& s, int m, int32_t* evicted, cudaStream_t st);
constexpr int SH_QUEUE_MAX = 2048;  // longest eviction queue launch_sh_queue sorts
cudaError_t launch_sh_queue(const kvc_sh_state& s, int m, int32_t* queue, cudaStream_t st);

// ----------------------------------------------------------------------------------------
// gathers (kvc_gather.cu)
// ----------------------------------------------------------------------------------------
cudaError_t launch_compact(const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv,
                           const int32_t* idx, int k, uint16_t* Ko, uint16_t* Vo, cudaStream_t st);
cudaError_t launch_write_slots(const uint16_t* kn, const uint16_t* vn, const int32_t* slot,
                               uint16_t* K, uint16_t* V, const kvc_kv_desc& kv, cudaStream_t st);
size_t channel_score_workspace(const kvc_kv_desc& kv, int k, bool has_idx);
// compaction (as launch_compact) that also writes the ThinK key-channel scores cs [B,KVH,D] of
// the kept keys; ws: compact_channels_workspace(kv, k) bytes
size_t compact_channels_workspace(const kvc_kv_desc& kv, int k);
cudaError_t launch_compact_channels(const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv, const int32_t* idx,
                                    int k, uint16_t* Ko, uint16_t* Vo, const uint16_t* q, int w, float* cs, void* ws,
                                    cudaStream_t st);
cudaError_t launch_channel_score(const uint16_t* q, int w, const uint16_t* K, const kvc_kv_desc& kv,
                                 const int32_t* idx, int k, float* cs, void* ws, cudaStream_t st);
cudaError_t launch_channel_prune(const float* cs, const uint16_t* K, const kvc_kv_desc& kv, int C,
                                 int zero_mode, int32_t* ch, uint16_t* Ko, cudaStream_t st);

// ----------------------------------------------------------------------------------------
// Scissorhands state kernels (kvc_scissorhands.cu)
// ----------------------------------------------------------------------------------------
cudaError_t launch_sh_init(const kvc_sh_state& s, int n_live, cudaStream_t st);
// queue == null: the lowest free slot; else the new token replaces slot queue[row * qm + qpos]
cudaError_t launch_sh_insert(const kvc_sh_state& s, const int32_t* queue, int qm, int qpos, const uint16_t* kn,
                             const uint16_t* vn, uint16_t* K, uint16_t* V, const kvc_kv_desc& kv, cudaStream_t st);
cudaError_t launch_sh_record(const kvc_sh_state& s, const float* p, cudaStream_t st);

}  // namespace kvc
