// Scissorhands state kernels (cold-compress PR 11, "Implement Scissorhands KV-cache
// compression & SnapKV prompt compression"): slot insertion (into a free slot, or over the
// next token of an eviction queue), and the circular history of
// "attention < 1/keys" flags kept as bit planes, one plane per step, with a running count
// of low flags per slot.  Eviction by low-attention fraction lives with the selection code.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void k_sh_init(kvc_sh_state s, int n_live) {
  pdl_wait();  // previous kernel on the stream complete and visible
  const int64_t rows = (int64_t)s.B * s.KVH;
  const int64_t nw = s.cap / 32;
  const int64_t n_hist = (int64_t)s.history * rows * nw;
  const int64_t n_slots = rows * s.cap;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t x0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (int64_t x = x0; x < n_hist; x += stride) s.hist[x] = 0u;
  for (int64_t x = x0; x < n_slots; x += stride) {
    s.low_count[x] = 0;
    s.insert_step[x] = 0;
  }
  for (int64_t x = x0; x < rows * nw; x += stride) {
    const int64_t w = x % nw;
    const int64_t lo = w * 32;
    uint32_t v;
    if (lo + 32 <= n_live) v = 0xffffffffu;
    else if (lo >= n_live) v = 0u;
    else v = (1u << (uint32_t)(n_live - lo)) - 1u;
    s.live[x] = v;
  }
  for (int64_t x = x0; x < rows; x += stride) s.slot[x] = -1;
}

// One warp per (b,kvh): pick the slot (the lowest free one, or with a queue the slot
// queue[row][pos], whose token is replaced), mark it live with a fresh insert step and no low
// flags, and copy the new K/V row into it.
template <int D>
__global__ void k_sh_insert(kvc_sh_state s, const int32_t* __restrict__ queue, int qm, int qpos,
                            const uint16_t* __restrict__ kn, const uint16_t* __restrict__ vn, uint16_t* K,
                            uint16_t* V, int64_t sb, int64_t sh, int64_t ss) {
  pdl_wait();  // previous kernel on the stream complete and visible
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= s.B * s.KVH) return;
  const int nw = s.cap / 32;
  uint32_t* lw = s.live + (int64_t)row * nw;
  int found = -1;
  if (queue) {
    const int32_t q = queue[(int64_t)row * qm + qpos];
    // a queued slot must hold a live token
    if (q >= 0 && q < s.cap && ((lw[q >> 5] >> (q & 31)) & 1u)) found = q;
  } else {
    for (int base = 0; base < nw; base += 32) {
      const uint32_t w = (base + lane < nw) ? lw[base + lane] : 0xffffffffu;
      const uint32_t bal = __ballot_sync(0xffffffffu, w != 0xffffffffu);
      if (bal) {
        const int f = __ffs(bal) - 1;
        const uint32_t word = __shfl_sync(0xffffffffu, w, f);
        found = (base + f) * 32 + (__ffs(~word) - 1);
        break;
      }
    }
  }
  if (found < 0) {
    if (lane == 0) set_device_status(KVC_ERR_DEVICE_BOUNDS);
    return;
  }
  __syncwarp();  // every lane has read the live word before lane 0 may change it
  if (lane == 0) {
    lw[found >> 5] |= 1u << (found & 31);
    s.insert_step[(int64_t)row * s.cap + found] = (int32_t)s.t;
    s.low_count[(int64_t)row * s.cap + found] = 0;
    s.slot[row] = found;
  }
  constexpr int TPR = D / 8;
  if (lane < TPR) {
    const int64_t b = row / s.KVH, kvh = row % s.KVH;
    const int64_t off = b * sb + kvh * sh + (int64_t)found * ss + lane * 8;
    *reinterpret_cast<uint4*>(K + off) = *reinterpret_cast<const uint4*>(kn + (int64_t)row * D + lane * 8);
    if (V) *reinterpret_cast<uint4*>(V + off) = *reinterpret_cast<const uint4*>(vn + (int64_t)row * D + lane * 8);
  }
}

// CTA (x, row) flags slots [256x, 256x + 256) of (b,kvh) row `row` for step t into plane
// t % history and updates their low counts; each CTA counts the row's live keys itself.
__global__ void __launch_bounds__(256) k_sh_record(kvc_sh_state s, const float* __restrict__ p) {
  pdl_wait();  // previous kernel on the stream complete and visible
  __shared__ uint32_t red[8];
  const int row = blockIdx.y;
  const int nw = s.cap / 32;
  const uint32_t* lw = s.live + (int64_t)row * nw;
  uint32_t cnt = 0;
  for (int w = threadIdx.x; w < nw; w += blockDim.x) cnt += __popc(lw[w]);
#pragma unroll
  for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  uint32_t keys = 0;
  for (int q = 0; q < (int)(blockDim.x >> 5); ++q) keys += red[q];
  // threshold: float32(1) / float32(keys), correctly rounded
  const float thr = __fdiv_rn(1.0f, (float)(keys > 0 ? keys : 1));
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= s.cap) return;  // cap % 32 == 0: whole warps leave together
  const int64_t plane = s.t % s.history;
  uint32_t* hp = s.hist + (plane * s.B * s.KVH + row) * (int64_t)nw;
  const int64_t x = (int64_t)row * s.cap + j;
  const int lane = threadIdx.x & 31, wi = j >> 5;
  const uint32_t lword = lw[wi];
  const bool live = (lword >> lane) & 1u;
  const bool flag = live && (p[x] < thr);
  const uint32_t bits = __ballot_sync(0xffffffffu, flag);
  const uint32_t old = hp[wi];
  if (live) {
    const bool old_valid = (s.t - (int64_t)s.insert_step[x]) >= (int64_t)s.history;
    const int oldbit = (old_valid && ((old >> lane) & 1u)) ? 1 : 0;
    s.low_count[x] = (uint16_t)((int)s.low_count[x] + (flag ? 1 : 0) - oldbit);
  }
  __syncwarp();
  if (lane == 0) hp[wi] = bits;
}

}  // namespace

cudaError_t launch_sh_init(const kvc_sh_state& s, int n_live, cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.KVH;
  const int64_t n = std::max<int64_t>((int64_t)s.history * rows * (s.cap / 32), rows * s.cap);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8));
  const cudaError_t e = launch_pdl(k_sh_init, dim3(blocks), dim3(256), 0, st, s, n_live);
  if (e != cudaSuccess) return e;
  return launched(1);
}

cudaError_t launch_sh_insert(const kvc_sh_state& s, const int32_t* queue, int qm, int qpos, const uint16_t* kn,
                             const uint16_t* vn, uint16_t* K, uint16_t* V, const kvc_kv_desc& kv, cudaStream_t st) {
  const int rows = s.B * s.KVH;
  const int blocks = (rows + 7) / 8;
  const cudaError_t e =
      kv.D == 64
          ? launch_pdl(k_sh_insert<64>, dim3(blocks), dim3(256), 0, st, s, queue, qm, qpos, kn, vn, K, V,
                       kv.stride_b, kv.stride_h, kv.stride_s)
          : launch_pdl(k_sh_insert<128>, dim3(blocks), dim3(256), 0, st, s, queue, qm, qpos, kn, vn, K, V,
                       kv.stride_b, kv.stride_h, kv.stride_s);
  if (e != cudaSuccess) return e;
  return launched(1);
}

cudaError_t launch_sh_record(const kvc_sh_state& s, const float* p, cudaStream_t st) {
  const cudaError_t e = launch_pdl(k_sh_record, dim3((s.cap + 255) / 256, s.B * s.KVH), dim3(256), 0, st, s, p);
  if (e != cudaSuccess) return e;
  return launched(1);
}

KVC_TU_STATUS(scissorhands)

}  // namespace kvc
