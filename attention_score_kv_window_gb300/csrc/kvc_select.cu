// Per-row selection: the k highest-ranked eligible items of one (b, kvh) row, written as
// ascending indices.  Ranking: higher key first; on equal keys the lower index first when
// keeping, the higher index first when evicting (the lowest-ranked token goes first).
//
// One 1024-thread CTA per row runs an MSB-first radix select over 32-bit order-preserving
// keys (4 digits of 8 bits, shared-memory histograms), which yields the k-th key T and how
// many items equal to T are taken.  A final pass in index order, with two block-wide scans
// (items equal to T, then chosen items), writes the chosen indices ascending.  Rows of up
// to 40960 items keep their keys in shared memory between passes; longer rows re-read
// global memory (they stay in L2).
//
// Users: token top-k for SnapKV/TOVA ("Add TOVA press"; cold-compress PR 11, SnapKV keeps
// the observation window) and Scissorhands eviction by low-attention fraction.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_ITEMS = 4;                 // consecutive items per thread in the output pass
constexpr int64_t SEL_CACHE_MAX = 40960;     // rows up to this length cache keys in smem

__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// token scores as keys (keep: larger score first; evict: smaller score first)
struct ScoreKeys {
  const float* row;
  const uint32_t* lw;  // live words of the row or null
  int64_t S;
  int64_t protect;     // tail positions forced in (keep only)
  int largest;
  __device__ __forceinline__ bool live(int64_t j) const {
    return lw == nullptr || ((__ldg(lw + (j >> 5)) >> (j & 31)) & 1u);
  }
  __device__ __forceinline__ bool forced(int64_t j) const { return j >= S - protect && live(j); }
  __device__ __forceinline__ bool eligible(int64_t j) const { return j < S - protect && live(j); }
  __device__ __forceinline__ uint32_t key(int64_t j) const {
    const uint32_t k = float_key(__ldg(row + j));
    return largest ? k : ~k;
  }
};

// Scissorhands: low-attention fraction low/n_obs as an exact integer key.  Two different
// fractions with denominators <= 4096 differ by at least 1/4096^2 = 2^-24, so
// floor(low * 2^31 / n_obs) keeps their order strictly, and equal fractions get equal keys.
struct FractionKeys {
  const uint16_t* low;
  const int32_t* ins;
  const uint32_t* lw;
  int64_t t_last;
  int history;
  __device__ __forceinline__ bool live(int64_t j) const { return (lw[j >> 5] >> (j & 31)) & 1u; }
  __device__ __forceinline__ bool forced(int64_t) const { return false; }
  __device__ __forceinline__ bool eligible(int64_t j) const { return live(j); }
  __device__ __forceinline__ uint32_t key(int64_t j) const {
    int64_t n = t_last - (int64_t)ins[j] + 1;
    n = n < 1 ? 1 : (n > history ? history : n);
    uint64_t c = low[j];
    if (c > (uint64_t)n) c = (uint64_t)n;
    return (uint32_t)((c << 31) / (uint64_t)n);
  }
};

struct SelShared {
  uint32_t hist[256];
  uint32_t warp_a[32];
  uint32_t warp_b[32];
  uint32_t prefix, remaining, eq_total, n_forced, n_elig, digit_above;
};

// inclusive block scan of one value per thread (1024 threads); returns inclusive, total in *tot
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* warp_buf, uint32_t* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_buf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_buf[lane] = w;
  }
  __syncthreads();
  const uint32_t base = warp ? warp_buf[warp - 1] : 0u;
  *tot = warp_buf[31];
  __syncthreads();
  return base + x;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* warp_buf) {
  uint32_t tot;
  block_scan(v, warp_buf, &tot);
  return tot;
}

template <class Fn, bool CACHE>
__device__ void select_row(const Fn& fn, int64_t n, int k, int32_t* out, uint32_t* kc,
                           SelShared& sh, bool evict_order) {
  const int tid = threadIdx.x;
  // count eligible and forced items; optionally cache keys
  uint32_t ce = 0, cf = 0;
  for (int64_t j = tid; j < n; j += SEL_THREADS) {
    if (fn.forced(j)) ++cf;
    else if (fn.eligible(j)) ++ce;
    if (CACHE) kc[j] = fn.key(j);
  }
  const uint32_t n_forced = block_sum(cf, sh.warp_a);
  const uint32_t n_elig = block_sum(ce, sh.warp_a);
  const int64_t need = std::max<int64_t>(0, (int64_t)k - (int64_t)n_forced);
  const bool take_all = (int64_t)n_elig <= need;

  uint32_t T = 0, take_eq = 0, eq_total = 0;
  if (!take_all && need > 0) {
    if (tid == 0) { sh.prefix = 0; sh.remaining = (uint32_t)need; }
    uint32_t mask = 0;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) sh.hist[tid] = 0;
      __syncthreads();
      const uint32_t prefix = sh.prefix;
      for (int64_t j = tid; j < n; j += SEL_THREADS) {
        if (!fn.eligible(j)) continue;
        const uint32_t key = CACHE ? kc[j] : fn.key(j);
        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        const int lane = tid;
        uint32_t s = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) s += sh.hist[255 - 8 * lane - q];
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - s;
        const uint32_t rem = sh.remaining;
        if (excl < rem && rem <= incl) {
          uint32_t run = excl;
          for (int q = 0; q < 8; ++q) {
            const int d = 255 - 8 * lane - q;
            const uint32_t h = sh.hist[d];
            if (run + h >= rem) {
              sh.prefix = prefix | ((uint32_t)d << shift);
              sh.remaining = rem - run;
              sh.eq_total = h;
              break;
            }
            run += h;
          }
        }
      }
      __syncthreads();
      mask |= 255u << shift;
    }
    T = sh.prefix;
    take_eq = sh.remaining;
    eq_total = sh.eq_total;
  }
  // items equal to T are taken in index order when keeping (the first take_eq), and from
  // the end when evicting (the last take_eq)
  const uint32_t skip_eq = evict_order ? (eq_total - take_eq) : 0u;

  uint32_t eq_base = 0, out_base = 0;
  for (int64_t c0 = 0; c0 < n; c0 += (int64_t)SEL_THREADS * SEL_ITEMS) {
    const int64_t j0 = c0 + (int64_t)tid * SEL_ITEMS;
    uint8_t f[SEL_ITEMS];  // 1 = taken for sure, 2 = equal to T
    uint32_t neq = 0;
#pragma unroll
    for (int q = 0; q < SEL_ITEMS; ++q) {
      const int64_t j = j0 + q;
      f[q] = 0;
      if (j < n) {
        if (fn.forced(j)) f[q] = 1;
        else if (fn.eligible(j)) {
          if (take_all) f[q] = 1;
          else if (need > 0) {
            const uint32_t key = CACHE ? kc[j] : fn.key(j);
            if (key > T) f[q] = 1;
            else if (key == T) { f[q] = 2; ++neq; }
          }
        }
      }
    }
    uint32_t eq_tot;
    const uint32_t eq_incl = block_scan(neq, sh.warp_a, &eq_tot);
    uint32_t er = eq_base + eq_incl - neq;  // equal-rank of this thread's first equal item
    uint32_t nsel = 0;
#pragma unroll
    for (int q = 0; q < SEL_ITEMS; ++q) {
      if (f[q] == 2) {
        f[q] = (er >= skip_eq && er < skip_eq + take_eq) ? 1 : 0;
        ++er;
      }
      nsel += f[q];
    }
    uint32_t sel_tot;
    const uint32_t sel_incl = block_scan(nsel, sh.warp_b, &sel_tot);
    uint32_t pos = out_base + sel_incl - nsel;
#pragma unroll
    for (int q = 0; q < SEL_ITEMS; ++q) {
      if (f[q] == 1) {
        if (pos < (uint32_t)k) out[pos] = (int32_t)(j0 + q);
        ++pos;
      }
    }
    eq_base += eq_tot;
    out_base += sel_tot;
  }
  for (int64_t p = (int64_t)out_base + tid; p < k; p += SEL_THREADS) out[p] = -1;
}

template <bool CACHE>
__global__ void __launch_bounds__(SEL_THREADS) k_topk(const float* __restrict__ scores, int KVH,
                                                      int64_t S, int k, int protect,
                                                      const uint32_t* __restrict__ live,
                                                      int largest, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint32_t kc[];
  __shared__ SelShared sh;
  const int64_t row = blockIdx.x;
  ScoreKeys fn;
  fn.row = scores + row * S;
  fn.lw = live ? live + row * ((S + 31) / 32) : nullptr;
  fn.S = S;
  fn.protect = protect;
  fn.largest = largest;
  select_row<ScoreKeys, CACHE>(fn, S, k, idx + row * k, kc, sh, !largest);
}

__global__ void __launch_bounds__(SEL_THREADS) k_sh_evict(kvc_sh_state s, int m, int32_t* evicted) {
  extern __shared__ __align__(16) uint32_t kc[];
  __shared__ SelShared sh;
  const int64_t row = blockIdx.x;
  const int64_t nw = s.cap / 32;
  FractionKeys fn;
  fn.low = s.low_count + row * s.cap;
  fn.ins = s.insert_step + row * s.cap;
  fn.lw = s.live + row * nw;
  fn.t_last = s.t - 1;
  fn.history = s.history;
  int32_t* out = evicted + row * m;
  select_row<FractionKeys, true>(fn, s.cap, m, out, kc, sh, false);
  __syncthreads();
  // clear the live bits of the evicted slots
  uint32_t* lw = s.live + row * nw;
  for (int p = threadIdx.x; p < m; p += SEL_THREADS) {
    const int32_t j = out[p];
    if (j >= 0 && j < s.cap) atomicAnd(lw + (j >> 5), ~(1u << (j & 31)));
  }
}

}  // namespace

cudaError_t launch_topk(const float* scores, int B, int KVH, int64_t S, int k, int protect_tail,
                        const uint32_t* live, int largest, int32_t* idx, cudaStream_t st) {
  const int rows = B * KVH;
  if (S <= SEL_CACHE_MAX) {
    const size_t smem = (size_t)S * 4;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(k_topk<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(SEL_CACHE_MAX * 4));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    k_topk<true><<<rows, SEL_THREADS, smem, st>>>(scores, KVH, S, k, protect_tail, live, largest, idx);
  } else {
    k_topk<false><<<rows, SEL_THREADS, 0, st>>>(scores, KVH, S, k, protect_tail, live, largest, idx);
  }
  return cudaGetLastError();
}

cudaError_t launch_sh_evict(const kvc_sh_state& s, int m, int32_t* evicted, cudaStream_t st) {
  const size_t smem = (size_t)s.cap * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_sh_evict, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_sh_evict<<<s.B * s.KVH, SEL_THREADS, smem, st>>>(s, m, evicted);
  return cudaGetLastError();
}

KVC_TU_STATUS(select)

}  // namespace kvc
