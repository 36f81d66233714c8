// Per-row selection: the k highest-ranked eligible items of one (b, kvh) row, written as
// ascending indices.  Ranking: higher key first; on equal keys the lower index first when
// keeping, the higher index first when evicting (the lowest-ranked token goes first).
//
// A row is split over a thread-block cluster of up to 8 CTAs (1024 threads each); each CTA
// loads its slice of keys into shared memory once.  An MSB-first radix select (digits of
// 11, 11 and 10 bits) builds shared-memory histograms with warp-aggregated atomics, sums
// them over the cluster through distributed shared memory, and finds the digit holding the
// k-th item with one block scan; this yields the k-th key T and how many keys equal to T
// are taken.  The output pass counts, per warp and per CTA, the keys certainly taken (> T)
// and those equal to T, exchanges the CTA counts over the cluster, and writes every taken
// index at (taken-for-sure before it) + (taken-equal before it): ascending order, no sort.
// Cluster barriers are hardware barriers; there are no spin-waits.
//
// Users: token top-k for SnapKV/TOVA ("Add TOVA press"; cold-compress PR 11, SnapKV keeps
// the observation window) and Scissorhands eviction by low-attention fraction.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

namespace cg = cooperative_groups;

constexpr int SEL_THREADS = 1024;
constexpr int64_t SLICE_MAX = 40960;  // keys one CTA keeps in shared memory
constexpr int MAX_CLUSTER = 8;

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
  uint32_t hist[2][2048];
  uint32_t warp_a[32];
  uint32_t warp_b[32];
  uint32_t cta_cnt[4];  // read by the other CTAs of the cluster: forced, eligible, sure, equal
  uint32_t prefix, remaining, eq_total;
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

template <class Fn>
__device__ void select_row(const Fn& fn, int64_t n, int k, int32_t* out, uint32_t* kc, SelShared& sh,
                           bool evict_order) {
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks();
  const int cr = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lower = (1u << lane) - 1u;
  // this CTA's slice [c0, c1) of the row, and this warp's contiguous segment [w0, w1) of it
  const int64_t per_cta = ((n + (int64_t)cs * 32 - 1) / ((int64_t)cs * 32)) * 32;
  const int64_t c0 = (int64_t)cr * per_cta;
  const int64_t c1 = c0 + per_cta < n ? c0 + per_cta : n;
  const int64_t len = c1 > c0 ? c1 - c0 : 0;
  const int64_t per_w = ((len + 1023) / 1024) * 32;
  const int64_t w0 = c0 + (int64_t)warp * per_w;
  const int64_t w1 = w0 + per_w < c1 ? w0 + per_w : c1;

  // keys of the slice into shared memory (independent loads, many in flight)
#pragma unroll 8
  for (int64_t j = c0 + tid; j < c1; j += SEL_THREADS) kc[j - c0] = fn.key(j);

  // 1. forced / eligible counts over the cluster
  uint32_t cf = 0, ce = 0;
  for (int64_t base = w0; base < w1; base += 32) {
    const int64_t j = base + lane;
    const bool in = j < w1;
    const bool f = in && fn.forced(j);
    const bool e = in && !f && fn.eligible(j);
    cf += __popc(__ballot_sync(0xffffffffu, f));
    ce += __popc(__ballot_sync(0xffffffffu, e));
  }
  if (lane == 0) {
    sh.warp_a[warp] = cf;
    sh.warp_b[warp] = ce;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, b = 0;
    for (int q = 0; q < 32; ++q) {
      a += sh.warp_a[q];
      b += sh.warp_b[q];
    }
    sh.cta_cnt[0] = a;
    sh.cta_cnt[1] = b;
  }
  cl.sync();
  uint32_t n_forced = 0, n_elig = 0;
  for (int r = 0; r < cs; ++r) {
    const SelShared* rs = cl.map_shared_rank(&sh, r);
    n_forced += rs->cta_cnt[0];
    n_elig += rs->cta_cnt[1];
  }
  const int64_t need = (int64_t)k - (int64_t)n_forced > 0 ? (int64_t)k - (int64_t)n_forced : 0;
  const bool take_all = (int64_t)n_elig <= need;
  const bool split_ties = !take_all && need > 0;

  // 2. radix select of the need-th largest eligible key over the cluster
  uint32_t T = 0, take_eq = 0, eq_total = 0;
  if (split_ties) {
    uint32_t prefix = 0, rem = (uint32_t)need, hi_mask = 0;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t nbins = pass == 2 ? 1024u : 2048u;
      uint32_t* hist = sh.hist[pass & 1];
      for (uint32_t i = tid; i < nbins; i += SEL_THREADS) hist[i] = 0u;
      __syncthreads();
      for (int64_t j0 = 0; j0 < len; j0 += SEL_THREADS) {
        const int64_t jl = j0 + tid;
        uint32_t d = 0xffffffffu;
        if (jl < len && fn.eligible(c0 + jl)) {
          const uint32_t key = kc[jl];
          if ((key & hi_mask) == prefix) d = (key >> shift) & (nbins - 1u);
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (d != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (uint32_t)__popc(peers));
      }
      cl.sync();
      // this thread's bins, in descending digit order, summed over the cluster
      const uint32_t bpt = nbins >> 10;
      uint32_t hb[2] = {0u, 0u};
      for (int r = 0; r < cs; ++r) {
        const uint32_t* rh = cl.map_shared_rank(hist, r);
        for (uint32_t q = 0; q < bpt; ++q) hb[q] += rh[nbins - 1u - (tid * bpt + q)];
      }
      const uint32_t hs = hb[0] + hb[1];
      uint32_t tot;
      const uint32_t incl = block_scan(hs, sh.warp_a, &tot);
      const uint32_t excl = incl - hs;
      if (excl < rem && rem <= incl) {
        uint32_t run = excl;
        for (uint32_t q = 0; q < bpt; ++q) {
          const uint32_t d = nbins - 1u - (tid * bpt + q);
          if (run + hb[q] >= rem) {
            sh.prefix = prefix | (d << shift);
            sh.remaining = rem - run;
            sh.eq_total = hb[q];
            break;
          }
          run += hb[q];
        }
      }
      __syncthreads();
      prefix = sh.prefix;
      rem = sh.remaining;
      hi_mask |= (nbins - 1u) << shift;
    }
    T = prefix;
    take_eq = rem;
    eq_total = sh.eq_total;
  }
  // keys equal to T: the first take_eq in index order when keeping, the last when evicting
  const uint32_t skip_eq = evict_order ? (eq_total - take_eq) : 0u;

  // 3. output, ascending
  uint32_t cd = 0, cq = 0;
  for (int64_t base = w0; base < w1; base += 32) {
    const int64_t j = base + lane;
    bool def = false, eq = false;
    if (j < w1) {
      if (fn.forced(j)) def = true;
      else if (fn.eligible(j)) {
        if (take_all) def = true;
        else if (split_ties) {
          const uint32_t key = kc[j - c0];
          def = key > T;
          eq = key == T;
        }
      }
    }
    cd += __popc(__ballot_sync(0xffffffffu, def));
    cq += __popc(__ballot_sync(0xffffffffu, eq));
  }
  if (lane == 0) {
    sh.warp_a[warp] = cd;
    sh.warp_b[warp] = cq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, b = 0;
    for (int q = 0; q < 32; ++q) {
      a += sh.warp_a[q];
      b += sh.warp_b[q];
    }
    sh.cta_cnt[2] = a;
    sh.cta_cnt[3] = b;
  }
  cl.sync();
  uint32_t d_run = 0, e_run = 0, d_total = 0;
  for (int r = 0; r < cs; ++r) {
    const SelShared* rs = cl.map_shared_rank(&sh, r);
    const uint32_t a = rs->cta_cnt[2], b = rs->cta_cnt[3];
    if (r < cr) {
      d_run += a;
      e_run += b;
    }
    d_total += a;
  }
  for (int q = 0; q < warp; ++q) {
    d_run += sh.warp_a[q];
    e_run += sh.warp_b[q];
  }
  for (int64_t base = w0; base < w1; base += 32) {
    const int64_t j = base + lane;
    bool def = false, eq = false;
    if (j < w1) {
      if (fn.forced(j)) def = true;
      else if (fn.eligible(j)) {
        if (take_all) def = true;
        else if (split_ties) {
          const uint32_t key = kc[j - c0];
          def = key > T;
          eq = key == T;
        }
      }
    }
    const uint32_t bd = __ballot_sync(0xffffffffu, def);
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const uint32_t eb = e_run + __popc(be & lower);  // keys equal to T before j
    const bool take = def || (eq && eb >= skip_eq && eb < skip_eq + take_eq);
    if (take) {
      const uint32_t teq = eb <= skip_eq ? 0u : (eb - skip_eq < take_eq ? eb - skip_eq : take_eq);
      const uint32_t pos = d_run + __popc(bd & lower) + teq;
      if (pos < (uint32_t)k) out[pos] = (int32_t)j;
    }
    d_run += __popc(bd);
    e_run += __popc(be);
  }
  if (cr == 0) {
    const uint32_t total = d_total + (split_ties ? take_eq : 0u);
    for (int64_t p = (int64_t)total + tid; p < k; p += SEL_THREADS) out[p] = -1;
  }
  cl.sync();  // no CTA leaves while the others may still read its shared memory
}

__global__ void __launch_bounds__(SEL_THREADS) k_topk(const float* __restrict__ scores, int64_t S, int k,
                                                      int protect, const uint32_t* __restrict__ live,
                                                      int largest, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint32_t kc[];
  __shared__ SelShared sh;
  const int64_t row = blockIdx.x / cg::this_cluster().num_blocks();
  ScoreKeys fn;
  fn.row = scores + row * S;
  fn.lw = live ? live + row * ((S + 31) / 32) : nullptr;
  fn.S = S;
  fn.protect = protect;
  fn.largest = largest;
  select_row<ScoreKeys>(fn, S, k, idx + row * k, kc, sh, !largest);
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
  select_row<FractionKeys>(fn, s.cap, m, out, kc, sh, false);
  // clear the live bits of the evicted slots (select_row ended with a barrier)
  uint32_t* lw = s.live + row * nw;
  for (int p = threadIdx.x; p < m; p += SEL_THREADS) {
    const int32_t j = out[p];
    if (j >= 0 && j < s.cap) atomicAnd(lw + (j >> 5), ~(1u << (j & 31)));
  }
}

int topk_cluster_size(int64_t S) {
  if (S <= 8192) return 1;
  return (int)std::min<int64_t>(MAX_CLUSTER, (S + 4095) / 4096);
}

}  // namespace

int64_t topk_max_len() { return SLICE_MAX * MAX_CLUSTER; }

cudaError_t launch_topk(const float* scores, int B, int KVH, int64_t S, int k, int protect_tail,
                        const uint32_t* live, int largest, int32_t* idx, cudaStream_t st) {
  const int cs = topk_cluster_size(S);
  const int64_t per_cta = ((S + (int64_t)cs * 32 - 1) / ((int64_t)cs * 32)) * 32;
  if (per_cta > SLICE_MAX) return cudaErrorInvalidValue;
  const size_t smem = (size_t)per_cta * 4;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(SLICE_MAX * 4));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)B * KVH * cs), 1, 1);
  cfg.blockDim = dim3(SEL_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_topk, scores, S, k, protect_tail, live, largest, idx);
}

cudaError_t launch_sh_evict(const kvc_sh_state& s, int m, int32_t* evicted, cudaStream_t st) {
  const size_t smem = (size_t)s.cap * 4;
  if ((int64_t)s.cap > SLICE_MAX) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_sh_evict, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_sh_evict<<<s.B * s.KVH, SEL_THREADS, smem, st>>>(s, m, evicted);
  return cudaGetLastError();
}

KVC_TU_STATUS(select)

}  // namespace kvc
