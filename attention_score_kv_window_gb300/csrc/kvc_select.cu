// Per-row selection: the k highest-ranked eligible items of one (b, kvh) row, written as
// ascending indices.  Ranking: higher key first; on equal keys the lower index first when
// keeping, the higher index first when evicting (the lowest-ranked token goes first).
//
// A row is split over a thread-block cluster of up to 8 CTAs (1024 threads each); each CTA
// loads its slice of keys into shared memory once.  An MSB-first radix select with 8-bit
// digits starts below the bits that every candidate shares (the cluster's min and max key
// have them in common).  Each pass builds a shared-memory histogram with shared atomics, adds
// the nonzero bins into every peer's copy of the cluster histogram with remote reductions
// (pushes do not stall; remote loads would), and after one cluster barrier one warp finds
// the digit holding the k-th item and a block barrier hands it to the others.  This yields the k-th key T and how many keys equal
// to T are taken.  Each CTA's counts of keys taken for sure (> T) and of keys equal to T
// follow from its own histograms; they are pushed to every peer while the CTA ballots its
// keys, and every taken index is written at (taken-for-sure before it) + (taken-equal before
// it): ascending order, no sort.  Cluster barriers are hardware barriers; there are no
// spin-waits.
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

struct __align__(16) SelShared {
  uint32_t hist[2][256];  // this CTA's counts for the current digit (two, used alternately)
  uint32_t hsum[4][256];  // cluster sums per digit pass, filled by every CTA's pushes
  union {
    uint32_t ballots[SEL_THREADS / 32][40][2];  // output pass: (sure, equal) ballots per 32-key group
    uint64_t sortbuf[SH_QUEUE_MAX];            // the eviction queue's re-sort, after the selection
  };
  uint32_t cnt_all[MAX_CLUSTER][4];  // per CTA: forced, eligible, min and max eligible key
  uint32_t out_all[MAX_CLUSTER][2];  // per CTA: keys taken for sure, keys equal to the threshold
  uint32_t warp_a[32];
  uint32_t warp_b[32];
  uint32_t warp_c[32];
  uint32_t warp_d[32];
  uint32_t pick[3];  // the pass's digit, keys in higher bins, keys in its bin (warp 0 -> all)
};

// Writes into the shared memory of CTA `rank` of the cluster.  They do not stall the issuing
// thread; the next cluster barrier (release/acquire) makes them visible.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
               : "=r"(ra)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  return ra;
}
__device__ __forceinline__ void push_add(const uint32_t* local, int rank, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;\n" ::"r"(cluster_addr(local, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void push_v4(const uint32_t* local, int rank, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(cluster_addr(local, rank)), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void push_v2(const uint32_t* local, int rank, uint32_t x, uint32_t y) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};\n" ::"r"(cluster_addr(local, rank)), "r"(x), "r"(y)
               : "memory");
}
// The two halves of a cluster barrier; work placed between them overlaps its latency.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_barrier() {
  cluster_arrive();
  cluster_wait();
}

// The digit holding the rem-th largest candidate, from the 256 cluster-summed bins h (one
// warp).  Lane l takes the bins 255 - 8l down to 248 - 8l.  Returns the digit; *above =
// candidates in higher bins, *in_bin = its count.
__device__ __forceinline__ uint32_t pick_digit(const uint32_t* h, uint32_t rem, uint32_t* above, uint32_t* in_bin) {
  const int lane = threadIdx.x & 31;
  const uint4 a = *reinterpret_cast<const uint4*>(h + 248 - 8 * lane);
  const uint4 b = *reinterpret_cast<const uint4*>(h + 252 - 8 * lane);
  const uint32_t hv[8] = {b.w, b.z, b.y, b.x, a.w, a.z, a.y, a.x};  // descending digits
  uint32_t sum = 0u;
#pragma unroll
  for (int q = 0; q < 8; ++q) sum += hv[q];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t excl = incl - sum;
  uint32_t pick = 0u, run_at = 0u, cnt = 0u;
  if (excl < rem && rem <= incl) {
    uint32_t run = excl;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (run < rem && run + hv[q] >= rem) {
        pick = 255u - 8u * lane - q;
        run_at = run;
        cnt = hv[q];
      }
      run += hv[q];
    }
  }
  const uint32_t src = __ffs(__ballot_sync(0xffffffffu, excl < rem && rem <= incl)) - 1;
  *above = __shfl_sync(0xffffffffu, run_at, src);
  *in_bin = __shfl_sync(0xffffffffu, cnt, src);
  return __shfl_sync(0xffffffffu, pick, src);
}

// One row over the cluster.  Selection: the need-th largest eligible key is found digit by
// digit (8 bits each, most significant first), starting below the bits that every eligible
// key shares (the cluster's min and max key have them in common).  A pass histograms the
// candidates that match the prefix so far into shared memory, adds the nonzero bins into
// every CTA's cluster sum (remote reductions), and after one cluster barrier warp 0 scans
// the sums and a block barrier passes the digit on (every warp scanning them itself cost more
// in issue slots than the barrier).  One plain shared atomic per candidate: grouping a warp's
// equal digits with match.any first measured 2.5-4x slower even on the concentrated first
// digit.  The passes stop once every key of the chosen bin is taken.  Each
// CTA's counts of keys taken for sure and of keys equal to the threshold follow from its own
// histograms, so the last exchange (those counts) overlaps the local ballot pass.
template <class Fn>
__device__ void select_row(const Fn& fn, int64_t n, int k, int32_t* out, uint32_t* kc, SelShared& sh,
                           bool evict_order) {
  const int cs = (int)cg::this_cluster().num_blocks();
  const int cr = (int)cg::this_cluster().block_rank();
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

  // 0. clear what the peers add into, then announce it (the wait comes after the sweep)
  for (uint32_t i = tid; i < 4u * 256u; i += SEL_THREADS) (&sh.hsum[0][0])[i] = 0u;
  if (tid < 256) sh.hist[0][tid] = 0u;
  cluster_arrive();

  // 1. one sweep: keys into shared memory, forced / eligible counts, min and max eligible key
  uint32_t cf = 0, ce = 0, kmin = 0xffffffffu, kmax = 0u;
  constexpr int KB = 4;  // keys per thread whose loads are in flight together
  for (int64_t j0 = 0; j0 < len; j0 += KB * SEL_THREADS) {
    uint32_t key[KB];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int64_t jl = j0 + u * SEL_THREADS + tid;
      key[u] = jl < len ? fn.key(c0 + jl) : 0u;
    }
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int64_t jl = j0 + u * SEL_THREADS + tid;
      bool f = false, e = false;
      if (jl < len) {
        kc[jl] = key[u];
        f = fn.forced(c0 + jl);
        e = !f && fn.eligible(c0 + jl);
      }
      cf += __popc(__ballot_sync(0xffffffffu, f));
      ce += __popc(__ballot_sync(0xffffffffu, e));
      if (e) {
        kmin = min(kmin, key[u]);
        kmax = max(kmax, key[u]);
      }
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    sh.warp_a[warp] = cf;
    sh.warp_b[warp] = ce;
    sh.warp_c[warp] = kmin;
    sh.warp_d[warp] = kmax;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = __reduce_add_sync(0xffffffffu, sh.warp_a[lane]);
    const uint32_t b = __reduce_add_sync(0xffffffffu, sh.warp_b[lane]);
    const uint32_t lo = __reduce_min_sync(0xffffffffu, sh.warp_c[lane]);
    const uint32_t hi = __reduce_max_sync(0xffffffffu, sh.warp_d[lane]);
    cluster_wait();  // every peer has started and cleared its sums
    if (lane < cs) push_v4(&sh.cnt_all[cr][0], lane, make_uint4(a, b, lo, hi));
  } else {
    cluster_wait();
  }
  cluster_barrier();
  uint32_t n_forced = 0, n_elig = 0;
  kmin = 0xffffffffu;
  kmax = 0u;
  for (int r = 0; r < cs; ++r) {
    n_forced += sh.cnt_all[r][0];
    n_elig += sh.cnt_all[r][1];
    kmin = min(kmin, sh.cnt_all[r][2]);
    kmax = max(kmax, sh.cnt_all[r][3]);
  }
  const uint32_t my_forced = sh.cnt_all[cr][0], my_elig = sh.cnt_all[cr][1];
  const int64_t need = (int64_t)k - (int64_t)n_forced > 0 ? (int64_t)k - (int64_t)n_forced : 0;
  const bool take_all = (int64_t)n_elig <= need;
  const bool split_ties = !take_all && need > 0;

  // 2. radix select of the need-th largest eligible key; bits [hi, 32) are common to all
  int hi = 32 - __clz(kmin ^ kmax);
  uint32_t mask = hi == 32 ? 0u : ~((1u << hi) - 1u);
  uint32_t T = kmin & mask, rem = (uint32_t)need, in_bin = n_elig;
  uint32_t my_above = 0u, my_eq = my_elig;  // this CTA's keys above T's bin and in it (thread 0)
  if (split_ties) {
#pragma unroll 1
    for (int pass = 0; hi > 0 && rem != in_bin; ++pass) {
      const int lo = hi > 8 ? hi - 8 : 0;
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
      uint32_t* h = sh.hist[pass & 1];
      for (int64_t j0 = 0; j0 < len; j0 += SEL_THREADS) {  // (warp-uniform trip count)
        const int64_t jl = j0 + tid;
        uint32_t dg = 0xffffffffu;  // this lane's digit, or none
        if (jl < len && fn.eligible(c0 + jl)) {
          const uint32_t key = kc[jl];
          if ((key & mask) == T) dg = (key >> lo) & dmask;
        }
        if (dg != 0xffffffffu) atomicAdd(&h[dg], 1u);
      }
      __syncthreads();
      // add the nonzero bins into every CTA's sums; clear the other histogram (its last
      // readers finished before the barrier above) for the next digit
      for (int i = tid; i < 256 * cs; i += SEL_THREADS) {
        const uint32_t v = h[i & 255];
        if (v) push_add(&sh.hsum[pass][i & 255], i >> 8, v);
      }
      if (tid < 256) sh.hist[(pass + 1) & 1][tid] = 0u;
      cluster_barrier();
      if (warp == 0) {
        uint32_t above, cnt;
        const uint32_t d = pick_digit(sh.hsum[pass], rem, &above, &cnt);
        // this CTA's own keys in the higher bins and in the chosen one
        uint32_t s = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t dq = 8u * lane + q;
          s += dq > d ? h[dq] : 0u;
        }
        my_above += __reduce_add_sync(0xffffffffu, s);
        my_eq = h[d];
        if (lane == 0) {
          sh.pick[0] = d;
          sh.pick[1] = above;
          sh.pick[2] = cnt;
        }
      }
      __syncthreads();
      const uint32_t d = sh.pick[0], above = sh.pick[1], cnt = sh.pick[2];
      T |= d << lo;
      mask |= dmask << lo;
      rem -= above;
      in_bin = cnt;
      hi = lo;
    }
  }
  const uint32_t take_eq = split_ties ? rem : 0u, eq_total = split_ties ? in_bin : 0u;
  // keys equal to T (under mask): the first take_eq in index order when keeping, the last when
  // evicting
  const uint32_t skip_eq = evict_order ? (eq_total - take_eq) : 0u;

  // 3. output, ascending.  Counts to every peer, then the local ballots while the barrier
  // completes.
  if (tid == 0) {
    const uint32_t sure = my_forced + (take_all ? my_elig : (split_ties ? my_above : 0u));
    const uint32_t eq = split_ties ? my_eq : 0u;
    for (int r = 0; r < cs; ++r) push_v2(&sh.out_all[cr][0], r, sure, eq);
  }
  cluster_arrive();
  const int n_grp = (int)((w1 - w0 + 31) / 32);  // <= ceil(SLICE_MAX / 1024) = 40
  uint32_t cd = 0, cq = 0;
  for (int it = 0; it < n_grp; ++it) {
    const int64_t j = w0 + (int64_t)it * 32 + lane;
    bool def = false, eq = false;
    if (j < w1) {
      if (fn.forced(j)) def = true;
      else if (fn.eligible(j)) {
        if (take_all) def = true;
        else if (split_ties) {
          const uint32_t key = kc[j - c0] & mask;  // the digits the select decided
          def = key > T;
          eq = key == T;
        }
      }
    }
    const uint32_t bd = __ballot_sync(0xffffffffu, def), be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) {
      sh.ballots[warp][it][0] = bd;
      sh.ballots[warp][it][1] = be;
    }
    cd += __popc(bd);
    cq += __popc(be);
  }
  if (lane == 0) {
    sh.warp_a[warp] = cd;
    sh.warp_b[warp] = cq;
  }
  __syncthreads();
  uint32_t d_run = 0, e_run = 0;
  for (int q = 0; q < warp; ++q) {
    d_run += sh.warp_a[q];
    e_run += sh.warp_b[q];
  }
  cluster_wait();
  uint32_t d_total = 0;
  for (int r = 0; r < cs; ++r) {
    const uint32_t a = sh.out_all[r][0], b = sh.out_all[r][1];
    if (r < cr) {
      d_run += a;
      e_run += b;
    }
    d_total += a;
  }
  for (int it = 0; it < n_grp; ++it) {
    const int64_t j = w0 + (int64_t)it * 32 + lane;
    const uint32_t bd = sh.ballots[warp][it][0], be = sh.ballots[warp][it][1];
    const bool def = (bd >> lane) & 1u, eq = (be >> lane) & 1u;
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
    const uint32_t total = d_total + take_eq;
    for (int64_t p = (int64_t)total + tid; p < k; p += SEL_THREADS) out[p] = -1;
  }
  // no remote access follows the last cluster barrier, so CTAs may leave independently
}

__global__ void __launch_bounds__(SEL_THREADS) k_topk(const float* __restrict__ scores, int64_t S, int k,
                                                      int protect, const uint32_t* __restrict__ live,
                                                      int largest, int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint32_t kc[];
  __shared__ SelShared sh;
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  __syncthreads();  // the evicted list written by all threads is now visible to the block
  // clear the live bits of the evicted slots
  uint32_t* lw = s.live + row * nw;
  for (int p = threadIdx.x; p < m; p += SEL_THREADS) {
    const int32_t j = out[p];
    if (j >= 0 && j < s.cap) atomicAnd(lw + (j >> 5), ~(1u << (j & 31)));
  }
}

// Eviction queue: the m slots bulk eviction would take, listed most evictable first (higher
// fraction key first, ties to the lower slot).  The selection writes them in slot order; the
// block then re-sorts the m composites (key, ~slot) descending with a bitonic network in the
// histogram space the selection no longer needs.  Live bits are not touched.
__global__ void __launch_bounds__(SEL_THREADS) k_sh_queue(kvc_sh_state s, int m, int32_t* queue) {
  extern __shared__ __align__(16) uint32_t kc[];
  __shared__ SelShared sh;
  pdl_wait();
  const int64_t row = blockIdx.x;
  FractionKeys fn;
  fn.low = s.low_count + row * s.cap;
  fn.ins = s.insert_step + row * s.cap;
  fn.lw = s.live + row * (s.cap / 32);
  fn.t_last = s.t - 1;
  fn.history = s.history;
  int32_t* out = queue + row * m;
  select_row<FractionKeys>(fn, s.cap, m, out, kc, sh, false);
  __syncthreads();  // the slot-ordered list written by all threads is visible to the block
  uint64_t* ck = sh.sortbuf;
  int n2 = 1;
  while (n2 < m) n2 <<= 1;
  for (int p = threadIdx.x; p < n2; p += SEL_THREADS) {
    uint64_t c = 0;  // empty entries (-1) sort last
    if (p < m) {
      const int32_t j = out[p];
      if (j >= 0) c = ((uint64_t)fn.key(j) << 32) | (uint32_t)~(uint32_t)j;
    }
    ck[p] = c;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n2 >> 1); i += SEL_THREADS) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = ck[lo], y = ck[hi];
        if ((x < y) == desc) {
          ck[lo] = y;
          ck[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int p = threadIdx.x; p < m; p += SEL_THREADS) {
    const uint64_t c = ck[p];
    out[p] = c ? (int32_t)~(uint32_t)c : -1;
  }
}

// ----------------------------------------------------------------------------------------
// Short rows (S <= 4096, many of them: batched prefill instances, decode steps): one
// 256-thread CTA per row.  Each eligible item becomes the 64-bit composite (key, tie) with
// tie = ~index when keeping (lower index first) and index when evicting (higher index
// first), so composites are distinct and their descending order is the ranking.  k == 1 is
// a block max; otherwise a bitonic sort (descending) in shared memory gives the need-th
// composite, and every eligible item at or above it is taken, written in index order.
// ----------------------------------------------------------------------------------------
constexpr int SHORT_THREADS = 256;
constexpr int SHORT_MAX = 4096;

__device__ __forceinline__ uint64_t u64max(uint64_t a, uint64_t b) { return a > b ? a : b; }

__global__ void __launch_bounds__(SHORT_THREADS) k_topk_short(const float* __restrict__ scores, int S, int k,
                                                              int protect, const uint32_t* __restrict__ live,
                                                              int largest, int32_t* __restrict__ idx) {
  __shared__ uint64_t ck[SHORT_MAX];
  __shared__ uint32_t wsum[SHORT_THREADS / 32];
  __shared__ uint64_t wmax[SHORT_THREADS / 32];
  __shared__ uint32_t s_nforced, s_nelig;
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ScoreKeys fn;
  fn.row = scores + row * (int64_t)S;
  fn.lw = live ? live + row * (((int64_t)S + 31) / 32) : nullptr;
  fn.S = S;
  fn.protect = protect;
  fn.largest = largest;
  int32_t* out = idx + row * (int64_t)k;
  int n2 = 1;
  while (n2 < S) n2 <<= 1;

  // composites; ineligible and padding items are 0 (below every real composite)
  uint32_t cf = 0, ce = 0;
  uint64_t best = 0;
  for (int j = tid; j < n2; j += SHORT_THREADS) {
    uint64_t c = 0;
    if (j < S) {
      if (fn.forced(j)) ++cf;
      else if (fn.eligible(j)) {
        ++ce;
        c = ((uint64_t)fn.key(j) << 32) | (uint32_t)(largest ? ~(uint32_t)j : (uint32_t)j);
      }
    }
    ck[j] = c;
    best = u64max(best, c);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    cf += __shfl_xor_sync(0xffffffffu, cf, o);
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
    best = u64max(best, __shfl_xor_sync(0xffffffffu, best, o));
  }
  if (lane == 0) {
    wsum[warp] = cf | (ce << 16);  // S <= 4096: both counts fit 16 bits
    wmax[warp] = best;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t f = 0, e = 0;
    uint64_t bb = 0;
    for (int q = 0; q < SHORT_THREADS / 32; ++q) {
      f += wsum[q] & 0xffffu;
      e += wsum[q] >> 16;
      bb = u64max(bb, wmax[q]);
    }
    s_nforced = f;
    s_nelig = e;
    wmax[0] = bb;
  }
  __syncthreads();
  const int64_t need = (int64_t)k - (int64_t)s_nforced > 0 ? (int64_t)k - (int64_t)s_nforced : 0;
  const bool take_all = (int64_t)s_nelig <= need;
  uint64_t thr = 0;  // take eligible items with composite >= thr (0: take all eligible)
  if (!take_all && need > 0) {
    if (need == 1) {
      thr = wmax[0];
    } else {
      __syncthreads();
      for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int i = tid; i < (n2 >> 1); i += SHORT_THREADS) {
            const int lo = 2 * i - (i & (stride - 1));
            const int hi = lo + stride;
            const bool desc = (lo & size) == 0;  // overall descending order
            const uint64_t x = ck[lo], y = ck[hi];
            if ((x < y) == desc) {
              ck[lo] = y;
              ck[hi] = x;
            }
          }
          __syncthreads();
        }
      }
      thr = ck[need - 1];
    }
  }
  // output in index order: thread t owns a contiguous run of items
  const int per = (S + SHORT_THREADS - 1) / SHORT_THREADS;
  const int j0 = tid * per;
  uint32_t cnt = 0;
  for (int j = j0; j < j0 + per && j < S; ++j) {
    bool take = false;
    if (fn.forced(j)) take = true;
    else if (fn.eligible(j)) {
      if (take_all) take = true;
      else if (need > 0) {
        const uint64_t c = ((uint64_t)fn.key(j) << 32) | (uint32_t)(largest ? ~(uint32_t)j : (uint32_t)j);
        take = c >= thr;
      }
    }
    cnt += take;
  }
  // exclusive scan of the per-thread counts
  uint32_t x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t base = 0, total = 0;
  for (int q = 0; q < SHORT_THREADS / 32; ++q) {
    if (q < warp) base += wsum[q];
    total += wsum[q];
  }
  uint32_t pos = base + x - cnt;
  for (int j = j0; j < j0 + per && j < S; ++j) {
    bool take = false;
    if (fn.forced(j)) take = true;
    else if (fn.eligible(j)) {
      if (take_all) take = true;
      else if (need > 0) {
        const uint64_t c = ((uint64_t)fn.key(j) << 32) | (uint32_t)(largest ? ~(uint32_t)j : (uint32_t)j);
        take = c >= thr;
      }
    }
    if (take) {
      if (pos < (uint32_t)k) out[pos] = j;
      ++pos;
    }
  }
  for (int p = (int)total + tid; p < k; p += SHORT_THREADS) out[p] = -1;
}

// Rows of at most 32 * NU keys (batched short prefill instances): one warp per row, lane l
// holding keys l + 32 u in registers.  A radix select over the 32-bit ranking key (four 8-bit
// digits, a 256-bin histogram per warp in shared memory) finds the need-th key T and how many
// keys equal to T are taken (the first ones in index order when keeping, the last ones when
// evicting); the output pass walks u in order and places taken keys with ballots, so the
// indices come out ascending.
constexpr int WARP_ROWS_PER_CTA = 8;

template <int NU>
__global__ void __launch_bounds__(WARP_ROWS_PER_CTA * 32) k_topk_warp(const float* __restrict__ scores, int S, int k,
                                                                     int protect, const uint32_t* __restrict__ live,
                                                                     int largest, int32_t* __restrict__ idx,
                                                                     int64_t rows) {
  __shared__ uint32_t hist[WARP_ROWS_PER_CTA][256];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * WARP_ROWS_PER_CTA + warp;
  if (row >= rows) return;
  ScoreKeys fn;
  fn.row = scores + row * (int64_t)S;
  fn.lw = live ? live + row * (((int64_t)S + 31) / 32) : nullptr;
  fn.S = S;
  fn.protect = protect;
  fn.largest = largest;
  uint32_t key[NU];
  uint32_t elig = 0u, forc = 0u;  // bit u: key u of this lane is eligible / forced
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const int j = lane + 32 * u;
    key[u] = 0u;
    if (j < S) {
      if (fn.forced(j)) forc |= 1u << u;
      else if (fn.eligible(j)) {
        elig |= 1u << u;
        key[u] = fn.key(j);
      }
    }
  }
  int n_forced = __popc(forc), n_elig = __popc(elig);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    n_forced += __shfl_xor_sync(0xffffffffu, n_forced, o);
    n_elig += __shfl_xor_sync(0xffffffffu, n_elig, o);
  }
  const int need = k - n_forced > 0 ? k - n_forced : 0;
  const bool take_all = n_elig <= need;
  uint32_t T = 0u, prefix_mask = 0u;
  int take_eq = 0, eq_total = 0;
  if (!take_all && need > 0) {
    uint32_t* h = hist[warp];
    int rem = need;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
#pragma unroll
      for (int q = 0; q < 8; ++q) h[lane * 8 + q] = 0u;
      __syncwarp();
#pragma unroll
      for (int u = 0; u < NU; ++u)
        if (((elig >> u) & 1u) && (key[u] & prefix_mask) == T) atomicAdd(&h[(key[u] >> shift) & 255u], 1u);
      __syncwarp();
      // lane l scans bins 255 - 8 l ... 248 - 8 l (descending digits)
      uint32_t hb[8], tot = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        hb[q] = h[255 - 8 * lane - q];
        tot += hb[q];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - tot;
      const bool mine = excl < (uint32_t)rem && (uint32_t)rem <= incl;
      uint32_t digit = 0u, above = 0u, inbin = 0u;
      if (mine) {
        uint32_t run = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run + hb[q] >= (uint32_t)rem) {
            digit = 255u - 8u * lane - q;
            above = run;
            inbin = hb[q];
            break;
          }
          run += hb[q];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src);
      above = __shfl_sync(0xffffffffu, above, src);
      inbin = __shfl_sync(0xffffffffu, inbin, src);
      T |= digit << shift;
      prefix_mask |= 255u << shift;
      rem -= (int)above;
      eq_total = (int)inbin;
      __syncwarp();  // the histogram is read before the next pass clears it
    }
    take_eq = rem;
  }
  // equal keys: the first take_eq in index order when keeping, the last take_eq when evicting
  const int skip_eq = largest ? 0 : eq_total - take_eq;
  const bool split = !take_all && need > 0;
  int32_t* out = idx + row * (int64_t)k;
  const uint32_t lower = (1u << lane) - 1u;
  int pos = 0, eq_seen = 0;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const bool f = (forc >> u) & 1u;
    const bool e = (elig >> u) & 1u;
    const bool sure = f || (e && (take_all || (split && key[u] > T)));
    const bool eq = split && e && key[u] == T;
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const int eb = eq_seen + __popc(be & lower);
    const bool take = sure || (eq && eb >= skip_eq && eb < skip_eq + take_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int p = pos + __popc(bt & lower);
      if (p < k) out[p] = lane + 32 * u;
    }
    pos += __popc(bt);
    eq_seen += __popc(be);
  }
  for (int p = pos + lane; p < k; p += 32) out[p] = -1;
}

// k = 1 without a protected tail (a TOVA decode step evicts one slot per row): one 256-thread
// CTA per row takes the maximum of the same (key, tie) composites as k_topk_short, so the
// ranking is identical; -1 when nothing is eligible.  Finite scores give keys >= 1, so every
// eligible composite is above the empty value 0.
__global__ void __launch_bounds__(SHORT_THREADS) k_top1(const float* __restrict__ scores, int64_t S,
                                                        const uint32_t* __restrict__ live, int largest,
                                                        int32_t* __restrict__ idx) {
  __shared__ uint64_t wbest[SHORT_THREADS / 32];
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ScoreKeys fn;
  fn.row = scores + row * S;
  fn.lw = live ? live + row * ((S + 31) / 32) : nullptr;
  fn.S = S;
  fn.protect = 0;
  fn.largest = largest;
  uint64_t best = 0;
  for (int64_t j0 = 0; j0 < S; j0 += 4 * SHORT_THREADS) {
    uint64_t c[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t j = j0 + u * SHORT_THREADS + tid;
      c[u] = 0;
      if (j < S && fn.eligible(j))
        c[u] = ((uint64_t)fn.key(j) << 32) | (uint32_t)(largest ? ~(uint32_t)j : (uint32_t)j);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) best = u64max(best, c[u]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) best = u64max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) wbest[warp] = best;
  __syncthreads();
  if (tid == 0) {
    for (int q = 0; q < SHORT_THREADS / 32; ++q) best = u64max(best, wbest[q]);
    idx[row] = best ? (int32_t)(largest ? ~(uint32_t)best : (uint32_t)best) : -1;
  }
}

// CTAs per row: a power of two (the histogram exchange splits 1024 or 2048 bins evenly)
int topk_cluster_size(int64_t S) {
  int cs = 1;
  while (cs < MAX_CLUSTER && S > (int64_t)cs * 4096) cs *= 2;
  return cs;
}

}  // namespace

int64_t topk_max_len() { return SLICE_MAX * MAX_CLUSTER; }

cudaError_t launch_topk(const float* scores, int B, int KVH, int64_t S, int k, int protect_tail,
                        const uint32_t* live, int largest, int32_t* idx, cudaStream_t st) {
  if (k == 1 && protect_tail == 0) {
    const cudaError_t e =
        launch_pdl(k_top1, dim3((unsigned)((int64_t)B * KVH)), dim3(SHORT_THREADS), 0, st, scores, S, live, largest, idx);
    if (e != cudaSuccess) return e;
    return launched(1);
  }
  if (S <= 1024) {
    const int64_t rows = (int64_t)B * KVH;
    const dim3 grid((unsigned)((rows + WARP_ROWS_PER_CTA - 1) / WARP_ROWS_PER_CTA));
    const dim3 block(WARP_ROWS_PER_CTA * 32);
    const int Si = (int)S;
    cudaError_t e;
    if (S <= 128) e = launch_pdl(k_topk_warp<4>, grid, block, 0, st, scores, Si, k, protect_tail, live, largest, idx, rows);
    else if (S <= 256) e = launch_pdl(k_topk_warp<8>, grid, block, 0, st, scores, Si, k, protect_tail, live, largest, idx, rows);
    else if (S <= 512) e = launch_pdl(k_topk_warp<16>, grid, block, 0, st, scores, Si, k, protect_tail, live, largest, idx, rows);
    else e = launch_pdl(k_topk_warp<32>, grid, block, 0, st, scores, Si, k, protect_tail, live, largest, idx, rows);
    if (e != cudaSuccess) return e;
    return launched(1);
  }
  if (S <= SHORT_MAX) {
    cudaLaunchAttribute attrs[2];
    const cudaLaunchConfig_t cfg =
        pdl_config(dim3((unsigned)((int64_t)B * KVH)), dim3(SHORT_THREADS), 0, st, attrs);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_topk_short, scores, (int)S, k, protect_tail, live, largest, idx);
    if (e != cudaSuccess) return e;
    return launched(1);
  }
  const int cs = topk_cluster_size(S);
  const int64_t per_cta = ((S + (int64_t)cs * 32 - 1) / ((int64_t)cs * 32)) * 32;
  if (per_cta > SLICE_MAX) return cudaErrorInvalidValue;
  const size_t smem = (size_t)per_cta * 4;
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(k_topk), (int)(SLICE_MAX * 4));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3((unsigned)((int64_t)B * KVH * cs)), dim3(SEL_THREADS), smem, st, attrs, cs);
  e = cudaLaunchKernelEx(&cfg, k_topk, scores, S, k, protect_tail, live, largest, idx);
  if (e != cudaSuccess) return e;
  return launched(1);
}

cudaError_t launch_sh_evict(const kvc_sh_state& s, int m, int32_t* evicted, cudaStream_t st) {
  const size_t smem = (size_t)s.cap * 4;
  if ((int64_t)s.cap > SLICE_MAX) return cudaErrorInvalidValue;
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(k_sh_evict), (int)(SLICE_MAX * 4));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(s.B * s.KVH)), dim3(SEL_THREADS), smem, st, attrs);
  e = cudaLaunchKernelEx(&cfg, k_sh_evict, s, m, evicted);
  if (e != cudaSuccess) return e;
  return launched(1);
}

cudaError_t launch_sh_queue(const kvc_sh_state& s, int m, int32_t* queue, cudaStream_t st) {
  const size_t smem = (size_t)s.cap * 4;
  if ((int64_t)s.cap > SLICE_MAX || m > SH_QUEUE_MAX) return cudaErrorInvalidValue;
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(k_sh_queue), (int)(SLICE_MAX * 4));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(s.B * s.KVH)), dim3(SEL_THREADS), smem, st, attrs);
  e = cudaLaunchKernelEx(&cfg, k_sh_queue, s, m, queue);
  if (e != cudaSuccess) return e;
  return launched(1);
}

KVC_TU_STATUS(select)

}  // namespace kvc
