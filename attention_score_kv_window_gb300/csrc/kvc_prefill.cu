// Fused prefill compression for short rows: window scores, top-k and gather-compaction of
// one (b, kvh) in one CTA, with K read from HBM exactly once.
//
// What it computes is kvc_compress_prefill's definition ("Add TOVA press": the scores are the
// last w rows of the attention matrix, averaged over query heads and, for TOVA, over all
// heads; cold-compress PR 11: SnapKV keeps the observation window and compresses the prefix).
//
// One CTA per (b, kvh) -- per batch row in all-heads mode (TOVA), whose scores are the mean
// over every KV head's query group -- 8 warps:
//  1. One thread copies a head's key block [S, D] into shared memory with TMA (tensor-map
//     boxes of 64 channels x up to 256 rows, 128-byte swizzle: 16-byte chunk c of a row's
//     64-channel panel lands at chunk c ^ (r & 7), so ldmatrix of 8 rows is conflict-free);
//     the CTA waits on one mbarrier (bounded).
//  2. Logits on the tensor cores (mma.sync m16n8k16, the G*w <= 16 query rows as M, 8 keys as
//     N); each warp keeps its keys' logits in registers.  In all-heads mode the next head's
//     key block is copied in as soon as the logits are out of shared memory.
//  3. Per query row (max, sum) over the whole sequence (registers -> quad -> 8 warps), then
//     p = exp2(x - c_r) from the same registers, summed over the group's query rows and added
//     (head by head, in head order) into the row's scores in shared memory.
//  4. The CTA selects the k highest-ranked tokens (radix select over the score bits; ties to
//     the lower index; the last protect_tail positions forced in) with ascending output; in
//     all-heads mode every KV head of the row gets the same scores and indices.
//  5. Kept K rows of the last head are written from shared memory, those of earlier heads
//     read back (from L2: the block passed through it moments before); kept V rows are read
//     from HBM once.
//
// Shared memory holds K of one KV head: 64 KiB for 512 keys of 64 channels, so three CTAs
// share an SM and one CTA's copy-in overlaps another's compute and write-out.  The only
// waits are the key copy's mbarrier (bounded) and block barriers.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int PF_THREADS = 256;  // 8 warps
constexpr int PF_MAX_HEADS = 8;  // KV heads one all-heads CTA scores in turn

struct PrefillArgs {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;  // may be null (keys only), may be mapped page-locked host memory
  int64_t sb, sh, ss;
  int B, H, KVH, G, w, R, k, protect;
  int S;
  float sl2;     // scale * log2(e)
  float inv_g;   // 1 / G
  int nh;        // KV heads per CTA: KVH in all-heads mode, 1 otherwise
  bool v_device;  // V is device memory (not page-locked host memory read in place)
  float inv_nh;  // 1 / nh
  float* scores;  // [B*KVH][S] or null
  int32_t* idx;   // [B*KVH][k]
  uint16_t* Ko;   // [B*KVH][k][D]
  uint16_t* Vo;   // [B*KVH][k][D] or null
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (2 s, %globaltimer) for the key-copy barrier's phase of the given parity;
// false on timeout.
__device__ __forceinline__ bool wait_keys(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!mbar_try_wait(bar, parity)) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 2000000000ull) return false;
  }
  return true;
}
// L2 eviction policies: a key block that is read again after the selection (earlier heads of
// an all-heads row) stays in L2 ahead of data read once (the last head's block, the kept V
// rows and the read-back itself)
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}
// L2 prefetch of one key box (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_4d_hint(const CUtensorMap* tm, int x, int y, int z, int w,
                                                     uint64_t policy) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.4d.L2.global.tile.L2::cache_hint [%0, {%1, %2, %3, %4}], %5;\n" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
      : "memory");
}
// a row read once: device memory with the evict-first policy, page-locked host memory (read in
// place over the host link) with a plain non-coherent load
__device__ __forceinline__ uint4 ld_once(const void* p, uint64_t policy, bool device) {
  if (!device) return __ldg(reinterpret_cast<const uint4*>(p));
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// scores are probabilities (>= 0): the float bits order them; -0 ranks as +0
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t ld_q32(const uint16_t* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }

// Keep the k highest-ranked of the S scores (a outranks b: higher score, or equal and lower
// index); positions >= S - protect are forced in.  Score j is acc[j] (times mul when nh > 1),
// written to the nh rows of scores_out (S apart) when that is given; the indices go to the nh
// rows of gidx (k apart) and to sidx.
// All PF_THREADS threads; thread t holds keys t + PF_THREADS * u.  An MSB-first radix select
// over the 32-bit key, starting below the bits every candidate shares (the block's min and max
// key give them): the scores of a row are close, so most of the 32 bits are settled at once,
// and the first 8-bit digit already spreads the keys over many bins (plain shared atomics then
// rarely collide; grouping lanes with match.any measured slower).  Warp 0 finds the bin
// holding the need-th key; two histograms alternate between digits (one filled while the other
// is cleared), so a digit costs two block barriers; the select stops as soon as that bin is
// taken whole.  The output pass counts, in index order, the keys taken for sure and the keys
// in the tie bin (one ballot scan for both), so the indices come out ascending.  Fewer than k
// candidates: all are taken and the rest of the row is -1.  hist: 2 x 256 words.
template <int KPT>
__device__ void block_select_keep(const float* acc, float mul, int nh, float* scores_out, int S, int k, int protect,
                                  int32_t* sidx, int32_t* gidx, uint32_t* hist) {
  constexpr int NW = PF_THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ uint32_t s_pick[3];  // digit, keys above its bin, keys in its bin
  uint32_t key[KPT];
  bool cand[KPT], forc[KPT];
  uint32_t nf = 0u, ne = 0u, kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    const int j = tid + PF_THREADS * u;
    forc[u] = j < S && j >= S - protect;
    cand[u] = j < S - protect;
    float sc = 0.f;
    if (j < S) {
      sc = acc[j];
      if (nh > 1) sc *= mul;
      if (scores_out)
        for (int h = 0; h < nh; ++h) scores_out[(int64_t)h * S + j] = sc;
    }
    key[u] = cand[u] ? score_key(sc) : 0u;
    nf += __popc(__ballot_sync(0xffffffffu, forc[u]));
    ne += __popc(__ballot_sync(0xffffffffu, cand[u]));
    kmin = min(kmin, cand[u] ? key[u] : 0xffffffffu);
    kmax = max(kmax, key[u]);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  uint32_t* const cnt = hist + 256;  // per-warp counts, read before the first digit clears them
  hist[tid] = 0u;                    // PF_THREADS == 256 bins: the first digit's histogram
  if (lane == 0) {
    cnt[warp] = nf;
    cnt[NW + warp] = ne;
    cnt[2 * NW + warp] = kmin;
    cnt[3 * NW + warp] = kmax;
  }
  __syncthreads();
  uint32_t n_forced = 0u, n_elig = 0u;
  kmin = 0xffffffffu;
  kmax = 0u;
#pragma unroll
  for (int q = 0; q < NW; ++q) {
    n_forced += cnt[q];
    n_elig += cnt[NW + q];
    kmin = min(kmin, cnt[2 * NW + q]);
    kmax = max(kmax, cnt[3 * NW + q]);
  }
  const uint32_t need = (uint32_t)k > n_forced ? (uint32_t)k - n_forced : 0u;
  const bool take_all = n_elig <= need;
  const bool split = !take_all && need > 0u;
  // bits [hi, 32) are common to every candidate key (they lie between kmin and kmax)
  int hi = 32 - __clz(kmin ^ kmax);
  uint32_t mask = hi == 32 ? 0u : ~((1u << hi) - 1u);
  uint32_t T = kmin & mask, rem = need, in_bin = n_elig;
  uint32_t* tot = cnt + 4 * NW;  // packed output counts: a region no thread touches by then
  if (split) {
#pragma unroll 1
    for (int pass = 0; hi > 0 && rem != in_bin; ++pass) {
      const int lo = hi > 8 ? hi - 8 : 0;
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
      uint32_t* h = hist + (pass & 1) * 256;
      // histogram of the next digit over the keys that match the prefix so far (h is zero)
#pragma unroll
      for (int u = 0; u < KPT; ++u)
        if (cand[u] && (key[u] & mask) == T) atomicAdd(&h[(key[u] >> lo) & dmask], 1u);
      __syncthreads();
      // the other histogram is idle until the next digit (its last readers passed the barrier
      // above; it is next filled after the one below): clear it
      uint32_t* other = hist + ((pass + 1) & 1) * 256;
      other[tid] = 0u;
      tot = other + 4 * NW;
      if (warp == 0) {
        // lane l scans bins 255 - 8l down to 248 - 8l (digits in descending order)
        uint32_t hv[8], sum = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          hv[q] = h[255 - 8 * lane - q];
          sum += hv[q];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - sum;
        if (excl < rem && rem <= incl) {
          uint32_t run = excl;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (run + hv[q] >= rem) {
              s_pick[0] = 255u - 8u * lane - q;
              s_pick[1] = run;
              s_pick[2] = hv[q];
              break;
            }
            run += hv[q];
          }
        }
      }
      __syncthreads();
      T |= s_pick[0] << lo;
      mask |= dmask << lo;
      rem -= s_pick[1];
      in_bin = s_pick[2];
      hi = lo;
    }
  }
  // taken: forced; all candidates (take_all); keys whose prefix is above T; and the first
  // `rem` keys (index order) whose prefix equals T
  const uint32_t lower = (1u << lane) - 1u;
  uint32_t sure_b[KPT], eq_b[KPT];
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    const uint32_t kp = key[u] & mask;
    const bool sure = forc[u] || (cand[u] && (take_all || (split && kp > T)));
    const bool eq = split && cand[u] && kp == T;
    sure_b[u] = __ballot_sync(0xffffffffu, sure);
    eq_b[u] = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) tot[u * NW + warp] = (uint32_t)__popc(sure_b[u]) | ((uint32_t)__popc(eq_b[u]) << 16);
  }
  __syncthreads();
  uint32_t before = 0u;  // packed (sure | eq << 16) counts of keys with a lower index
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    uint32_t b = before;
    for (int q = 0; q < warp; ++q) b += tot[u * NW + q];
    b += (uint32_t)__popc(sure_b[u] & lower) | ((uint32_t)__popc(eq_b[u] & lower) << 16);
    const bool sure = (sure_b[u] >> lane) & 1u, eq = (eq_b[u] >> lane) & 1u;
    const uint32_t eq_before = b >> 16, sure_before = b & 0xffffu;
    if (sure || (eq && eq_before < rem)) {
      const uint32_t p = sure_before + (eq_before < rem ? eq_before : rem);
      if (p < (uint32_t)k) {
        sidx[p] = tid + PF_THREADS * u;
        for (int h = 0; h < nh; ++h) gidx[(int64_t)h * k + p] = tid + PF_THREADS * u;
      }
    }
    for (int q = 0; q < NW; ++q) before += tot[u * NW + q];
  }
  const uint32_t taken = (before & 0xffffu) + ((before >> 16) < rem ? (before >> 16) : rem);
  for (int p = (int)taken + tid; p < k; p += PF_THREADS) {
    sidx[p] = -1;
    for (int h = 0; h < nh; ++h) gidx[(int64_t)h * k + p] = -1;
  }
}

// One level of the sum over lane bit `bit`: with N >= 2 values a lane keeps the half selected
// by its bit and receives the partner's copy of it (off: first value index kept); with one
// value both lanes add and the one with the bit set becomes a duplicate.
template <int N>
__device__ __forceinline__ void reduce_level(float* v, int& off, bool& dup, int lane, int bit) {
  const bool up = (lane & bit) != 0;
  if constexpr (N >= 2) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = up ? v[i] : v[N / 2 + i];
      const float keep = up ? v[N / 2 + i] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
    off += up ? N / 2 : 0;
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], bit);
    dup = dup || up;
  }
}

// Byte offset of 16-byte chunk c of key row r in the staged block of `sp` rows: the rows'
// 64-channel panels one after another (128-byte rows), chunks swizzled by the row (the layout
// TMA writes with the 128-byte swizzle).
__device__ __forceinline__ uint32_t kaddr(int r, int c, int sp) {
  return (uint32_t)((c >> 3) * sp * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// rows per TMA box: the staged block is 64 * NT rows
constexpr int box_rows(int nt) { return 64 * nt < 256 ? 64 * nt : 256; }

// D channels, NT 8-key n-tiles per warp (the key block is padded to 64 * NT rows).  CTA x
// handles the a.nh units (b, kvh) starting at x * a.nh: one in GQA mode, every KV head of
// batch row x in all-heads mode.
// (A persistent variant that copies the next unit's keys in during the V gather measured no
// faster: three CTAs per SM already overlap one CTA's copy with another's compute.)
template <int D, int NT>
__global__ void __launch_bounds__(PF_THREADS, (D == 64 && NT <= 8) ? 3 : 1)
    k_prefill_fused(const PrefillArgs a, const __grid_constant__ CUtensorMap tmK) {
  extern __shared__ unsigned char smem_raw[];
  // TMA's 128-byte swizzle wants the staged block 1024-byte aligned
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int CH = D / 8;        // 16-byte chunks per key row
  constexpr int KS = D / 16;       // k-steps of the MMA
  constexpr int SP = 64 * NT;      // padded key rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int S = a.S, nh = a.nh;
  const int64_t bk0 = (int64_t)blockIdx.x * nh;  // first unit (b * KVH + kvh) of this CTA
  const int64_t b = bk0 / a.KVH;
  const int kvh0 = (int)(bk0 % a.KVH);

  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);                        // [SP][D], swizzled chunks
  float* acc = reinterpret_cast<float*>(Ks + SP * D);                      // [SP] scores, summed over heads
  int32_t* sidx = reinterpret_cast<int32_t*>(acc + SP);                    // [SP]
  float2* red = reinterpret_cast<float2*>(sidx + SP);                      // [8 warps][16 rows]
  uint32_t* hist = reinterpret_cast<uint32_t*>(red + 8 * 16);              // [2][256]
  const uint32_t kbar = smem_u32(hist + 512);                              // the key copy's mbarrier
  const uint32_t ks0 = smem_u32(Ks);
  constexpr int BR = box_rows(NT);
  auto copy_keys = [&](int kvh) {  // one thread: the key block of head kvh, one barrier phase
    mbar_expect_tx(kbar, (uint32_t)(SP * D * 2));
    const uint64_t pol = kvh < kvh0 + nh - 1 ? l2_policy_evict_last() : l2_policy_evict_first();
    for (int p = 0; p < D / 64; ++p)
      for (int r0 = 0; r0 < SP; r0 += BR)
        tma_load_4d_hint(ks0 + (uint32_t)(p * SP * 128 + r0 * 128), &tmK, p * 64, r0, kvh, (int)b, kbar, pol);
  };
  // The next head's key block, requested into L2 (evict-last) one copy ahead, so that its copy
  // (issued once the stage is free) is an L2 hit and the CTA keeps more reads in flight.  Only
  // with V in device memory: when the kept V rows come over the host link the pinned blocks
  // slowed the whole pipeline, and without the evict-last hint the prefetch gained nothing.
  auto prefetch_keys = [&](int kvh) {
    if (kvh >= kvh0 + nh || !a.v_device) return;
    const uint64_t keep = l2_policy_evict_last();
    for (int p = 0; p < D / 64; ++p)
      for (int r0 = 0; r0 < SP; r0 += BR) tma_prefetch_4d_hint(&tmK, p * 64, r0, kvh, (int)b, keep);
  };

  pdl_wait();   // previous kernel on the stream complete and visible
  pdl_trigger();

  // last key each of the two rows held by this lane may see (causal window; -1: no row)
  const int limA = g < a.R ? S - a.w + (g % a.w) : -1;
  const int limB = g + 8 < a.R ? S - a.w + ((g + 8) % a.w) : -1;

  // 1. the first head's key block: one thread issues the TMA boxes (rows >= S arrive zero-filled)
  // and requests the second head's block into L2
  if (tid == 0) {
    mbar_init(kbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    copy_keys(kvh0);
    prefetch_keys(kvh0 + 1);
  }
  __syncthreads();  // the barrier is initialised before anyone waits on it
  bool keys_ok = true;
  int phase = 0;  // key copies waited for so far
  for (int hh = 0; hh < nh; ++hh) {
    const int kvh = kvh0 + hh;
    // 2. query fragments of the group's R rows (row r = head-in-group * w + window row)
    const uint16_t* Qg = a.q + (b * a.H + kvh * a.G) * (int64_t)a.w * D;
    uint32_t aq[KS][4];
    {
      const bool rA = g < a.R, rB = g + 8 < a.R;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int col = ks * 16 + 2 * t;
        aq[ks][0] = rA ? ld_q32(Qg + g * D + col) : 0u;
        aq[ks][1] = rB ? ld_q32(Qg + (g + 8) * D + col) : 0u;
        aq[ks][2] = rA ? ld_q32(Qg + g * D + col + 8) : 0u;
        aq[ks][3] = rB ? ld_q32(Qg + (g + 8) * D + col + 8) : 0u;
      }
    }
    keys_ok = __syncthreads_and(wait_keys(kbar, (uint32_t)(phase & 1)) ? 1 : 0) != 0;
    ++phase;
    if (!keys_ok) {  // (the same decision in every thread)
      if (tid == 0) set_device_status(KVC_ERR_TIMEOUT);
      break;
    }

    // 3. logits (log2 domain) of this warp's keys, kept in registers
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int key0 = (warp * NT + nt) * 8;
#pragma unroll
      for (int e = 0; e < 4; ++e) c[nt][e] = 0.f;
      const int r = key0 + (lane & 7);
#pragma unroll
      for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
        uint32_t b0, b1, b2, b3;
        const int ch = ks2 * 4 + (lane >> 3);
        ldsm_x4(ks0 + kaddr(r, ch, SP), b0, b1, b2, b3);
        mma16816(c[nt], aq[2 * ks2], b0, b1);
        mma16816(c[nt], aq[2 * ks2 + 1], b2, b3);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = key0 + 2 * t + e;
        c[nt][e] = j <= limA ? c[nt][e] * a.sl2 : -CUDART_INF_F;
        c[nt][2 + e] = j <= limB ? c[nt][2 + e] * a.sl2 : -CUDART_INF_F;
      }
    }
    if (hh + 1 < nh) {
      // every warp's keys are in registers: the next head's block may overwrite the stage
      // (the generic-proxy reads above are ordered before the copy by the barrier and fence)
      __syncthreads();
      if (tid == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        copy_keys(kvh + 1);
        prefetch_keys(kvh + 2);
      }
    }

    // 4. per row (max, sum) over the whole sequence: lane, quad, then the 8 warps
    float mA = -CUDART_INF_F, mB = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mA = fmaxf(mA, fmaxf(c[nt][0], c[nt][1]));
      mB = fmaxf(mB, fmaxf(c[nt][2], c[nt][3]));
    }
    float lA = 0.f, lB = 0.f;
    if (mA != -CUDART_INF_F) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) lA += ex2(c[nt][0] - mA) + ex2(c[nt][1] - mA);
    }
    if (mB != -CUDART_INF_F) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) lB += ex2(c[nt][2] - mB) + ex2(c[nt][3] - mB);
    }
    auto merge2 = [](float& m, float& l, float m2, float l2) {
      const float mn = fmaxf(m, m2);
      if (mn != -CUDART_INF_F) {
        l = l * ex2(m - mn) + l2 * ex2(m2 - mn);
        m = mn;
      }
    };
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      merge2(mA, lA, __shfl_xor_sync(0xffffffffu, mA, o), __shfl_xor_sync(0xffffffffu, lA, o));
      merge2(mB, lB, __shfl_xor_sync(0xffffffffu, mB, o), __shfl_xor_sync(0xffffffffu, lB, o));
    }
    // (the previous head's readers of red passed the barrier at this head's key wait)
    if (t == 0) {
      red[warp * 16 + g] = make_float2(mA, lA);
      red[warp * 16 + g + 8] = make_float2(mB, lB);
    }
    __syncthreads();
    // every lane merges the 8 warps' partials of its two rows itself (no second barrier);
    // the normaliser in the log2 domain is M + log2(L), +inf for a row that sees no key
    float cA, cB;
    {
      float MA = -CUDART_INF_F, LA = 0.f, MB = -CUDART_INF_F, LB = 0.f;
#pragma unroll
      for (int q = 0; q < PF_THREADS / 32; ++q) {
        const float2 pa = red[q * 16 + g], pb = red[q * 16 + g + 8];
        merge2(MA, LA, pa.x, pa.y);
        merge2(MB, LB, pb.x, pb.y);
      }
      cA = LA > 0.f ? MA + log2f(LA) : CUDART_INF_F;
      cB = LB > 0.f ? MB + log2f(LB) : CUDART_INF_F;
    }

    // 5. group-mean probability per key: rows g and g + 8 in this lane, then the sum over the
    //    8 g's (lane bits 2..4) as a transpose-reduce: at each level a lane keeps half of its
    //    values and adds the partner's copy of that half, so the 2 * NT sums of a lane take
    //    14 shuffles (NT = 8) instead of 48, and every lane ends with its own keys; those are
    //    added into the row's scores (each key has one owner lane: no two lanes write it)
    constexpr int NV = 2 * NT;  // value m = 2 * nt + e: key (warp * NT + nt) * 8 + 2t + e
    float v[NV];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        v[2 * nt + e] = (limA >= 0 ? ex2(c[nt][e] - cA) : 0.f) + (limB >= 0 ? ex2(c[nt][2 + e] - cB) : 0.f);
    int off = 0;
    bool dup = false;  // this lane's sums are also held by a lane with lower g (it writes them)
    reduce_level<NV>(v, off, dup, lane, 4);
    reduce_level<(NV >= 2 ? NV / 2 : 1)>(v, off, dup, lane, 8);
    reduce_level<(NV >= 4 ? NV / 4 : 1)>(v, off, dup, lane, 16);
    constexpr int NF = NV >= 8 ? NV / 8 : 1;  // sums left in this lane: values off .. off + NF - 1
    if (!dup) {
#pragma unroll
      for (int i = 0; i < NF; ++i) {
        const int m = off + i;
        const int j = (warp * NT + (m >> 1)) * 8 + 2 * t + (m & 1);
        const float gm = v[i] * a.inv_g;
        acc[j] = hh == 0 ? gm : acc[j] + gm;
      }
    }
  }
  if (keys_ok) {
    __syncthreads();  // every head's scores are in acc
    // 6. selection (all threads), ascending indices to shared memory and to every head's output
    block_select_keep<(64 * NT + PF_THREADS - 1) / PF_THREADS>(acc, a.inv_nh, nh,
                                                                a.scores ? a.scores + bk0 * S : nullptr, S, a.k,
                                                                a.protect, sidx, a.idx + bk0 * a.k, hist);
    __syncthreads();

    // 7. kept rows of every head: V from HBM, K of the last head from shared memory and of the
    //    earlier heads from global memory (a batch's loads issued before the stores).  (An L2
    //    prefetch of every head's kept V rows ahead of the gather measured 9 % slower.)
    const int total = a.k * CH;
    const uint64_t once = l2_policy_evict_first();
    for (int hh = 0; hh < nh; ++hh) {
      const int kvh = kvh0 + hh;
      const uint16_t* Vb = a.V ? a.V + b * a.sb + kvh * a.sh : nullptr;
      uint16_t* Ko = a.Ko + (bk0 + hh) * a.k * (int64_t)D;
      uint16_t* Vo = a.Vo ? a.Vo + (bk0 + hh) * a.k * (int64_t)D : nullptr;
      if (hh == nh - 1) {
        constexpr int BATCH = 8;
        for (int base = 0; base < total; base += PF_THREADS * BATCH) {
          uint4 vv[BATCH];
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            const int x = base + u * PF_THREADS + tid;
            const int j = x < total ? sidx[x / CH] : -1;
            vv[u] = make_uint4(0u, 0u, 0u, 0u);
            if (Vb && j >= 0) vv[u] = ld_once(Vb + (int64_t)j * a.ss + (x % CH) * 8, once, a.v_device);
          }
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            const int x = base + u * PF_THREADS + tid;
            if (x < total) {
              const int j = sidx[x / CH], cc = x % CH;
              uint4 kv = make_uint4(0u, 0u, 0u, 0u);
              if (j >= 0) kv = *reinterpret_cast<const uint4*>(smem + kaddr(j, cc, SP));
              __stcs(reinterpret_cast<uint4*>(Ko + (int64_t)x * 8), kv);
              if (Vo) __stcs(reinterpret_cast<uint4*>(Vo + (int64_t)x * 8), vv[u]);
            }
          }
        }
      } else {
        const uint16_t* Kb = a.K + b * a.sb + kvh * a.sh;
        constexpr int BATCH = 8;
        for (int base = 0; base < total; base += PF_THREADS * BATCH) {
          uint4 vv[BATCH], kk[BATCH];
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            const int x = base + u * PF_THREADS + tid;
            const int j = x < total ? sidx[x / CH] : -1;
            vv[u] = make_uint4(0u, 0u, 0u, 0u);
            kk[u] = vv[u];
            if (j >= 0) {
              const int64_t o = (int64_t)j * a.ss + (x % CH) * 8;
              kk[u] = ld_once(Kb + o, once, true);
              if (Vb) vv[u] = ld_once(Vb + o, once, a.v_device);
            }
          }
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            const int x = base + u * PF_THREADS + tid;
            if (x < total) {
              __stcs(reinterpret_cast<uint4*>(Ko + (int64_t)x * 8), kk[u]);
              if (Vo) __stcs(reinterpret_cast<uint4*>(Vo + (int64_t)x * 8), vv[u]);
            }
          }
        }
      }
    }
  } else if (tid == 0) {
    // a key copy that did not arrive in time is waited for once more (bounded) before leaving
    wait_keys(kbar, (uint32_t)((phase - 1) & 1));
  }
}

int prefill_nt(int D, int64_t S) {
  const int max_nt = D == 64 ? 16 : 8;
  for (int nt = 1; nt <= max_nt; nt *= 2)
    if (64 * (int64_t)nt >= S) return nt;
  return 0;
}

size_t prefill_smem(int D, int nt) {
  const size_t sp = 64 * (size_t)nt;
  // + the key copy's mbarrier and 1024 bytes for the staged block's alignment
  return sp * D * 2 + sp * 4 + sp * 4 + 8 * 16 * sizeof(float2) + 2 * 256 * 4 + 16 + 1024;
}

// TMA maps of the caches last used (encoding costs host microseconds), per host thread
const CUtensorMap* key_map(const uint16_t* K, const kvc_kv_desc& kv, int rows) {
  struct Entry {
    CUtensorMap map;
    const void* K;
    int64_t S, ss, sh, sb;
    int B, KVH, D, rows;
    bool valid = false, ok = false;
  };
  thread_local Entry cache[8];
  thread_local int next = 0;
  for (Entry& e : cache)
    if (e.valid && e.K == K && e.S == kv.S && e.ss == kv.stride_s && e.sh == kv.stride_h && e.sb == kv.stride_b &&
        e.B == kv.B && e.KVH == kv.KVH && e.D == kv.D && e.rows == rows)
      return e.ok ? &e.map : nullptr;
  Entry& e = cache[next];
  next = (next + 1) % 8;
  e.K = K;
  e.S = kv.S;
  e.ss = kv.stride_s;
  e.sh = kv.stride_h;
  e.sb = kv.stride_b;
  e.B = kv.B;
  e.KVH = kv.KVH;
  e.D = kv.D;
  e.rows = rows;
  e.valid = true;
  e.ok = make_cache_tensor_map(K, kv, &e.map, rows);
  return e.ok ? &e.map : nullptr;
}

template <int D, int NT>
cudaError_t launch_fused_t(const PrefillArgs& a, const kvc_kv_desc& kv, cudaStream_t st) {
  const CUtensorMap* tm = key_map(a.K, kv, box_rows(NT));
  if (!tm) return cudaErrorInvalidValue;
  const size_t smem = prefill_smem(D, NT);
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(k_prefill_fused<D, NT>), (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3((unsigned)((int64_t)a.B * a.KVH / a.nh)), dim3(PF_THREADS), smem, st, attrs);
  e = cudaLaunchKernelEx(&cfg, k_prefill_fused<D, NT>, a, *tm);
  if (e != cudaSuccess) return e;
  return launched(1);
}

}  // namespace

bool prefill_fused_supported(const kvc_kv_desc& kv, int w, int k, int reduce) {
  const int G = kv.H / kv.KVH;
  if ((int64_t)G * w > 16) return false;
  if (reduce == KVC_REDUCE_ALL_HEADS && kv.KVH > PF_MAX_HEADS) return false;
  const int nt = prefill_nt(kv.D, kv.S);
  if (nt == 0 || (int64_t)k > 64 * (int64_t)nt) return false;
  if ((int64_t)kv.B * kv.KVH > 2147483647LL) return false;
  return prefill_smem(kv.D, nt) <= 227 * 1024;
}

cudaError_t launch_prefill_fused(const uint16_t* q, const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv, int w,
                                 float scale, int reduce, int k, int protect, float* scores, int32_t* idx,
                                 uint16_t* Ko, uint16_t* Vo, cudaStream_t st) {
  if (!prefill_fused_supported(kv, w, k, reduce)) return cudaErrorNotSupported;
  PrefillArgs a{};
  a.q = q;
  a.K = K;
  a.V = V;
  a.sb = kv.stride_b;
  a.sh = kv.stride_h;
  a.ss = kv.stride_s;
  a.B = kv.B;
  a.H = kv.H;
  a.KVH = kv.KVH;
  a.G = kv.H / kv.KVH;
  a.w = w;
  a.R = a.G * w;
  a.k = k;
  a.protect = protect;
  a.S = (int)kv.S;
  a.sl2 = scale * 1.4426950408889634f;
  a.inv_g = 1.f / (float)a.G;
  a.nh = reduce == KVC_REDUCE_ALL_HEADS ? kv.KVH : 1;
  a.inv_nh = 1.f / (float)a.nh;
  a.scores = scores;
  a.idx = idx;
  a.Ko = Ko;
  a.Vo = V ? Vo : nullptr;
  a.v_device = true;
  if (V) {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, V) == cudaSuccess) a.v_device = pa.type == cudaMemoryTypeDevice;
    else cudaGetLastError();
  }
  const int nt = prefill_nt(kv.D, kv.S);
  if (kv.D == 64) {
    switch (nt) {
      case 1: return launch_fused_t<64, 1>(a, kv, st);
      case 2: return launch_fused_t<64, 2>(a, kv, st);
      case 4: return launch_fused_t<64, 4>(a, kv, st);
      case 8: return launch_fused_t<64, 8>(a, kv, st);
      default: return launch_fused_t<64, 16>(a, kv, st);
    }
  }
  switch (nt) {
    case 1: return launch_fused_t<128, 1>(a, kv, st);
    case 2: return launch_fused_t<128, 2>(a, kv, st);
    case 4: return launch_fused_t<128, 4>(a, kv, st);
    default: return launch_fused_t<128, 8>(a, kv, st);
  }
}

KVC_TU_STATUS(prefill)

}  // namespace kvc
