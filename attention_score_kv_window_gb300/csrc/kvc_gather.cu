// Memory-bound row movers: K/V gather-compaction, slot writes, and the ThinK key-channel
// score and pruning ("Add ThinK_Press", kvpress PR 18).  All rows are moved as 16-byte
// vectors (8 bf16); grids are sized in multiples of the SM count and grid-stride.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

__device__ __forceinline__ uint4 ld16(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st16(uint16_t* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }

// ----------------------------------------------------------------------------------------
// compaction: Ko[b,kvh,t] = K[b,kvh,idx[b,kvh,t]] (V likewise); -1 -> zero row
// ----------------------------------------------------------------------------------------
// One warp per 16 output rows: lanes 0-15 load the rows' indices and source offsets once,
// then every lane issues all of its 16-byte loads for the 16 rows (K and V) before any
// store, so a warp keeps 16 x 2 x D x 2 bytes of gather in flight.
constexpr int COMPACT_RPW = 16;  // output rows per warp
template <int D>
__global__ void __launch_bounds__(256) k_compact(const uint16_t* __restrict__ K,
                                                 const uint16_t* __restrict__ V, int64_t sb,
                                                 int64_t sh, int64_t ss, int KVH, int64_t S,
                                                 const int32_t* __restrict__ idx, int k,
                                                 int64_t rows, uint16_t* __restrict__ Ko,
                                                 uint16_t* __restrict__ Vo) {
  pdl_wait();
  pdl_trigger();
  constexpr int TPR = D / 8;              // 16-byte chunks per row
  constexpr int RPI = 32 / TPR;           // rows per warp-wide step
  constexpr int ITER = COMPACT_RPW / RPI; // steps per warp
  const int lane = threadIdx.x & 31;
  const int c = lane % TPR;
  const int64_t warp_g = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r0 = warp_g * COMPACT_RPW; r0 < rows; r0 += nwarps * COMPACT_RPW) {
    int64_t off = -1;  // lane < 16: source offset of row r0 + lane (-1: zero row)
    if (lane < COMPACT_RPW && r0 + lane < rows) {
      const int64_t row = r0 + lane;
      const int32_t j = __ldg(idx + row);
      if (j >= 0 && j < S) {
        const int64_t bk = row / k;
        off = (bk / KVH) * sb + (bk % KVH) * sh + (int64_t)j * ss;
      } else if (j >= S || j < -1) {
        set_device_status(KVC_ERR_DEVICE_BOUNDS);
      }
    }
    uint4 kv[ITER], vv[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t o = __shfl_sync(0xffffffffu, off, it * RPI + lane / TPR);
      kv[it] = make_uint4(0, 0, 0, 0);
      vv[it] = kv[it];
      if (o >= 0) {
        kv[it] = ld16(K + o + c * 8);
        if (V) vv[it] = ld16(V + o + c * 8);
      }
    }
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t row = r0 + it * RPI + lane / TPR;
      if (row < rows) {
        st16(Ko + row * D + c * 8, kv[it]);
        if (Vo) st16(Vo + row * D + c * 8, vv[it]);
      }
    }
  }
}

template <int D>
__global__ void k_write_slots(const uint16_t* __restrict__ kn, const uint16_t* __restrict__ vn,
                              const int32_t* __restrict__ slot, uint16_t* K, uint16_t* V, int64_t sb,
                              int64_t sh, int64_t ss, int KVH, int64_t S, int rows) {
  pdl_wait();  // previous kernel on the stream complete and visible
  constexpr int TPR = D / 8;
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= rows * TPR) return;
  const int row = x / TPR, c = x % TPR;
  const int32_t j = slot[row];
  if (j < 0 || j >= S) {
    set_device_status(KVC_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t b = row / KVH, kvh = row % KVH;
  const int64_t off = b * sb + kvh * sh + (int64_t)j * ss + c * 8;
  *reinterpret_cast<uint4*>(K + off) = ld16(kn + (int64_t)row * D + c * 8);
  if (V) *reinterpret_cast<uint4*>(V + off) = ld16(vn + (int64_t)row * D + c * 8);
}

// ----------------------------------------------------------------------------------------
// ThinK channel score: cs = (mean over group of sum_i q^2) * sum_j k^2 (per channel)
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ void acc_sq8(float* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xffff0000u);
    acc[2 * i] = fmaf(lo, lo, acc[2 * i]);
    acc[2 * i + 1] = fmaf(hi, hi, acc[2 * i + 1]);
  }
}

// Query half of the ThinK channel score, one share: the CTA (split of nsplit) of KV head (b,
// kvh) sums q^2 per channel over the group's window rows split, split + nsplit, ... (the G*w
// rows are contiguous: [b][kvh*G .. kvh*G + G)[w][D]) and stores qpart[split][b*KVH+kvh][D].
// 256 threads, TPR per row; red is the caller's [256/TPR][D+1] reduction array, free on entry.
template <int D>
__device__ __forceinline__ void q_sq_partial(const uint16_t* __restrict__ q, int H, int w, int KVH, int b, int kvh,
                                             int split, int nsplit, int nbk, float (*red)[D + 1],
                                             float* __restrict__ qpart) {
  constexpr int TPR = D / 8, RPP = 256 / TPR, U = 4;
  const int c = threadIdx.x % TPR, rl = threadIdx.x / TPR;
  const int G = H / KVH, nq = G * w;
  const uint16_t* qg = q + ((int64_t)(b * H + kvh * G) * w) * D;
  float qa[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r0 = split + rl * nsplit; r0 < nq; r0 += U * RPP * nsplit) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + u * RPP * nsplit;
      v[u] = r < nq ? ld16(qg + (int64_t)r * D + c * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) acc_sq8(qa, v[u]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[rl][c * 8 + i] = qa[i];
  __syncthreads();
  const int bk = b * KVH + kvh;
  for (int d = threadIdx.x; d < D; d += 256) {
    float sum = 0.f;
    for (int rr = 0; rr < RPP; ++rr) sum += red[rr][d];
    qpart[((int64_t)split * nbk + bk) * D + d] = sum;
  }
}

// Compaction of one (b, kvh)'s kept rows, chunk by chunk (grid: nsplit x B*KVH), that also
// sums the squares of every kept key per channel: ThinK's key-channel norms come from the
// compaction's own read of the kept K rows ("Add ThinK_Press": sum_j k_jd^2 over the kept
// tokens), so no later call reads K_out again.  Each CTA stores its partial sums
// kpart[split][b*KVH+kvh][D] and the query half of the score (q_sq_partial); warps move 16
// rows at a time as in k_compact.  Sums are in a fixed order: runs are bit-identical.
template <int D>
__global__ void __launch_bounds__(256) k_compact_ksq(const uint16_t* __restrict__ K,
                                                     const uint16_t* __restrict__ V, int64_t sb, int64_t sh,
                                                     int64_t ss, int KVH, int64_t S,
                                                     const int32_t* __restrict__ idx, int k, int64_t chunk,
                                                     uint16_t* __restrict__ Ko, uint16_t* __restrict__ Vo,
                                                     float* __restrict__ kpart, const uint16_t* __restrict__ q,
                                                     int H, int w, float* __restrict__ qpart) {
  pdl_wait();
  constexpr int TPR = D / 8, RPI = 32 / TPR, ITER = COMPACT_RPW / RPI, RPP = 256 / TPR;
  __shared__ float red[RPP][D + 1];
  const int split = blockIdx.x, bk = blockIdx.y;
  const int b = bk / KVH, kvh = bk % KVH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, c = lane % TPR;
  const int64_t r_beg = (int64_t)split * chunk, r_end = std::min<int64_t>(k, r_beg + chunk);
  const int64_t row0 = (int64_t)bk * k;  // this (b, kvh)'s first output row
  const uint16_t* Kb = K + (int64_t)b * sb + (int64_t)kvh * sh;
  const uint16_t* Vb = V ? V + (int64_t)b * sb + (int64_t)kvh * sh : nullptr;
  pdl_trigger();
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int64_t r0 = r_beg + (int64_t)warp * COMPACT_RPW; r0 < r_end; r0 += 8 * COMPACT_RPW) {
    int64_t off = -1;  // lane < 16: source offset of row r0 + lane (-1: zero row)
    if (lane < COMPACT_RPW && r0 + lane < r_end) {
      const int32_t j = __ldg(idx + row0 + r0 + lane);
      if (j >= 0 && j < S) off = (int64_t)j * ss;
      else if (j >= S || j < -1) set_device_status(KVC_ERR_DEVICE_BOUNDS);
    }
    uint4 kv[ITER], vv[ITER];
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t o = __shfl_sync(0xffffffffu, off, it * RPI + lane / TPR);
      kv[it] = make_uint4(0, 0, 0, 0);
      vv[it] = kv[it];
      if (o >= 0) {
        kv[it] = ld16(Kb + o + c * 8);
        if (Vb) vv[it] = ld16(Vb + o + c * 8);
      }
    }
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t r = r0 + it * RPI + lane / TPR;
      if (r < r_end) {
        st16(Ko + (row0 + r) * D + c * 8, kv[it]);
        if (Vo) st16(Vo + (row0 + r) * D + c * 8, vv[it]);
      }
      acc_sq8(acc, kv[it]);  // zero rows add nothing
    }
  }
  // lanes with the same channel block: reduce in shared memory (slot = warp x RPI + lane / TPR)
#pragma unroll
  for (int i = 0; i < 8; ++i) red[warp * RPI + lane / TPR][c * 8 + i] = acc[i];
  __syncthreads();
  const int nbk = gridDim.y;
  for (int d = threadIdx.x; d < D; d += 256) {
    float sum = 0.f;
    for (int rr = 0; rr < RPP; ++rr) sum += red[rr][d];
    kpart[((int64_t)split * nbk + bk) * D + d] = sum;
  }
  __syncthreads();  // red is reused
  q_sq_partial<D>(q, H, w, KVH, b, kvh, split, gridDim.x, nbk, red, qpart);
}

// partial sums of squares over one range of rows, weighted by wts[b*KVH+kvh][row] when
// given: part[split][b*KVH+kvh][D].  With q given, the CTA also sums q^2 over its share of the
// group's window rows (rows split, split + nsplit, ...): qpart[split][b*KVH+kvh][D], so that
// the final step reads two partials per split and nothing else.
template <int D>
__global__ void __launch_bounds__(256) k_channel_partial(const uint16_t* __restrict__ K, int64_t sb,
                                                         int64_t sh, int64_t ss, int64_t S,
                                                         const int32_t* __restrict__ idx, int k,
                                                         int64_t nrows, int64_t chunk,
                                                         float* __restrict__ part, int KVH,
                                                         const float* __restrict__ wts,
                                                         const uint16_t* __restrict__ q, int H, int w,
                                                         float* __restrict__ qpart) {
  pdl_wait();  // previous kernel on the stream complete and visible
  constexpr int TPR = D / 8;
  constexpr int RPP = 256 / TPR;  // rows per pass
  __shared__ float red[RPP][D + 1];
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int bk = b * KVH + kvh;
  const int c = threadIdx.x % TPR, rl = threadIdx.x / TPR;
  const int64_t r0 = (int64_t)split * chunk, r1 = std::min(nrows, r0 + chunk);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* Kb = K + b * sb + kvh * sh;
  // four rows per thread in flight: their indices first, then their loads
  constexpr int U = 4;
  for (int64_t rb = r0 + rl; rb < r1; rb += U * RPP) {
    int64_t j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = rb + (int64_t)u * RPP;
      j[u] = -1;
      if (r < r1) {
        j[u] = idx ? (int64_t)__ldg(idx + (int64_t)bk * k + r) : r;
        if (j[u] >= S) {
          set_device_status(KVC_ERR_DEVICE_BOUNDS);
          j[u] = -1;
        }
      }
    }
    uint4 v[U];
    float wj[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      v[u] = j[u] >= 0 ? ld16(Kb + j[u] * ss + c * 8) : make_uint4(0u, 0u, 0u, 0u);
      wj[u] = (wts && j[u] >= 0) ? __ldg(wts + (int64_t)bk * S + j[u]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (wts) {
        float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        acc_sq8(t, v[u]);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[u], t[i], acc[i]);
      } else {
        acc_sq8(acc, v[u]);  // zero rows (index -1 or past the range) add nothing
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[rl][c * 8 + i] = acc[i];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += 256) {
    float s = 0.f;
    for (int rr = 0; rr < RPP; ++rr) s += red[rr][d];
    part[((int64_t)split * gridDim.z * KVH + bk) * D + d] = s;
  }
  if (q == nullptr) return;
  __syncthreads();  // red is reused
  q_sq_partial<D>(q, H, w, KVH, b, kvh, split, gridDim.x, gridDim.z * KVH, red, qpart);
}

// cs[b*KVH+kvh][d] = the sum of the key-range partials: one CTA per (b, kvh), thread (grp, d)
// adding every ngrp-th range with its loads in flight at once, the groups then added in
// shared memory in group order
__global__ void __launch_bounds__(1024) k_channel_sum(const float* __restrict__ part, int nsplit, int rows, int D,
                                                      float* __restrict__ cs) {
  pdl_wait();  // previous kernel on the stream complete and visible
  __shared__ float red[16][128];
  const int bk = blockIdx.x;
  const int d = threadIdx.x % D, grp = threadIdx.x / D, ngrp = blockDim.x / D;
  constexpr int BATCH = 16;
  float acc = 0.f;
  for (int s0 = grp; s0 < nsplit; s0 += BATCH * ngrp) {
    float v[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int sp = s0 + u * ngrp;
      v[u] = sp < nsplit ? __ldg(part + ((int64_t)sp * rows + bk) * D + d) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) acc += v[u];
  }
  red[grp][d] = acc;
  __syncthreads();
  if (grp == 0) {
    float t = 0.f;
    for (int g2 = 0; g2 < ngrp; ++g2) t += red[g2][d];
    cs[(int64_t)bk * D + d] = t;
  }
}

// one CTA per (b, kvh): thread (grp, d) adds every ngrp-th split's key and query partials of
// channel d, all of its loads in flight at once; the groups are then added in shared memory
// in group order, and cs = (query sum / G) * key sum
__global__ void __launch_bounds__(1024) k_channel_final(const float* __restrict__ part,
                                                        const float* __restrict__ qpart, int nsplit, int B,
                                                        int KVH, int G, int D, float* __restrict__ cs) {
  pdl_wait();  // previous kernel on the stream complete and visible
  __shared__ float qred[16][128];
  __shared__ float kred[16][128];
  const int bk = blockIdx.x;
  const int d = threadIdx.x % D, grp = threadIdx.x / D, ngrp = blockDim.x / D;
  constexpr int BATCH = 16;
  float kn = 0.f, sq = 0.f;
  for (int s0 = grp; s0 < nsplit; s0 += BATCH * ngrp) {
    float kv[BATCH], qv[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int sp = s0 + u * ngrp;
      const int64_t o = ((int64_t)sp * B * KVH + bk) * D + d;
      kv[u] = sp < nsplit ? __ldg(part + o) : 0.f;
      qv[u] = sp < nsplit ? __ldg(qpart + o) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      kn += kv[u];
      sq += qv[u];
    }
  }
  qred[grp][d] = sq;
  kred[grp][d] = kn;
  __syncthreads();
  if (grp == 0) {
    float qs = 0.f, ks = 0.f;
    for (int g2 = 0; g2 < ngrp; ++g2) {
      qs += qred[g2][d];
      ks += kred[g2][d];
    }
    cs[(int64_t)bk * D + d] = (qs / (float)G) * ks;
  }
}

// ----------------------------------------------------------------------------------------
// ThinK channel pruning
// ----------------------------------------------------------------------------------------
// The C highest channel scores of row bk (ties: the lower channel), as an ascending channel list
// in chs (shared memory).  Every CTA of the row takes the same decision from the same scores, so
// the list needs no launch of its own; the row's first CTA also writes it to ch.  Threads
// d < D (D <= 128) rank channel d; the block has at least D threads.
__device__ __forceinline__ void select_channels(const float* __restrict__ cs, int bk, int D, int C, int32_t* chs,
                                                int32_t* __restrict__ ch) {
  __shared__ float v[128];
  __shared__ uint32_t wb[4];
  const int d = threadIdx.x;
  if (d < D) v[d] = cs[(int64_t)bk * D + d];
  __syncthreads();
  bool sel = false;
  if (d < D) {
    const float x = v[d];
    int rank = 0;
    for (int e = 0; e < D; ++e) {
      const float y = v[e];
      rank += (y > x) || (y == x && e < d);
    }
    sel = rank < C;
  }
  const int lane = d & 31, warp = d >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, sel);
  if (lane == 0 && warp < 4) wb[warp] = __popc(bal);
  __syncthreads();
  if (sel) {
    int base = 0;
    for (int q = 0; q < warp; ++q) base += wb[q];
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    chs[pos] = d;
    if (blockIdx.x == 0) ch[(int64_t)bk * C + pos] = d;
  }
  __syncthreads();
}

// compact mode: ch = the selected channels, Ko[b,kvh,t,c] = K[b,kvh,t,ch[c]] — 64 rows per
// pass staged in shared memory.  Each thread's 16-byte loads of a pass are in flight together,
// the first pass's during the channel selection and each next pass's during this pass's stores.
template <int D>
__global__ void __launch_bounds__(256) k_channel_gather(const float* __restrict__ cs, const uint16_t* __restrict__ K,
                                                        int64_t sb, int64_t sh, int64_t ss, int64_t S, int KVH,
                                                        int32_t* __restrict__ ch, int C,
                                                        uint16_t* __restrict__ Ko) {
  pdl_wait();  // previous kernel on the stream complete and visible
  constexpr int NT = 256, TPR = D / 8, RB = 64, LPT = RB * TPR / NT;
  static_assert(LPT * NT == RB * TPR, "whole rows per pass");
  __shared__ __align__(16) uint16_t tile[RB][D + 8];
  __shared__ int32_t chs[128];
  const int tid = threadIdx.x;
  const int bk = blockIdx.y;
  const int64_t b = bk / KVH, kvh = bk % KVH;
  const uint16_t* Kb = K + b * sb + kvh * sh;
  uint16_t* Ob = Ko + (int64_t)bk * S * C;
  const int64_t step = (int64_t)gridDim.x * RB;
  uint4 buf[LPT];
  auto load = [&](int64_t r0) {
#pragma unroll
    for (int u = 0; u < LPT; ++u) {
      const int x = u * NT + tid, r = x / TPR, c = x % TPR;
      buf[u] = r0 + r < S ? ld16(Kb + (r0 + r) * ss + c * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int64_t r0 = (int64_t)blockIdx.x * RB;
  if (r0 < S) load(r0);
  select_channels(cs, bk, D, C, chs, ch);  // (ends with a block barrier)
  const int out_chunks = C / 8;
  for (; r0 < S; r0 += step) {
#pragma unroll
    for (int u = 0; u < LPT; ++u) {
      const int x = u * NT + tid, r = x / TPR, c = x % TPR;
      *reinterpret_cast<uint4*>(&tile[r][c * 8]) = buf[u];
    }
    __syncthreads();
    if (r0 + step < S) load(r0 + step);
    for (int x = tid; x < RB * out_chunks; x += NT) {
      const int r = x / out_chunks, oc = x % out_chunks;
      if (r0 + r >= S) continue;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = tile[r][chs[oc * 8 + 2 * i] & (D - 1)];
        const uint32_t hi = tile[r][chs[oc * 8 + 2 * i + 1] & (D - 1)];
        w[i] = lo | (hi << 16);
      }
      st16(Ob + (r0 + r) * C + oc * 8, make_uint4(w[0], w[1], w[2], w[3]));
    }
    __syncthreads();  // the tile is rewritten next pass
  }
}

// zero mode: Ko = K with unselected channels zeroed (Ko dense [B,KVH,S,D]; may equal K)
template <int D>
__global__ void __launch_bounds__(256) k_channel_zero(const float* __restrict__ cs, const uint16_t* K, int64_t sb,
                                                      int64_t sh, int64_t ss, int64_t S, int KVH,
                                                      int32_t* __restrict__ ch, int C, uint16_t* Ko) {
  pdl_wait();  // previous kernel on the stream complete and visible
  constexpr int TPR = D / 8;
  __shared__ uint32_t keepw[4];
  __shared__ int32_t chs[128];
  const int bk = blockIdx.y;
  const int64_t b = bk / KVH, kvh = bk % KVH;
  if (threadIdx.x < 4) keepw[threadIdx.x] = 0;
  select_channels(cs, bk, D, C, chs, ch);  // (ends with a block barrier)
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const int d = chs[c];
    atomicOr(&keepw[d >> 5], 1u << (d & 31));
  }
  __syncthreads();
  const uint16_t* Kb = K + b * sb + kvh * sh;
  uint16_t* Ob = Ko + (int64_t)bk * S * D;
  const int64_t total = S * TPR;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = x / TPR;
    const int c = (int)(x % TPR);
    uint4 v = *reinterpret_cast<const uint4*>(Kb + r * ss + c * 8);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d0 = c * 8 + 2 * i, d1 = d0 + 1;
      if (!((keepw[d0 >> 5] >> (d0 & 31)) & 1u)) w[i] &= 0xffff0000u;
      if (!((keepw[d1 >> 5] >> (d1 & 31)) & 1u)) w[i] &= 0x0000ffffu;
    }
    *reinterpret_cast<uint4*>(Ob + r * D + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Row ranges per (b, kvh) for the channel sums: about per_sm CTAs per SM over all units, at
// least 64 rows each.  Measured best on the ThinK 128K shapes: 2 for the compaction (fewer,
// longer CTAs overlap their stores with the next rows' loads), 8 for the weighted value sums.
constexpr int SPLITS_COMPACT = 2, SPLITS_PLAIN = 4, SPLITS_WEIGHTED = 8;
int channel_splits(const kvc_kv_desc& kv, int64_t nrows, int per_sm) {
  const int64_t units = (int64_t)kv.B * kv.KVH;
  const int64_t target = (int64_t)num_sms() * per_sm;
  int64_t ns = std::max<int64_t>(1, (target + units - 1) / units);
  ns = std::min<int64_t>(ns, std::max<int64_t>(1, nrows / 64));
  return (int)ns;
}

}  // namespace

cudaError_t launch_compact(const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv,
                           const int32_t* idx, int k, uint16_t* Ko, uint16_t* Vo, cudaStream_t st) {
  const int64_t rows = (int64_t)kv.B * kv.KVH * k;
  const int64_t warps = (rows + COMPACT_RPW - 1) / COMPACT_RPW;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((warps + 7) / 8, (int64_t)num_sms() * 16));
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(blocks), dim3(256), 0, st, attrs);
  cudaError_t e;
  if (kv.D == 64)
    e = cudaLaunchKernelEx(&cfg, k_compact<64>, K, V, kv.stride_b, kv.stride_h, kv.stride_s, kv.KVH, kv.S, idx, k, rows,
                           Ko, Vo);
  else
    e = cudaLaunchKernelEx(&cfg, k_compact<128>, K, V, kv.stride_b, kv.stride_h, kv.stride_s, kv.KVH, kv.S, idx, k,
                           rows, Ko, Vo);
  if (e != cudaSuccess) return e;
  return launched(1);
}

cudaError_t launch_weighted_channel_norm(const float* wts, const uint16_t* V, const kvc_kv_desc& kv, float* cs,
                                         void* ws, cudaStream_t st) {
  const int ns = channel_splits(kv, kv.S, SPLITS_WEIGHTED);
  // the caller's scratch is channel_score_workspace(kv, 0, false) bytes: 2 x ceil(4 x SMs /
  // units) partials per unit, never fewer than ceil(8 x SMs / units)
  if ((size_t)ns * kv.B * kv.KVH * kv.D * sizeof(float) > channel_score_workspace(kv, 0, false))
    return cudaErrorInvalidValue;
  const int64_t chunk = (kv.S + ns - 1) / ns;
  float* part = reinterpret_cast<float*>(ws);
  const dim3 grid(ns, kv.KVH, kv.B);
  cudaError_t e =
      kv.D == 64 ? launch_pdl(k_channel_partial<64>, grid, dim3(256), 0, st, V, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.S, (const int32_t*)nullptr, 0, kv.S, chunk, part, kv.KVH, wts,
                              (const uint16_t*)nullptr, 0, 0, (float*)nullptr)
                 : launch_pdl(k_channel_partial<128>, grid, dim3(256), 0, st, V, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.S, (const int32_t*)nullptr, 0, kv.S, chunk, part, kv.KVH, wts,
                              (const uint16_t*)nullptr, 0, 0, (float*)nullptr);
  if (e != cudaSuccess) return e;
  const int rows = kv.B * kv.KVH;
  e = launch_pdl(k_channel_sum, dim3((unsigned)rows), dim3(1024), 0, st, (const float*)part, ns, rows, kv.D, cs);
  if (e != cudaSuccess) return e;
  return launched(2);
}

cudaError_t launch_write_slots(const uint16_t* kn, const uint16_t* vn, const int32_t* slot,
                               uint16_t* K, uint16_t* V, const kvc_kv_desc& kv, cudaStream_t st) {
  const int rows = kv.B * kv.KVH;
  const int n = rows * (kv.D / 8);
  const int blocks = (n + 255) / 256;
  const cudaError_t e =
      kv.D == 64 ? launch_pdl(k_write_slots<64>, dim3(blocks), dim3(256), 0, st, kn, vn, slot, K, V, kv.stride_b,
                              kv.stride_h, kv.stride_s, kv.KVH, kv.S, rows)
                 : launch_pdl(k_write_slots<128>, dim3(blocks), dim3(256), 0, st, kn, vn, slot, K, V, kv.stride_b,
                              kv.stride_h, kv.stride_s, kv.KVH, kv.S, rows);
  if (e != cudaSuccess) return e;
  return launched(1);
}

// key partials, then query partials: [2][nsplit][B*KVH][D] floats
size_t channel_score_workspace(const kvc_kv_desc& kv, int k, bool has_idx) {
  const int64_t nrows = has_idx ? k : kv.S;
  const int ns = channel_splits(kv, nrows, SPLITS_PLAIN);
  return 2 * (size_t)ns * kv.B * kv.KVH * kv.D * sizeof(float);
}

cudaError_t launch_channel_score(const uint16_t* q, int w, const uint16_t* K, const kvc_kv_desc& kv,
                                 const int32_t* idx, int k, float* cs, void* ws, cudaStream_t st) {
  const int64_t nrows = idx ? k : kv.S;
  const int ns = channel_splits(kv, nrows, SPLITS_PLAIN);
  const int64_t chunk = (nrows + ns - 1) / ns;
  float* part = static_cast<float*>(ws);
  float* qpart = part + (size_t)ns * kv.B * kv.KVH * kv.D;
  dim3 grid(ns, kv.KVH, kv.B);
  cudaError_t e =
      kv.D == 64 ? launch_pdl(k_channel_partial<64>, grid, dim3(256), 0, st, K, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.S, idx, k, nrows, chunk, part, kv.KVH, (const float*)nullptr, q, kv.H, w, qpart)
                 : launch_pdl(k_channel_partial<128>, grid, dim3(256), 0, st, K, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.S, idx, k, nrows, chunk, part, kv.KVH, (const float*)nullptr, q, kv.H, w, qpart);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_channel_final, dim3(kv.B * kv.KVH), dim3(1024), 0, st, (const float*)part, (const float*)qpart, ns,
                 kv.B, kv.KVH, kv.H / kv.KVH, kv.D, cs);
  if (e != cudaSuccess) return e;
  return launched(2);
}

// key partials, then query partials, of the compaction that also scores the key channels
size_t compact_channels_workspace(const kvc_kv_desc& kv, int k) {
  return 2 * (size_t)channel_splits(kv, k, SPLITS_COMPACT) * kv.B * kv.KVH * kv.D * sizeof(float);
}

cudaError_t launch_compact_channels(const uint16_t* K, const uint16_t* V, const kvc_kv_desc& kv, const int32_t* idx,
                                    int k, uint16_t* Ko, uint16_t* Vo, const uint16_t* q, int w, float* cs, void* ws,
                                    cudaStream_t st) {
  const int ns = channel_splits(kv, k, SPLITS_COMPACT);
  const int64_t chunk = (k + ns - 1) / ns;
  float* part = static_cast<float*>(ws);
  float* qpart = part + (size_t)ns * kv.B * kv.KVH * kv.D;
  const dim3 grid(ns, kv.B * kv.KVH);
  cudaError_t e =
      kv.D == 64 ? launch_pdl(k_compact_ksq<64>, grid, dim3(256), 0, st, K, V, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.KVH, kv.S, idx, k, chunk, Ko, Vo, part, q, kv.H, w, qpart)
                 : launch_pdl(k_compact_ksq<128>, grid, dim3(256), 0, st, K, V, kv.stride_b, kv.stride_h, kv.stride_s,
                              kv.KVH, kv.S, idx, k, chunk, Ko, Vo, part, q, kv.H, w, qpart);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_channel_final, dim3(kv.B * kv.KVH), dim3(1024), 0, st, (const float*)part, (const float*)qpart, ns,
                 kv.B, kv.KVH, kv.H / kv.KVH, kv.D, cs);
  if (e != cudaSuccess) return e;
  return launched(2);
}

cudaError_t launch_channel_prune(const float* cs, const uint16_t* K, const kvc_kv_desc& kv, int C,
                                 int zero_mode, int32_t* ch, uint16_t* Ko, cudaStream_t st) {
  const int rows = kv.B * kv.KVH;
  cudaError_t e;
  const int per = (int)std::max<int64_t>(1, std::min<int64_t>((kv.S + 63) / 64, ((int64_t)num_sms() * 8 + rows - 1) / rows));
  const dim3 grid(per, rows);
  if (zero_mode)
    e = kv.D == 64 ? launch_pdl(k_channel_zero<64>, grid, dim3(256), 0, st, cs, K, kv.stride_b, kv.stride_h, kv.stride_s,
                                kv.S, kv.KVH, ch, C, Ko)
                   : launch_pdl(k_channel_zero<128>, grid, dim3(256), 0, st, cs, K, kv.stride_b, kv.stride_h, kv.stride_s,
                                kv.S, kv.KVH, ch, C, Ko);
  else
    e = kv.D == 64 ? launch_pdl(k_channel_gather<64>, grid, dim3(256), 0, st, cs, K, kv.stride_b, kv.stride_h, kv.stride_s,
                                kv.S, kv.KVH, ch, C, Ko)
                   : launch_pdl(k_channel_gather<128>, grid, dim3(256), 0, st, cs, K, kv.stride_b, kv.stride_h,
                                kv.stride_s, kv.S, kv.KVH, ch, C, Ko);
  if (e != cudaSuccess) return e;
  return launched(1);
}

KVC_TU_STATUS(gather)

}  // namespace kvc
