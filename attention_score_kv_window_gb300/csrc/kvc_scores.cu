// Window-attention token scores: s = scale * q_win K^T, a softmax over the whole sequence,
// then the sum over window rows of the head-mean probability ("Add TOVA press", SimJeg's
// shape walk-through; cold-compress PR 11, attention mean-pooled over grouped queries).
//
// The [H, w, S] probabilities never reach memory.  Two passes over K per (b, kvh):
//   pass 1 (queries on the MMA M axis): per query row, running max m and sum l of
//           exp2(s*log2e - m) over one key range -> partial (m, l) per range;
//   merge:  per row, combine the ranges -> c_r = M_r + log2(L_r)  (log2-domain normaliser);
//   pass 2 (keys on the MMA M axis): per key j, sum_r exp2(s_rj*log2e - c_r), times 1/G.
// Putting keys on M in pass 2 makes the reduction over query rows a per-thread sum plus a
// 4-lane shuffle, so no cross-warp column reduction is needed.
//
// Both passes stage K tiles (64 keys x D) in shared memory with a 3-stage cp.async
// pipeline and run bf16 mma.sync m16n8k16 with fp32 accumulation.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "kvc_internal.cuh"

namespace kvc {

namespace {

constexpr int TK = 64;        // keys per shared-memory tile
constexpr int NTHREADS = 256; // 8 warps
constexpr int STAGES = 3;
constexpr int P1_MAX_ROWS = 256;  // query rows per pass-1 CTA (row groups beyond)
constexpr int MAX_RPAD = 512;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
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
__device__ __forceinline__ bool live_bit(const uint32_t* lw, int64_t j) {
  return (__ldg(lw + (j >> 5)) >> (j & 31)) & 1u;
}
// last key index row r may see (-1: padded row)
__device__ __forceinline__ int64_t row_limit(const ScoresArgs& a, int r) {
  if (r >= a.R) return -1;
  return a.causal ? (a.S - a.w + (r % a.w)) : (a.S - 1);
}

// Stage K rows [kt0, kt0+TK) of one (b,kvh) into a shared tile (rows >= kend zero-filled).
template <int D>
__device__ __forceinline__ void load_k_tile(uint16_t* dst, const uint16_t* Kb, int64_t ss,
                                            int64_t kt0, int64_t kend, int tid) {
  constexpr int P = D + 8, CH = D / 8;
#pragma unroll
  for (int c = tid; c < TK * CH; c += NTHREADS) {
    const int r = c / CH, cc = c % CH;
    const int64_t j = kt0 + r;
    const bool ok = j < kend;
    const uint16_t* src = ok ? (Kb + j * ss + cc * 8) : Kb;
    cp_async16(smem_u32(dst + r * P + cc * 8), src, ok ? 16 : 0);
  }
}

// Stage query rows [row0, row0+rows) of the group (rows >= R zero-filled).
template <int D>
__device__ __forceinline__ void load_q_rows(uint16_t* dst, const uint16_t* Qg, int row0, int rows,
                                            int R, int tid) {
  constexpr int P = D + 8, CH = D / 8;
  for (int c = tid; c < rows * CH; c += NTHREADS) {
    const int r = c / CH, cc = c % CH;
    const int gr = row0 + r;
    const bool ok = gr < R;
    const uint16_t* src = ok ? (Qg + (int64_t)gr * D + cc * 8) : Qg;
    cp_async16(smem_u32(dst + r * P + cc * 8), src, ok ? 16 : 0);
  }
}

// ----------------------------------------------------------------------------------------
// pass 1: per-row (max, sum) over one key range
// ----------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(NTHREADS) k_scores_pass1(const ScoresArgs a) {
  pdl_wait();  // previous kernel on the stream complete and visible
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int P = D + 8, KS = D / 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y % a.KVH, rg = blockIdx.y / a.KVH;
  const int b = blockIdx.z;
  const int bk = b * a.KVH + kvh;
  const int row0 = rg * P1_MAX_ROWS;
  const int rows = min(P1_MAX_ROWS, a.Rpad - row0);
  const int n_mt = rows >> 4;
  int64_t kbeg, kend;
  key_range(a, split, &kbeg, &kend);
  const int ntiles = (int)((kend - kbeg + TK - 1) / TK);

  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + rows * P;
  float2* mrg = reinterpret_cast<float2*>(Ks + STAGES * TK * P);  // [8][16]

  const uint16_t* Kb = a.K + b * a.sb + kvh * a.sh;
  const uint16_t* Qg = a.q + ((int64_t)(b * a.H + kvh * a.G) * a.w) * D;
  const uint32_t* lw = a.live ? a.live + (int64_t)bk * a.live_words : nullptr;

  load_q_rows<D>(Qs, Qg, row0, rows, a.R, tid);
  cp_async_commit();
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ntiles) load_k_tile<D>(Ks + s * TK * P, Kb, a.ss, kbeg + (int64_t)s * TK, kend, tid);
    cp_async_commit();
  }

  // warp roles: >= 8 m-tiles: each warp owns up to 2 m-tiles and all keys of a tile;
  // fewer (1, 2 or 4): warps split the tile's 8 key n-tiles into kg groups.
  int kg, n_my, mt0, mt1, nt_begin;
  if (n_mt >= 8) {
    kg = 1; mt0 = warp; mt1 = warp + 8; n_my = (mt1 < n_mt) ? 2 : 1; nt_begin = 0;
  } else {
    // kg = largest power of two with n_mt * kg <= 8; warps beyond n_mt * kg stay idle
    kg = (n_mt == 1) ? 8 : (n_mt == 2 || n_mt == 3) ? 4 - 2 * (n_mt == 3) : (n_mt == 4) ? 2 : 1;
    mt0 = warp % n_mt; mt1 = mt0; nt_begin = warp / n_mt;
    n_my = (warp < n_mt * kg) ? 1 : 0;
  }
  const int nts = n_my ? 8 / kg : 0;  // n-tiles per warp per key tile

  int64_t lim[2][2];
  {
    const int rA0 = row0 + mt0 * 16 + g, rA1 = row0 + mt1 * 16 + g;
    lim[0][0] = row_limit(a, rA0);
    lim[0][1] = row_limit(a, rA0 + 8);
    lim[1][0] = row_limit(a, rA1);
    lim[1][1] = row_limit(a, rA1 + 8);
  }
  float m_run[2][2], l_run[2][2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h) { m_run[i][h] = -CUDART_INF_F; l_run[i][h] = 0.f; }

  uint32_t aq[2][KS][4];
  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int mt = mi == 0 ? mt0 : mt1;
        if (mi < n_my) {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int c = ks * 16 + ((lane >> 4) & 1) * 8;
            ldsm_x4(smem_u32(Qs + r * P + c), aq[mi][ks][0], aq[mi][ks][1], aq[mi][ks][2], aq[mi][ks][3]);
          }
        }
      }
    }
    {
      const int nx = it + STAGES - 1;
      if (nx < ntiles)
        load_k_tile<D>(Ks + (nx % STAGES) * TK * P, Kb, a.ss, kbeg + (int64_t)nx * TK, kend, tid);
      cp_async_commit();
    }
    const uint16_t* Kt = Ks + (it % STAGES) * TK * P;
    const int64_t kt0 = kbeg + (int64_t)it * TK;
    const bool clean = (kt0 + TK <= kend) && (lw == nullptr) && (!a.causal || kt0 + TK - 1 <= a.S - a.w);

    float c[2][8][4];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int nt = nt_begin + q * kg;
      if (q < nts) {
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[mi][q][e] = 0.f;
#pragma unroll
        for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
          uint32_t b0, b1, b2, b3;
          const int r = nt * 8 + (lane & 7);
          const int cc = ks2 * 32 + (lane >> 3) * 8;
          ldsm_x4(smem_u32(Kt + r * P + cc), b0, b1, b2, b3);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            if (mi < n_my) {
              mma16816(c[mi][q], aq[mi][2 * ks2], b0, b1);
              mma16816(c[mi][q], aq[mi][2 * ks2 + 1], b2, b3);
            }
          }
        }
      }
    }
    // online (max, sum) update per owned row
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      if (mi < n_my) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[16];
          float tmax = -CUDART_INF_F;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float x = -CUDART_INF_F;
              if (q < nts) {
                x = c[mi][q][2 * hh + e] * a.sl2;
                if (!clean) {
                  const int64_t j = kt0 + (nt_begin + q * kg) * 8 + 2 * t + e;
                  const bool vis = (j < kend) && (j <= lim[mi][hh]) && (lw == nullptr || live_bit(lw, j));
                  if (!vis) x = -CUDART_INF_F;
                } else if (lim[mi][hh] < 0) {
                  x = -CUDART_INF_F;
                }
              }
              v[q * 2 + e] = x;
              tmax = fmaxf(tmax, x);
            }
          }
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
          const float mnew = fmaxf(m_run[mi][hh], tmax);
          if (mnew != -CUDART_INF_F) {
            float s = l_run[mi][hh] * ex2(m_run[mi][hh] - mnew);
#pragma unroll
            for (int z = 0; z < 16; ++z) s += ex2(v[z] - mnew);
            l_run[mi][hh] = s;
            m_run[mi][hh] = mnew;
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  // reduce l over the quad (m is already quad-uniform)
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float l = l_run[mi][hh];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      l_run[mi][hh] = l;
    }
  if (kg == 1) {
    if (t == 0) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        if (mi < n_my) {
          const int r = row0 + (mi == 0 ? mt0 : mt1) * 16 + g;
          a.part[part_index(a, bk, r, split)] = range_lse(m_run[mi][0], l_run[mi][0]);
          a.part[part_index(a, bk, r + 8, split)] = range_lse(m_run[mi][1], l_run[mi][1]);
        }
      }
    }
  } else {
    __syncthreads();
    if (t == 0) {
      mrg[warp * 16 + g] = make_float2(m_run[0][0], l_run[0][0]);
      mrg[warp * 16 + g + 8] = make_float2(m_run[0][1], l_run[0][1]);
    }
    __syncthreads();
    if (tid < rows) {
      const int mt = tid >> 4, rr = tid & 15;
      float M = -CUDART_INF_F;
      for (int kgi = 0; kgi < kg; ++kgi) {
        const float2 v = mrg[(kgi * n_mt + mt) * 16 + rr];
        if (v.y > 0.f) M = fmaxf(M, v.x);
      }
      float L = 0.f;
      for (int kgi = 0; kgi < kg; ++kgi) {
        const float2 v = mrg[(kgi * n_mt + mt) * 16 + rr];
        if (v.y > 0.f) L += v.y * ex2(v.x - M);
      }
      a.part[part_index(a, bk, row0 + tid, split)] = range_lse(M, L);
    }
  }
}

// ----------------------------------------------------------------------------------------
// merge: per row, combine the key ranges' partials into one log2-domain normaliser
// ----------------------------------------------------------------------------------------
__global__ void k_scores_merge(const ScoresArgs a) {
  pdl_wait();  // previous kernel on the stream complete and visible
  const int bk = blockIdx.x;
  for (int r = threadIdx.x; r < a.Rpad; r += blockDim.x) a.mrow[(int64_t)bk * a.Rpad + r] = merge_row(a, bk, r);
}

// ----------------------------------------------------------------------------------------
// pass 2: per key, sum over query rows of exp2(s*log2e - c_r), times 1/G
// ----------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(NTHREADS) k_scores_pass2(const ScoresArgs a) {
  pdl_wait();  // previous kernel on the stream complete and visible
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int P = D + 8, KS = D / 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int bk = b * a.KVH + kvh;
  int64_t kbeg, kend;
  key_range(a, split, &kbeg, &kend);
  const int ntiles = (int)((kend - kbeg + TK - 1) / TK);
  const int Rpad = a.Rpad;

  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + Rpad * P;
  float* cr = reinterpret_cast<float*>(Ks + STAGES * TK * P);  // [Rpad]
  long long* lim = reinterpret_cast<long long*>(cr + Rpad);    // [Rpad] (8-byte aligned: Rpad%16==0)
  float* ksum = reinterpret_cast<float*>(lim + Rpad);          // [2][TK]

  const uint16_t* Kb = a.K + b * a.sb + kvh * a.sh;
  const uint16_t* Qg = a.q + ((int64_t)(b * a.H + kvh * a.G) * a.w) * D;
  const uint32_t* lw = a.live ? a.live + (int64_t)bk * a.live_words : nullptr;

  load_q_rows<D>(Qs, Qg, 0, Rpad, a.R, tid);
  cp_async_commit();
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ntiles) load_k_tile<D>(Ks + s * TK * P, Kb, a.ss, kbeg + (int64_t)s * TK, kend, tid);
    cp_async_commit();
  }
  for (int r = tid; r < Rpad; r += NTHREADS) {
    cr[r] = a.mrow[(int64_t)bk * Rpad + r] * a.pw;
    lim[r] = row_limit(a, r);
  }

  const int km = warp & 3;  // key m-tile (16 keys) inside the 64-key tile
  const int ch = warp >> 2; // half of the query-row n-tiles
  const int NT = Rpad >> 3;
  const int nt_lo = ch * (NT >> 1), nt_hi = nt_lo + (NT >> 1);
  float* out = a.out + (int64_t)bk * a.S;

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nx = it + STAGES - 1;
      if (nx < ntiles)
        load_k_tile<D>(Ks + (nx % STAGES) * TK * P, Kb, a.ss, kbeg + (int64_t)nx * TK, kend, tid);
      cp_async_commit();
    }
    const uint16_t* Kt = Ks + (it % STAGES) * TK * P;
    const int64_t kt0 = kbeg + (int64_t)it * TK;
    const bool clean = (kt0 + TK <= kend) && (lw == nullptr) && (!a.causal || kt0 + TK - 1 <= a.S - a.w);

    uint32_t ak[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int r = km * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = ks * 16 + ((lane >> 4) & 1) * 8;
      ldsm_x4(smem_u32(Kt + r * P + c), ak[ks][0], ak[ks][1], ak[ks][2], ak[ks][3]);
    }
    const int64_t jA = kt0 + km * 16 + g, jB = jA + 8;
    bool visA = true, visB = true;
    if (!clean) {
      visA = jA < kend && (lw == nullptr || live_bit(lw, jA));
      visB = jB < kend && (lw == nullptr || live_bit(lw, jB));
    }
    float acc0 = 0.f, acc1 = 0.f;
    for (int nt = nt_lo; nt < nt_hi; ++nt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
        uint32_t b0, b1, b2, b3;
        const int r = nt * 8 + (lane & 7);
        const int cc = ks2 * 32 + (lane >> 3) * 8;
        ldsm_x4(smem_u32(Qs + r * P + cc), b0, b1, b2, b3);
        mma16816(c, ak[2 * ks2], b0, b1);
        mma16816(c, ak[2 * ks2 + 1], b2, b3);
      }
      const int r0 = nt * 8 + 2 * t;
      const float c0 = cr[r0], c1 = cr[r0 + 1];
      const float sl2p = a.sl2 * a.pw;
      if (clean) {
        acc0 += ex2(fmaf(c[0], sl2p, -c0)) + ex2(fmaf(c[1], sl2p, -c1));
        acc1 += ex2(fmaf(c[2], sl2p, -c0)) + ex2(fmaf(c[3], sl2p, -c1));
      } else {
        const long long l0 = lim[r0], l1 = lim[r0 + 1];
        acc0 += ((visA && jA <= l0) ? ex2(fmaf(c[0], sl2p, -c0)) : 0.f) +
                ((visA && jA <= l1) ? ex2(fmaf(c[1], sl2p, -c1)) : 0.f);
        acc1 += ((visB && jB <= l0) ? ex2(fmaf(c[2], sl2p, -c0)) : 0.f) +
                ((visB && jB <= l1) ? ex2(fmaf(c[3], sl2p, -c1)) : 0.f);
      }
    }
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 1);
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, 2);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 1);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 2);
    if (t == 0) {
      ksum[ch * TK + km * 16 + g] = acc0;
      ksum[ch * TK + km * 16 + g + 8] = acc1;
    }
    __syncthreads();
    if (tid < TK) {
      const int64_t j = kt0 + tid;
      if (j < kend) out[j] = (ksum[tid] + ksum[TK + tid]) * a.out_mul;
    }
  }
  cp_async_wait<0>();
}

// ----------------------------------------------------------------------------------------
// single-pass kernel for few query rows (R = G*w <= 16: decode steps, TOVA): K is read once.
// A cluster of CS CTAs splits one (b, kvh)'s keys; each CTA keeps the logits of its slice in
// shared memory (log2 domain, masked ones -inf), computes per-row (max, sum), pushes them to
// every peer, and after one cluster barrier merges them and writes its slice's scores.
// ----------------------------------------------------------------------------------------
// per-warp ring stages of 8-key chunks: 64-channel rows are half as long, so twice the
// chunks stay in flight for the same bytes
constexpr int small_stages(int D) { return D == 64 ? 6 : 3; }
constexpr int SMALL_LOGIT_BYTES = 16 * 1024;  // per CTA; keeps three CTAs per SM

size_t smem_small(int D, int R, int64_t per) {
  return (size_t)(16 + 64 * small_stages(D)) * (D + 8) * 2 + (size_t)R * per * 4 + 16 * 8 * sizeof(float2) +
         8 * 16 * sizeof(float2) + 16 * sizeof(float) + 64;
}

__device__ __forceinline__ uint32_t cluster_addr_s(const void* local, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
               : "=r"(ra)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  return ra;
}

template <int D, bool R16>
__global__ void __launch_bounds__(NTHREADS, 3) k_scores_small(const ScoresArgs a, int64_t per) {
  pdl_wait();  // previous kernel on the stream complete and visible
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int P = D + 8, KS = D / 16;
  constexpr int RM = R16 ? 16 : 8;  // query rows the accumulators can hold
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  unsigned int cs, cr;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cs));
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(cr));
  const int bk = blockIdx.x / cs;
  const int b = bk / a.KVH, kvh = bk % a.KVH;
  const int R = a.R;
  const int64_t kbeg = (int64_t)cr * per;
  const int64_t kend = min(a.S, kbeg + per);
  const int len = kend > kbeg ? (int)(kend - kbeg) : 0;

  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + 16 * P;
  constexpr int WST = small_stages(D);  // stages per warp (8 warps x WST x 8 key rows)
  float* lg = reinterpret_cast<float*>(Ks + 64 * WST * P);                  // [R][per]
  float2* xch = reinterpret_cast<float2*>(lg + (int64_t)R * per);            // [8 ranks][16 rows], pushed by peers
  float2* red = xch + 8 * 16;                                                // [8 warps][16 rows]
  float* crow = reinterpret_cast<float*>(red + 8 * 16);                      // [16]

  const uint16_t* Kb = a.K + b * a.sb + kvh * a.sh;
  const uint16_t* Qg = a.q + ((int64_t)(b * a.H + kvh * a.G) * a.w) * D;
  const uint32_t* lw = a.live ? a.live + (int64_t)bk * a.live_words : nullptr;

  // Query rows once (all warps), then each warp streams its own 8-key chunks (chunk c of the
  // slice goes to warp c % 8) through a private ring of WST stages: no block barrier inside
  // the key loop, only the warp's own copies and a warp barrier.
  load_q_rows<D>(Qs, Qg, 0, 16, R, tid);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  uint32_t aq[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = ks * 16 + ((lane >> 4) & 1) * 8;
    ldsm_x4(smem_u32(Qs + r * P + c), aq[ks][0], aq[ks][1], aq[ks][2], aq[ks][3]);
  }
  constexpr int CH = D / 8;               // 16-byte pieces per key row
  constexpr int PPL = 8 * CH / 32;        // pieces per lane per chunk
  const uint32_t ring = smem_u32(Ks + warp * WST * 8 * P);
  const int nchunks = (len + 7) / 8;
  const int my = nchunks > warp ? (nchunks - warp + 7) / 8 : 0;
  // this lane's pieces of a chunk: rows r0 + RPP * u, the same 16 bytes of each
  constexpr int RPP = 32 / CH;            // key rows per 32 pieces
  const int r0 = lane / CH, cc = lane % CH;
  const uint32_t dlane = (uint32_t)(r0 * P + cc * 8) * 2;
  const int64_t slane = (int64_t)r0 * a.ss + cc * 8;
  // a decode step's new token: its slot (slice-relative) reads the new key instead of the cache
  int wf = -1;
  const uint16_t* knew_lane = nullptr;
  int keys = 0;  // Scissorhands: live keys once the new token is in
  if (a.wslot || a.shs.B) {
    int64_t f = -1;
    if (a.wslot) {
      f = __ldg(a.wslot + bk);
    } else {
      // every CTA of the row finds the lowest free slot (or reads the queued one) and counts
      // the live keys; the live words of the row are not written until after the scores
      __shared__ int s_cnt[NTHREADS / 32], s_free[NTHREADS / 32];
      const int nw = a.shs.cap / 32;
      const uint32_t* lwr = a.shs.live + (int64_t)bk * nw;
      int cnt = 0, ff = 0x7fffffff;
      for (int x = tid; x < nw; x += NTHREADS) {
        const uint32_t v = lwr[x];
        cnt += __popc(v);
        if (v != 0xffffffffu) ff = min(ff, x * 32 + __ffs(~v) - 1);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        ff = min(ff, __shfl_xor_sync(0xffffffffu, ff, o));
      }
      if (lane == 0) {
        s_cnt[warp] = cnt;
        s_free[warp] = ff;
      }
      __syncthreads();
      cnt = 0;
      ff = 0x7fffffff;
      for (int q = 0; q < NTHREADS / 32; ++q) {
        cnt += s_cnt[q];
        ff = min(ff, s_free[q]);
      }
      if (a.queue) {
        f = __ldg(a.queue + (int64_t)bk * a.qm + a.qpos);
        if (f >= 0 && f < a.S && !((lwr[f >> 5] >> (f & 31)) & 1u)) f = -1;  // a queued slot must be live
        keys = cnt;
      } else {
        f = ff < a.S ? ff : -1;
        keys = cnt + 1;
      }
    }
    if (f < 0 || f >= a.S) {
      if (tid == 0 && cr == 0) set_device_status(KVC_ERR_DEVICE_BOUNDS);
      if (a.shs.B && keys > 0 && !a.queue) --keys;  // nothing was inserted
    } else if (f >= kbeg && f < kend) {
      wf = (int)(f - kbeg);
      knew_lane = a.knew + (int64_t)bk * D + cc * 8;
      if (warp == 0 && lane < CH) {  // the cache row for later steps
        const int64_t off = b * a.sb + kvh * a.sh + (int64_t)f * a.ss + lane * 8;
        *reinterpret_cast<uint4*>(a.Kw + off) = *reinterpret_cast<const uint4*>(a.knew + (int64_t)bk * D + lane * 8);
        if (a.Vw) *reinterpret_cast<uint4*>(a.Vw + off) = *reinterpret_cast<const uint4*>(a.vnew + (int64_t)bk * D + lane * 8);
      }
    }
  }
  auto load_chunk = [&](int i, int st) {
    const int k0 = (warp + 8 * i) * 8;  // slice-relative
    const uint16_t* src0 = Kb + (kbeg + k0) * a.ss + slane;
    const uint32_t dst0 = ring + (uint32_t)(st * 8 * P) * 2 + dlane;
#pragma unroll
    for (int u = 0; u < PPL; ++u) {
      const int r = k0 + r0 + RPP * u;
      const bool ok = r < len;
      const uint16_t* src = ok ? src0 + (int64_t)RPP * u * a.ss : Kb;
      cp_async16(dst0 + (uint32_t)(RPP * u * P) * 2, r == wf ? knew_lane : src, ok ? 16 : 0);
    }
  };
#pragma unroll
  for (int st = 0; st < WST - 1; ++st) {
    if (st < my) load_chunk(st, st);
    cp_async_commit();
  }
  // row limits of the two rows this lane's accumulator fragment holds (slice-relative)
  const int64_t limA = (g < R) ? (a.causal ? a.S - a.w + (g % a.w) : a.S - 1) - kbeg : -1;
  const int64_t limB = (R16 && g + 8 < R) ? (a.causal ? a.S - a.w + ((g + 8) % a.w) : a.S - 1) - kbeg : -1;
  float* lgA = lg + (int64_t)g * per;
  float* lgB = lg + (int64_t)(g + 8) * per;
  // running (max, sum) of rows g and g + 8 over this lane's keys, log2 domain
  float mA = -CUDART_INF_F, lA = 0.f, mB = -CUDART_INF_F, lB = 0.f;
  for (int i = 0; i < my; ++i) {
    cp_async_wait<WST - 2>();
    __syncwarp();  // the chunk's rows, copied by all lanes, are visible; stage (i-1) % WST is free
    {
      const int nx = i + WST - 1;
      if (nx < my) load_chunk(nx, nx % WST);
      cp_async_commit();
    }
    const uint32_t kt = ring + (uint32_t)((i % WST) * 8 * P) * 2;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kt + (uint32_t)((lane & 7) * P + ks2 * 32 + (lane >> 3) * 8) * 2, b0, b1, b2, b3);
      mma16816(c, aq[2 * ks2], b0, b1);
      mma16816(c, aq[2 * ks2 + 1], b2, b3);
    }
    const int j0 = (warp + 8 * i) * 8 + 2 * t;  // slice-relative key of c[0]
    float sA[2], sB[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = j0 + e;
      const bool in = j < len;
      const bool lv = in && (lw == nullptr || j == wf || live_bit(lw, kbeg + j));
      sA[e] = (lv && j <= limA) ? c[e] * a.sl2 : -CUDART_INF_F;
      sB[e] = (lv && j <= limB) ? c[2 + e] * a.sl2 : -CUDART_INF_F;
      if (g < R && in) lgA[j] = sA[e];
      if (R16 && g + 8 < R && in) lgB[j] = sB[e];
    }
    {
      const float mn = fmaxf(mA, fmaxf(sA[0], sA[1]));
      if (mn != -CUDART_INF_F) {
        lA = lA * ex2(mA - mn) + ex2(sA[0] - mn) + ex2(sA[1] - mn);
        mA = mn;
      }
    }
    if (R16) {
      const float mn = fmaxf(mB, fmaxf(sB[0], sB[1]));
      if (mn != -CUDART_INF_F) {
        lB = lB * ex2(mB - mn) + ex2(sB[0] - mn) + ex2(sB[1] - mn);
        mB = mn;
      }
    }
  }
  cp_async_wait<0>();

  // rows' (max, sum): the 4 lanes of a row, then the 8 warps, then the cluster's CTAs
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
    if (R16) merge2(mB, lB, __shfl_xor_sync(0xffffffffu, mB, o), __shfl_xor_sync(0xffffffffu, lB, o));
  }
  if (t == 0) {
    red[warp * 16 + g] = make_float2(mA, lA);
    red[warp * 16 + g + 8] = make_float2(mB, lB);
  }
  __syncthreads();  // logits and warp partials complete
  if (tid < R) {
    float mm = -CUDART_INF_F, l = 0.f;
    for (int q = 0; q < NTHREADS / 32; ++q) merge2(mm, l, red[q * 16 + tid].x, red[q * 16 + tid].y);
    for (unsigned int p = 0; p < cs; ++p) {
      const uint32_t ra = cluster_addr_s(&xch[cr * 16 + tid], (int)p);
      asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(ra), "f"(mm), "f"(l) : "memory");
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
  if (tid < R) {
    float M = -CUDART_INF_F, L = 0.f;
    for (unsigned int p = 0; p < cs; ++p) {
      const float2 o = xch[p * 16 + tid];
      if (o.y > 0.f) merge2(M, L, o.x, o.y);
    }
    crow[tid] = L > 0.f ? M + log2f(L) : CUDART_INF_F;
  }
  __syncthreads();
  float* out = a.out + (int64_t)bk * a.S + kbeg;
  float cv[RM];
  const float pw = a.pw;
#pragma unroll
  for (int r = 0; r < RM; ++r) cv[r] = r < R ? crow[r] * pw : 0.f;
  const float thr = __fdiv_rn(1.0f, (float)(keys > 0 ? keys : 1));  // Scissorhands: float32(1)/float32(keys)
  for (int j = tid; j < len; j += NTHREADS) {
    float sc = 0.f;
#pragma unroll
    for (int r = 0; r < RM; ++r)
      if (r < R) sc += ex2(fmaf(lg[(int64_t)r * per + j], pw, -cv[r]));
    const float p = sc * a.out_mul;
    out[j] = p;
    if (a.shs.B) {
      // record: a slice is whole live words (it starts at a multiple of 64 keys and its
      // length is a multiple of 32), so lane l of a warp holds bit l of word (kbeg + j) / 32
      const int64_t gj = kbeg + j;
      const bool fresh = j == wf;
      const bool live = fresh || live_bit(lw, gj);
      const bool flag = live && p < thr;
      const uint32_t bits = __ballot_sync(0xffffffffu, flag);
      const int64_t nw = a.shs.cap / 32;
      uint32_t* hp = a.shs.hist + ((a.shs.t % a.shs.history) * a.shs.B * a.shs.KVH + bk) * nw + (gj >> 5);
      const uint32_t old = *hp;
      if (live) {
        const int64_t x = (int64_t)bk * a.shs.cap + gj;
        const int64_t ins = fresh ? a.shs.t : (int64_t)a.shs.insert_step[x];
        const int oldbit = ((a.shs.t - ins) >= a.shs.history && ((old >> lane) & 1u)) ? 1 : 0;
        const int lowv = fresh ? 0 : (int)a.shs.low_count[x];
        a.shs.low_count[x] = (uint16_t)(lowv + (flag ? 1 : 0) - oldbit);
        if (fresh) a.shs.insert_step[x] = (int32_t)a.shs.t;
      }
      __syncwarp();
      if (lane == 0) *hp = bits;
    }
  }
  if (a.shs.B && wf >= 0 && tid == 0) {  // the new token's slot is live from the next kernel on
    const int64_t f = kbeg + wf;
    atomicOr(a.shs.live + (int64_t)bk * (a.shs.cap / 32) + (f >> 5), 1u << (f & 31));
    a.shs.slot[bk] = (int32_t)f;
  }
  // no remote access follows the cluster barrier: CTAs may leave independently
}

// all-heads reduction: mean over KV heads of the per-group scores, written to every kvh
__global__ void k_scores_allheads(const float* __restrict__ grp, float* __restrict__ out, int B,
                                  int KVH, int64_t S) {
  pdl_wait();  // previous kernel on the stream complete and visible
  const int64_t n = (int64_t)B * S;
  const float inv = 1.f / (float)KVH;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = x / S, j = x % S;
    float s = 0.f;
    for (int kv = 0; kv < KVH; ++kv) s += grp[(b * KVH + kv) * S + j];
    s *= inv;
    for (int kv = 0; kv < KVH; ++kv) out[(b * KVH + kv) * S + j] = s;
  }
}

// TOVA decode: the all-heads mean (as k_scores_allheads) fused with the eviction of the
// lowest-ranked slot per batch row (lowest score; equal scores: the highest slot), written
// to slot[b*KVH+kvh] for every kvh.  A cluster of CTAs per batch row splits the slots; each
// CTA stores its best composite into rank 0's shared memory, and after one cluster barrier
// rank 0 picks the winner.
constexpr int EVICT_CLUSTER = 8;

__global__ void __launch_bounds__(256) k_allheads_evict1(const float* __restrict__ grp, float* __restrict__ out,
                                                         int KVH, int64_t S, int64_t per, int32_t* __restrict__ slot) {
  __shared__ unsigned long long wbest[8];
  __shared__ unsigned long long cbest[EVICT_CLUSTER];
  pdl_wait();  // previous kernel on the stream complete and visible
  unsigned int cs, cr;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cs));
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(cr));
  const int64_t b = blockIdx.x / cs;
  const int64_t j0 = (int64_t)cr * per, j1 = min(S, j0 + per);
  const float inv = 1.f / (float)KVH;
  unsigned long long best = 0ull;
  for (int64_t j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    float s = 0.f;
    for (int kv = 0; kv < KVH; ++kv) s += grp[(b * KVH + kv) * S + j];
    s *= inv;
    for (int kv = 0; kv < KVH; ++kv) out[(b * KVH + kv) * S + j] = s;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;  // -0 ranks as +0
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    // evicting: the composite (~key, slot) is largest for the lowest score, then the highest slot
    const unsigned long long c = ((unsigned long long)(~key) << 32) | (uint32_t)j;
    best = c > best ? c : best;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y > best ? y : best;
  }
  if ((threadIdx.x & 31) == 0) wbest[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (unsigned int q = 1; q < (blockDim.x >> 5); ++q) best = wbest[q] > best ? wbest[q] : best;
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
                 : "=r"(ra)
                 : "r"((uint32_t)__cvta_generic_to_shared(&cbest[cr])), "r"(0));
    asm volatile("st.shared::cluster.u64 [%0], %1;\n" ::"r"(ra), "l"(best) : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
  if (cr == 0 && threadIdx.x < 32) {
    unsigned long long w = 0ull;
    for (unsigned int q = 0; q < cs; ++q) w = cbest[q] > w ? cbest[q] : w;
    for (int kv = threadIdx.x; kv < KVH; kv += 32) slot[b * KVH + kv] = w ? (int32_t)(uint32_t)w : -1;
  }
  // no remote access follows the cluster barrier: CTAs may leave independently
}

size_t smem_pass1(int D, int rows) { return (size_t)(rows + STAGES * TK) * (D + 8) * 2 + 8 * 16 * sizeof(float2); }
size_t smem_pass2(int D, int Rpad) {
  return (size_t)(Rpad + STAGES * TK) * (D + 8) * 2 + (size_t)Rpad * (4 + 8) + 2 * TK * 4;
}

template <int D>
cudaError_t set_smem_attrs() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_scores_pass1<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_pass1(D, P1_MAX_ROWS));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_scores_pass2<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_pass2(D, MAX_RPAD));
  if (e != cudaSuccess) return e;
  for (auto kern : {k_scores_small<D, false>, k_scores_small<D, true>}) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_small(D, 16, SMALL_LOGIT_BYTES / (16 * 4)) + 1024);
    if (e != cudaSuccess) return e;
  }
  if (dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// Cluster size and keys per CTA for the single-pass small-row kernel; 0 when the logits of
// one (b, kvh) do not fit the shared memory of an 8-CTA cluster.  Among the sizes whose
// slices fit, the largest one whose clusters are all resident at once (as the occupancy
// calculator counts them: GPCs hold whole clusters, so fewer fit than SMs * 3 / size) with
// slices of at least 256 keys.
int64_t small_per(const ScoresArgs& a, int cs) { return ((a.S + cs - 1) / cs + TK - 1) / TK * TK; }

template <int D>
int max_active_clusters(const ScoresArgs& a, int cs) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int64_t, bool>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t per = small_per(a, cs);
  const auto key = std::make_tuple(dev, D, cs, (int64_t)a.R * per, a.R > 8);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3((unsigned)cs), dim3(NTHREADS), smem_small(D, a.R, per), nullptr, attrs, cs);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, a.R > 8 ? k_scores_small<D, true> : k_scores_small<D, false>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();  // clear the query's error; fall back to the SM count rule
    n = 3 * num_sms() / cs;
  }
  cache[key] = n;
  return n;
}

template <int D>
int small_cluster(const ScoresArgs& a, int64_t* per_out) {
  if (a.R > 16) return 0;
  const int64_t units = (int64_t)a.B * a.KVH;
  if (units * 8 > 2147483647LL) return 0;
  int cs_min = 1;
  while (cs_min <= 8 && (int64_t)a.R * small_per(a, cs_min) * 4 > SMALL_LOGIT_BYTES) ++cs_min;
  if (cs_min > 8) return 0;
  int cs = cs_min;
  for (int c = cs_min + 1; c <= 8; ++c) {
    if (small_per(a, c) < 256) break;
    if (units <= (int64_t)max_active_clusters<D>(a, c)) cs = c;
  }
  *per_out = small_per(a, cs);
  return cs;
}

template <int D>
cudaError_t launch_small(const ScoresArgs& a, int cs, int64_t per, cudaStream_t st) {
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)((int64_t)a.B * a.KVH * cs)), dim3(NTHREADS),
                                            smem_small(D, a.R, per), st, attrs, cs);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, a.R > 8 ? k_scores_small<D, true> : k_scores_small<D, false>, a, per);
  if (e != cudaSuccess) return e;
  return launched(1);
}

template <int D>
cudaError_t launch_impl(const ScoresArgs& a, int reduce, float* scores, cudaStream_t st) {
  cudaError_t e = set_smem_attrs<D>();
  if (e != cudaSuccess) return e;
  int64_t per = 0;
  const int cs = small_cluster<D>(a, &per);
  if (cs > 0) {
    e = launch_small<D>(a, cs, per, st);
    if (e != cudaSuccess) return e;
  } else if (tc_supported(a, D)) {
    e = launch_scores_tc(a, D, st);
    if (e != cudaSuccess) return e;
  } else {
    const int n_rg = (a.Rpad + P1_MAX_ROWS - 1) / P1_MAX_ROWS;
    const int rows1 = std::min(P1_MAX_ROWS, a.Rpad);
    dim3 g1(a.nsplit, a.KVH * n_rg, a.B);
    e = launch_pdl(k_scores_pass1<D>, g1, dim3(NTHREADS), smem_pass1(D, rows1), st, a);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_scores_merge, dim3(a.B * a.KVH), dim3(256), 0, st, a);
    if (e != cudaSuccess) return e;
    const dim3 g2(a.nsplit, a.KVH, a.B);
    e = launch_pdl(k_scores_pass2<D>, g2, dim3(NTHREADS), smem_pass2(D, a.Rpad), st, a);
    if (e != cudaSuccess) return e;
    e = launched(3);
    if (e != cudaSuccess) return e;
  }
  if (reduce == KVC_REDUCE_ALL_HEADS) {
    const int64_t n = (int64_t)a.B * a.S;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8);
    e = launch_pdl(k_scores_allheads, dim3(blocks), dim3(256), 0, st, (const float*)a.out, scores, a.B, a.KVH, a.S);
    if (e != cudaSuccess) return e;
    return launched(1);
  }
  return cudaGetLastError();
}

}  // namespace

ScoresPlan plan_scores(const kvc_kv_desc& kv, int w, int reduce) {
  ScoresPlan p{};
  const int G = kv.H / kv.KVH;
  p.R = G * w;
  if (p.R <= 16) p.Rpad = 16;
  else if (p.R <= 32) p.Rpad = 32;
  else if (p.R <= 64) p.Rpad = 64;
  else if (p.R <= 128) p.Rpad = 128;
  else if (p.R <= 256) p.Rpad = (p.R + 63) / 64 * 64;
  else p.Rpad = (p.R + 15) / 16 * 16;
  // key ranges of whole 128-key units, balanced: about one wave of CTAs for the tensor-core
  // shapes (one CTA per SM), four CTAs per SM for the small-row (decode) shapes
  const int64_t units = (int64_t)kv.B * kv.KVH;
  const int64_t target = (int64_t)num_sms() * (p.Rpad >= 64 ? 1 : 4);
  p.units = (kv.S + KEY_UNIT - 1) / KEY_UNIT;
  int64_t nsplit = std::max<int64_t>(1, target / units);
  nsplit = std::min<int64_t>(nsplit, std::max<int64_t>(1, p.units / 2));  // >= 2 units per range
  nsplit = std::min<int64_t>(nsplit, 65535);
  p.nsplit = (int)nsplit;
  p.part_bytes = (size_t)units * nsplit * p.Rpad * sizeof(float) + (size_t)units * p.Rpad * sizeof(float);
  p.part_bytes = (p.part_bytes + 255) / 256 * 256;
  p.sync_bytes = ((size_t)(1 + units * nsplit) * sizeof(unsigned long long) + 255) / 256 * 256;
  p.group_bytes = reduce == KVC_REDUCE_ALL_HEADS ? (size_t)units * kv.S * sizeof(float) : 0;
  return p;
}

size_t scores_workspace(const kvc_kv_desc& kv, int w, int reduce) {
  const ScoresPlan p = plan_scores(kv, w, reduce);
  return p.part_bytes + p.sync_bytes + p.group_bytes;
}

namespace {
ScoresArgs make_args(const uint16_t* q, const uint16_t* K, const kvc_kv_desc& kv, int w, float scale, int causal,
                     const uint32_t* live, int reduce, float* scores, void* ws, int power) {
  const ScoresPlan p = plan_scores(kv, w, reduce);
  ScoresArgs a{};
  a.q = q;
  a.K = K;
  a.sb = kv.stride_b;
  a.sh = kv.stride_h;
  a.ss = kv.stride_s;
  a.B = kv.B;
  a.H = kv.H;
  a.KVH = kv.KVH;
  a.w = w;
  a.G = kv.H / kv.KVH;
  a.R = p.R;
  a.Rpad = p.Rpad;
  a.S = kv.S;
  a.causal = causal;
  a.live = live;
  a.live_words = (kv.S + 31) / 32;
  a.sl2 = scale * 1.4426950408889634f;
  a.pw = (float)power;
  a.nsplit = p.nsplit;
  a.units = p.units;
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.part = reinterpret_cast<float*>(base);
  a.mrow = reinterpret_cast<float*>(base + (size_t)kv.B * kv.KVH * p.nsplit * p.Rpad * sizeof(float));
  a.sync = reinterpret_cast<unsigned long long*>(base + p.part_bytes);
  a.out = reduce == KVC_REDUCE_ALL_HEADS ? reinterpret_cast<float*>(base + p.part_bytes + p.sync_bytes) : scores;
  a.out_mul = 1.f / (float)a.G;
  a.wait_ns = 2000000000ull;
  a.withhold = -1;
  return a;
}
}  // namespace

cudaError_t launch_window_scores(const uint16_t* q, const uint16_t* K, const kvc_kv_desc& kv, int w,
                                 float scale, int causal, const uint32_t* live, int reduce,
                                 float* scores, void* ws, cudaStream_t st, int power) {
  const ScoresArgs a = make_args(q, K, kv, w, scale, causal, live, reduce, scores, ws, power);
  if (kv.D == 64) return launch_impl<64>(a, reduce, scores, st);
  return launch_impl<128>(a, reduce, scores, st);
}

cudaError_t launch_sh_update_fused(const kvc_sh_state& sh, const int32_t* queue, int qm, int qpos, const uint16_t* q,
                                   const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                                   const kvc_kv_desc& kv, float scale, float* probs, void* ws, cudaStream_t st) {
  {
    const cudaError_t es = launch_sh_update_stream(sh, queue, qm, qpos, q, knew, vnew, K, V, kv, scale, probs, st);
    if (es != cudaErrorNotSupported) return es;
  }
  ScoresArgs a = make_args(q, K, kv, 1, scale, 0, sh.live, KVC_REDUCE_GQA_GROUP, probs, ws, 1);
  int64_t per = 0;
  cudaError_t e0 = kv.D == 64 ? set_smem_attrs<64>() : set_smem_attrs<128>();
  if (e0 != cudaSuccess) return e0;
  const int cs = kv.D == 64 ? small_cluster<64>(a, &per) : small_cluster<128>(a, &per);
  if (cs == 0 || a.R > 16) return cudaErrorNotSupported;
  a.shs = sh;
  a.queue = queue;
  a.qm = qm;
  a.qpos = qpos;
  a.knew = knew;
  a.vnew = vnew;
  a.Kw = K;
  a.Vw = V;
  cudaError_t e = kv.D == 64 ? set_smem_attrs<64>() : set_smem_attrs<128>();
  if (e != cudaSuccess) return e;
  return kv.D == 64 ? launch_small<64>(a, cs, per, st) : launch_small<128>(a, cs, per, st);
}

cudaError_t launch_tova_decode(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                               const kvc_kv_desc& kv, float scale, int32_t* free_slot, float* scores, void* ws,
                               cudaStream_t st) {
  // the whole step in one kernel where its head clusters fit
  {
    const cudaError_t e1 = launch_tova_step_stream(q, knew, vnew, K, V, kv, scale, free_slot, scores, st);
    if (e1 != cudaErrorNotSupported) return e1;
  }
  ScoresArgs a = make_args(q, K, kv, 1, scale, 0, nullptr, KVC_REDUCE_ALL_HEADS, scores, ws, 1);
  // group-mean scores into the workspace: the TMA-streamed kernel, else the small-row kernel
  cudaError_t e = launch_decode_scores_stream(q, knew, vnew, K, V, kv, scale, free_slot, a.out, st);
  if (e == cudaErrorNotSupported) {
    int64_t per = 0;
    e = kv.D == 64 ? set_smem_attrs<64>() : set_smem_attrs<128>();
    if (e != cudaSuccess) return e;
    const int cs = kv.D == 64 ? small_cluster<64>(a, &per) : small_cluster<128>(a, &per);
    if (cs == 0) return cudaErrorNotSupported;
    a.wslot = free_slot;
    a.knew = knew;
    a.vnew = vnew;
    a.Kw = K;
    a.Vw = V;
    e = kv.D == 64 ? launch_small<64>(a, cs, per, st) : launch_small<128>(a, cs, per, st);
  }
  if (e != cudaSuccess) return e;
  const int ecs = EVICT_CLUSTER;
  const int64_t eper = (kv.S + ecs - 1) / ecs;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(kv.B * ecs)), dim3(256), 0, st, attrs, ecs);
  e = cudaLaunchKernelEx(&cfg, k_allheads_evict1, (const float*)a.out, scores, kv.KVH, kv.S, eper, free_slot);
  if (e != cudaSuccess) return e;
  return launched(1);
}

// ----------------------------------------------------------------------------------------
// Fixed scratch for kvc_window_scores_noalloc: a file-scope device array that every GPU
// which loads the library holds until the process exits.  Host code cannot use the array's
// name as a device address (it is a host-side stand-in), so the address is looked up once
// per device with cudaGetSymbolAddress while that device is current, and passed to the
// kernels like any caller-provided workspace.
// ----------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

cudaError_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

KVC_TU_STATUS(scores)

}  // namespace kvc
