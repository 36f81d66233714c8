// Decoding over the channel-pruned key cache ("Add ThinK_Press", options 3b and 3c).
//
// k_decode_attn: attention of one new query per head over a cache whose keys keep Ck of the
// head's D channels.  Option 3c prunes the query to the kept channels (ch) and reads the
// pruned keys directly; with ch == null and Ck == D it is plain decoding attention (which is
// also what option 3b runs after k_zero_add_back rebuilt the full-width keys).
//
// The step is HBM-bound (Ck*2 + D*2 bytes per key against 4 heads x (Ck + D) multiply-adds),
// but done on CUDA cores its multiply-adds, shuffles and bf16 unpacking issue ~75 warp
// instructions per key, more than the SM can issue at HBM speed.  mma.sync m16n8k16 with the
// query heads as the 16 rows does a 16-key chunk's logits in 2 * Ck/16 instructions and its
// value product in 4 * D/16: the tensor cores here only save issue slots.  (tcgen05's
// smallest M is 64 and its accumulator would have to come back from TMEM every chunk.)
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kvc_decode.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int CHUNK = 16;   // keys per warp step (the k of the value product)
constexpr int WST = 2;      // per-warp ring stages
constexpr int HROWS = 16;   // query heads per CTA: the M of m16n8k16

// Warps per CTA and shared memory for a (kept key channels, head width) pair: per warp a
// ring of WST chunks, rows padded by 8 elements so that ldmatrix reads are conflict-free.
template <int CK, int D>
struct DaShape {
  static constexpr int PK = CK + 8, PV = D + 8;               // padded row pitches (elements)
  static constexpr uint32_t STAGE = CHUNK * (PK + PV) * 2;    // bytes per chunk
  static constexpr int NW = STAGE * WST * 16 <= 220 * 1024 ? 16 : 12;
  static constexpr int THREADS = NW * 32;
  static constexpr uint32_t SMEM = NW * WST * STAGE;
  static_assert(NW * HROWS * (D + 2) * 4 <= SMEM, "merge area");
};

struct DecodeArgs {
  const uint16_t* q;    // [B, H, D]
  const int32_t* ch;    // [B, KVH, Ck] kept channels or null
  const uint16_t* K;    // [B, KVH, S, Ck], rows dense
  const uint16_t* V;    // [B, KVH, S, D], rows dense
  int64_t ksb, ksh, vsb, vsh;
  int H, KVH, G;
  int64_t S;
  const uint32_t* live;
  int64_t live_words;
  float sl2;            // scale * log2(e)
  int nsplit;
  int64_t chunks;       // CHUNK-key chunks per row
  float* po;            // [rows][nsplit][G][D]
  float2* pml;          // [rows][nsplit][G]  (m in log2 units, l)
  float* out;           // [B, H, D]
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two floats -> bf16x2 (round to nearest even), first argument in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// p = hi + lo with hi = bf16(p) and lo = bf16(p - hi): 16 significant bits for the value
// product (a single bf16 rounding of p would bound its relative error only by 2^-9)
__device__ __forceinline__ void split_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(p0, p1);
  lo = pack_bf16(p0 - bf_lo(hi), p1 - bf_hi(hi));
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
#define NEG_INF (-__int_as_float(0x7f800000))

// One CTA per (b, kvh, key range, group of up to 16 query heads), one per SM.  Each warp
// streams its own 16-key chunks (chunk c of the range goes to warp c % NW) through a private
// two-stage cp.async ring, so the key loop has no block barrier:
//   logits  S[h, key] = q[h] . K[key]   m16n8k16 with the query heads as the 16 rows (A, held
//           in registers; option 3c gathers the kept channels into it) and the chunk's keys
//           as B (ldmatrix from the padded rows);
//   softmax online per warp in the log2 domain (running max and sum per head row);
//   values  O[h, :] += P[h, keys] V[keys, :]   the logits' accumulator layout is the A layout
//           of the next product, so P stays in registers, split into bf16 hi + lo halves;
//           V comes in with ldmatrix.trans.
// Dead or missing keys are zero-filled by the copy (no stale data reaches the products) and
// masked to -inf before the softmax.  The warps then merge through shared memory into one
// (m, l, o) partial per head; k_decode_combine merges the key ranges (when a row is one
// range, the kernel normalises and writes the output itself).
template <int CK, int D, bool H16>
__global__ void __launch_bounds__(DaShape<CK, D>::THREADS, 1) k_decode_attn(DecodeArgs a) {
  using Sh = DaShape<CK, D>;
  constexpr int NW = Sh::NW, PK = Sh::PK, PV = Sh::PV;
  constexpr int KS = CK / 16;  // k-steps of the logits
  constexpr int NT = D / 8;    // n-tiles of the value product
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x, row = blockIdx.y, hg = blockIdx.z;  // row = b * KVH + kvh
  const int b = row / a.KVH, kvh = row % a.KVH;
  const int64_t c0 = (int64_t)split * a.chunks / a.nsplit;
  const int64_t c1 = (int64_t)(split + 1) * a.chunks / a.nsplit;
  const int my = (int)((c1 - c0 - warp + NW - 1) / NW);  // chunks of this warp (may be 0)
  const uint16_t* Kg = a.K + (int64_t)b * a.ksb + (int64_t)kvh * a.ksh;
  const uint16_t* Vg = a.V + (int64_t)b * a.vsb + (int64_t)kvh * a.vsh;
  const uint32_t* lw = a.live ? a.live + (int64_t)row * a.live_words : nullptr;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + warp * WST * Sh::STAGE;
  pdl_wait();  // the previous kernel's writes (q, K, V, live) are visible from here on

  // chunk i of this warp -> stage st: K rows then V rows, 16 bytes per copy; rows past the
  // sequence or dead are zero-filled
  auto load_chunk = [&](int i, int st) {
    const int64_t j0 = (c0 + warp + (int64_t)i * NW) * CHUNK;
    const uint32_t sk = ring + st * Sh::STAGE, sv = sk + CHUNK * PK * 2;
    constexpr int KP = CK / 8, VP = D / 8;  // 16-byte pieces per row
#pragma unroll
    for (int x = lane; x < CHUNK * KP; x += 32) {
      const int r = x / KP, c = x % KP;
      const int64_t j = j0 + r;
      const bool ok = j < a.S && (lw == nullptr || ((__ldg(lw + (j >> 5)) >> (j & 31)) & 1u));
      cp_async16(sk + (uint32_t)(r * PK + c * 8) * 2, Kg + (ok ? j : 0) * CK + c * 8, ok ? 16 : 0);
    }
#pragma unroll
    for (int x = lane; x < CHUNK * VP; x += 32) {
      const int r = x / VP, c = x % VP;
      const int64_t j = j0 + r;
      const bool ok = j < a.S && (lw == nullptr || ((__ldg(lw + (j >> 5)) >> (j & 31)) & 1u));
      cp_async16(sv + (uint32_t)(r * PV + c * 8) * 2, Vg + (ok ? j : 0) * D + c * 8, ok ? 16 : 0);
    }
  };
  if (my > 0) load_chunk(0, 0);
  cp_async_commit();

  // query rows of this CTA as A fragments: rows gid (a0, a2) and gid + 8 (a1, a3); channel
  // c of the kept keys is channel ch[c] of the query
  uint32_t qa[KS][4];
  {
    const int h0 = hg * HROWS + gid, h1 = h0 + 8;
    const uint16_t* q0 = a.q + ((int64_t)b * a.H + (int64_t)kvh * a.G + h0) * D;
    const uint16_t* q1 = a.q + ((int64_t)b * a.H + (int64_t)kvh * a.G + h1) * D;
    auto qv = [&](const uint16_t* qh, bool hv, int c) -> uint32_t {
      int d = c;
      if (a.ch) {
        d = __ldg(a.ch + (int64_t)row * CK + c);
        if (d < 0 || d >= D) {
          set_device_status(KVC_ERR_DEVICE_BOUNDS);
          return 0u;
        }
      }
      return hv ? (uint32_t)__ldg(qh + d) : 0u;
    };
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int c = ks * 16 + 2 * tig;
      const bool v0 = h0 < a.G, v1 = H16 && h1 < a.G;
      qa[ks][0] = qv(q0, v0, c) | (qv(q0, v0, c + 1) << 16);
      qa[ks][1] = v1 ? (qv(q1, v1, c) | (qv(q1, v1, c + 1) << 16)) : 0u;
      qa[ks][2] = qv(q0, v0, c + 8) | (qv(q0, v0, c + 9) << 16);
      qa[ks][3] = v1 ? (qv(q1, v1, c + 8) | (qv(q1, v1, c + 9) << 16)) : 0u;
    }
  }

  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;  // rows gid and gid + 8
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int i = 0; i < my; ++i) {
    if (i + 1 < my) load_chunk(i + 1, (i + 1) % WST);
    cp_async_commit();
    cp_async_wait<1>();  // chunk i has landed (this lane's copies)
    __syncwarp();        // ... and every lane's
    const uint32_t sk = ring + (i % WST) * Sh::STAGE, sv = sk + CHUNK * PK * 2;
    // logits: n-tile 0 = keys 0-7, n-tile 1 = keys 8-15 of the chunk
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sk + (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * PK + ks * 16 + ((lane >> 3) & 1) * 8) * 2, b0, b1,
              b2, b3);
      mma_bf16(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }
    // mask and scale: this thread's keys are 8n + 2 tig + {0, 1}
    const int64_t j0 = (c0 + warp + (int64_t)i * NW) * CHUNK;
    const uint32_t lword = lw ? __ldg(lw + (j0 >> 5)) : 0xffffffffu;  // a chunk lies in one live word
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kk = 8 * n + 2 * tig + e;
        const int64_t j = j0 + kk;
        const bool ok = j < a.S && ((lword >> ((j0 & 31) + kk)) & 1u);
        s[n][e] = ok ? s[n][e] * a.sl2 : NEG_INF;
        s[n][e + 2] = ok ? s[n][e + 2] * a.sl2 : NEG_INF;
      }
    }
    // online softmax per head row (the 4 lanes of a row hold its 16 keys)
    float mt0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mt1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 1));
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 2));
    if (H16) {
      mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 1));
      mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 2));
    }
    const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
    const float r0 = mn0 == NEG_INF ? 1.f : ex2f(m0 - mn0);
    const float r1 = (!H16 || mn1 == NEG_INF) ? 1.f : ex2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float p[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      p[n][0] = mn0 == NEG_INF ? 0.f : ex2f(s[n][0] - mn0);
      p[n][1] = mn0 == NEG_INF ? 0.f : ex2f(s[n][1] - mn0);
      p[n][2] = (!H16 || mn1 == NEG_INF) ? 0.f : ex2f(s[n][2] - mn1);
      p[n][3] = (!H16 || mn1 == NEG_INF) ? 0.f : ex2f(s[n][3] - mn1);
    }
    l0 = l0 * r0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l1 = l1 * r1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
    if (__any_sync(0xffffffffu, r0 != 1.f || r1 != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= r0;
        o[n][1] *= r0;
        o[n][2] *= r1;
        o[n][3] *= r1;
      }
    }
    // P as the A operand (rows = heads, k = the chunk's 16 keys), hi and lo halves
    uint32_t ph[4], pl[4];
    split_bf16(p[0][0], p[0][1], ph[0], pl[0]);
    split_bf16(p[0][2], p[0][3], ph[1], pl[1]);
    split_bf16(p[1][0], p[1][1], ph[2], pl[2]);
    split_bf16(p[1][2], p[1][3], ph[3], pl[3]);
#pragma unroll
    for (int cb = 0; cb < NT / 2; ++cb) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sv + (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * PV + cb * 16 + (lane >> 4) * 8) * 2, b0, b1,
                b2, b3);
      mma_bf16(o[2 * cb], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_bf16(o[2 * cb], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_bf16(o[2 * cb + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_bf16(o[2 * cb + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
    __syncwarp();  // every lane is done with this stage before the next copy into it
  }
  cp_async_wait<0>();

  // ---- merge the warps: per head row its (m, l) and o[D] ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();  // every warp is done with its ring
  float* mw = reinterpret_cast<float*>(smem);  // [warp][HROWS][D + 2]: m, l, o[D]
  {
    float* e0 = mw + (warp * HROWS + gid) * (D + 2);
    float* e1 = mw + (warp * HROWS + gid + 8) * (D + 2);
    if (tig == 0) {
      e0[0] = m0;
      e0[1] = l0;
      e1[0] = m1;
      e1[1] = l1;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      *reinterpret_cast<float2*>(e0 + 2 + 8 * n + 2 * tig) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(e1 + 2 + 8 * n + 2 * tig) = make_float2(o[n][2], o[n][3]);
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < HROWS * D; x += Sh::THREADS) {
    const int g = x / D, d = x % D;
    const int gh = hg * HROWS + g;
    if (gh >= a.G) continue;
    float M = NEG_INF;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mw[(w * HROWS + g) * (D + 2)]);
    float ov = 0.f, lv = 0.f;
    if (M != NEG_INF) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* e = mw + (w * HROWS + g) * (D + 2);
        if (e[0] == NEG_INF) continue;  // a warp that saw no live key
        const float f = ex2f(e[0] - M);
        ov += e[2 + d] * f;
        lv += e[1] * f;
      }
    }
    if (a.nsplit == 1) {  // the CTA saw the whole row: normalise here, no combine kernel
      a.out[((int64_t)b * a.H + (int64_t)kvh * a.G + gh) * D + d] = lv > 0.f ? ov / lv : 0.f;
      continue;
    }
    const int64_t pi = ((int64_t)row * a.nsplit + split) * a.G + gh;
    a.po[pi * D + d] = ov;
    if (d == 0) a.pml[pi] = make_float2(M, lv);
  }
}

// One warp per (b, kvh, head of the group): merge the key ranges' partials and normalise.
template <int D>
__global__ void __launch_bounds__(256) k_decode_combine(DecodeArgs a, int64_t heads) {
  pdl_wait();
  const int64_t x = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (x >= heads) return;
  const int64_t row = x / a.G;
  const int g = (int)(x % a.G);
  constexpr int PER = D / 32;
  float M = NEG_INF;
  for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, __ldcg(&a.pml[(row * a.nsplit + s) * a.G + g].x));
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float ov[PER] = {}, lv = 0.f;
  if (M != NEG_INF) {
    for (int s = 0; s < a.nsplit; ++s) {
      const int64_t pi = (row * a.nsplit + s) * a.G + g;
      const float2 ml = __ldcg(&a.pml[pi]);
      const float f = ex2f(ml.x - M);
      lv += ml.y * f;
#pragma unroll
      for (int i = 0; i < PER; ++i) ov[i] += __ldcg(&a.po[pi * D + lane * PER + i]) * f;
    }
  }
  const int64_t b = row / a.KVH, kvh = row % a.KVH;
  float* dst = a.out + ((b * a.H) + kvh * a.G + g) * D + lane * PER;
  const float inv = lv > 0.f ? 1.f / lv : 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) dst[i] = ov[i] * inv;
}

// Option 3b: rebuild the full-width keys, zeros in the dropped channels.  One thread per
// 8 output channels of a row: it gathers them from the pruned row through the inverse map.
template <int D>
__global__ void __launch_bounds__(256) k_zero_add_back(const uint16_t* __restrict__ Kp, int C, int64_t psb,
                                                       int64_t psh, int64_t pss, const int32_t* __restrict__ ch,
                                                       uint16_t* __restrict__ Ko, int64_t osb, int64_t osh,
                                                       int64_t oss, int KVH, int64_t S) {
  __shared__ int16_t inv[D];  // output channel -> pruned channel, or -1
  pdl_wait();
  const int row = blockIdx.y;
  const int b = row / KVH, kvh = row % KVH;
  for (int d = threadIdx.x; d < D; d += blockDim.x) inv[d] = -1;
  __syncthreads();
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const int d = ch[(int64_t)row * C + c];
    if (d >= 0 && d < D) inv[d] = (int16_t)c;
    else set_device_status(KVC_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  constexpr int TPR = D / 8;  // threads per row
  const int64_t n = S * TPR;
  const uint16_t* src = Kp + (int64_t)b * psb + (int64_t)kvh * psh;
  uint16_t* dst = Ko + (int64_t)b * osb + (int64_t)kvh * osh;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = x / TPR;
    const int d0 = (int)(x % TPR) * 8;
    uint16_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = inv[d0 + i];
      v[i] = c >= 0 ? __ldg(src + j * pss + c) : (uint16_t)0;
    }
    uint4 w;
    w.x = v[0] | ((uint32_t)v[1] << 16);
    w.y = v[2] | ((uint32_t)v[3] << 16);
    w.z = v[4] | ((uint32_t)v[5] << 16);
    w.w = v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4*>(dst + j * oss + d0) = w;
  }
}

template <int CK, int D>
cudaError_t run_decode(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  using Sh = DaShape<CK, D>;
  auto kern = a.G > 8 ? k_decode_attn<CK, D, true> : k_decode_attn<CK, D, false>;
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(kern), (int)Sh::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(Sh::THREADS), Sh::SMEM, st, a);
}

}  // namespace

bool decode_shape_supported(int Ck, int D) {
  return (D == 64 || D == 128) && (Ck == 64 || Ck == 128) && Ck <= D;
}

DecodePlan plan_decode(const kvc_kv_desc& vd) {
  DecodePlan p;
  const int G = vd.H / vd.KVH;
  p.head_groups = (G + HROWS - 1) / HROWS;
  p.chunks = (vd.S + CHUNK - 1) / CHUNK;
  const int64_t units = (int64_t)vd.B * vd.KVH * p.head_groups;
  const int64_t sms = num_sms();  // one CTA per SM
  constexpr int64_t NW = 16;
  // the split count with the least modelled time: waves of CTAs times the chunks of the
  // busiest warp of a CTA, plus about one chunk's worth of per-CTA setup and merge
  const int64_t nmax = std::max<int64_t>(1, std::min<int64_t>(p.chunks / NW, 1024));
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int64_t n = 1; n <= nmax; ++n) {
    const int64_t waves = (units * n + sms - 1) / sms;
    const int64_t per_cta = (p.chunks + n - 1) / n;
    const int64_t cost = waves * ((per_cta + NW - 1) / NW + 1);
    if (cost < best_cost) {
      best_cost = cost;
      best = (int)n;
    }
  }
  p.nsplit = best;
  p.part_bytes = (size_t)vd.B * vd.KVH * p.nsplit * G * ((size_t)vd.D * 4 + 8);
  return p;
}

cudaError_t launch_decode_attention(const uint16_t* q, const int32_t* ch, const uint16_t* K, const kvc_kv_desc& kd,
                                    const uint16_t* V, const kvc_kv_desc& vd, const uint32_t* live, float scale,
                                    float* out, void* ws, cudaStream_t st) {
  const DecodePlan p = plan_decode(vd);
  DecodeArgs a;
  a.q = q;
  a.ch = ch;
  a.K = K;
  a.V = V;
  a.ksb = kd.stride_b;
  a.ksh = kd.stride_h;
  a.vsb = vd.stride_b;
  a.vsh = vd.stride_h;
  a.H = vd.H;
  a.KVH = vd.KVH;
  a.G = vd.H / vd.KVH;
  a.S = vd.S;
  a.live = live;
  a.live_words = (vd.S + 31) / 32;
  a.sl2 = scale * 1.4426950408889634f;
  a.nsplit = p.nsplit;
  a.chunks = p.chunks;
  const int64_t rows = (int64_t)vd.B * vd.KVH;
  a.po = reinterpret_cast<float*>(ws);
  a.pml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) + (size_t)rows * p.nsplit * a.G * vd.D * 4);
  a.out = out;
  const dim3 grid((unsigned)p.nsplit, (unsigned)rows, (unsigned)p.head_groups);
  const int Ck = kd.D, D = vd.D;
  cudaError_t e;
  if (Ck == 64 && D == 64) e = run_decode<64, 64>(a, grid, st);
  else if (Ck == 64 && D == 128) e = run_decode<64, 128>(a, grid, st);
  else if (Ck == 128 && D == 128) e = run_decode<128, 128>(a, grid, st);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  if (p.nsplit == 1) return launched(1);  // rows were not split: already normalised
  const int64_t heads = rows * a.G;
  const dim3 cgrid((unsigned)((heads + 7) / 8));
  e = D == 64 ? launch_pdl(k_decode_combine<64>, cgrid, dim3(256), 0, st, a, heads)
              : launch_pdl(k_decode_combine<128>, cgrid, dim3(256), 0, st, a, heads);
  if (e != cudaSuccess) return e;
  return launched(2);
}

cudaError_t launch_zero_add_back(const uint16_t* Kp, const kvc_kv_desc& pd, const int32_t* ch, uint16_t* Ko,
                                 const kvc_kv_desc& od, cudaStream_t st) {
  const int64_t rows = (int64_t)od.B * od.KVH;
  const int64_t per_row = od.S * (od.D / 8);
  const int64_t want = std::max<int64_t>(1, (int64_t)num_sms() * 8 / std::max<int64_t>(1, rows));
  const int64_t bx = std::min<int64_t>((per_row + 255) / 256, want);
  const dim3 grid((unsigned)std::max<int64_t>(1, bx), (unsigned)rows);
  const cudaError_t e =
      od.D == 64 ? launch_pdl(k_zero_add_back<64>, grid, dim3(256), 0, st, Kp, pd.D, pd.stride_b, pd.stride_h,
                              pd.stride_s, ch, Ko, od.stride_b, od.stride_h, od.stride_s, od.KVH, od.S)
                 : launch_pdl(k_zero_add_back<128>, grid, dim3(256), 0, st, Kp, pd.D, pd.stride_b, pd.stride_h,
                              pd.stride_s, ch, Ko, od.stride_b, od.stride_h, od.stride_s, od.KVH, od.S);
  if (e != cudaSuccess) return e;
  return launched(1);
}

KVC_TU_STATUS(decode)

}  // namespace kvc
