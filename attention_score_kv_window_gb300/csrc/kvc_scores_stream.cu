// Decode-step scoring streamed by TMA: one new query per head (G query rows per KV head,
// G <= 8) against every slot of the cache, the new token written into its slot on the way.
// Used for a TOVA decode step ("Add TOVA press": the last query's attention, averaged over all
// heads; the lowest-scored slot is evicted) and a Scissorhands update (cold-compress PR 11:
// attention mean-pooled over the grouped queries, "attention < 1/keys" flags recorded into the
// circular history).  Either a cluster of CTAs splits one (b, kvh)'s slots and exchanges the
// per-row (max, sum), or (TOVA, one CTA per (b, kvh)) the KVH CTAs of a batch row form the
// cluster: each keeps its head's probabilities in shared memory, every CTA averages a slice of
// slots over the heads through distributed shared memory and offers its eviction candidate to
// rank 0, which writes the evicted slot for every head: the whole step is one kernel.
//
// CTA: warp 8 is the producer (one thread issues TMA loads of 128-slot tiles, both 64-channel
// panels, 128-byte swizzle, into a ring of mbarrier-tracked stages, 128 KiB in flight);
// warps 0-7 each take one 16-slot m-tile of every tile: mma.sync m16n8k16 with the slots on M
// (ldmatrix of the swizzled panel, conflict-free) and the <= 8 query rows on N (in registers),
// so a thread holds two slots x two query rows.  Logits go to shared memory (log2 domain) for
// the output pass, and each thread keeps a running (max, sum) per query row.  The new token's
// slot is scored from the new key itself: the warp whose m-tile holds it writes k_new over the
// staged row before reading the tile (the cache row is being rewritten during the step).  Every wait is bounded (2 s, %globaltimer): on timeout
// KVC_ERR_TIMEOUT is recorded and copies in flight are waited for (bounded) before the CTA
// ends.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int ST_TILE = 128;                       // slots per TMA tile
constexpr int ST_CWARPS = 8;                       // consumer warps: one 16-slot m-tile each
constexpr int ST_THREADS = (ST_CWARPS + 1) * 32;   // + the producer warp
constexpr int ST_PRODUCER = ST_CWARPS;
constexpr int ST_RMAX = 8;                         // query rows per KV head (the MMA's N)
constexpr uint64_t ST_WAIT_NS = 2000000000ull;
constexpr int ST_LG_PAD = 4;                       // logit row stride = slots + 4 (spreads banks)
constexpr size_t ST_SMEM_MAX = 220 * 1024;         // dynamic shared memory limit requested

// default ring depth (128 / 96 KiB in flight), and the shallower ring that lets two CTAs of
// the head cluster share an SM (64 / 48 KiB)
template <int D>
constexpr int ring_deep() { return D == 128 ? 4 : 6; }
template <int D>
constexpr int ring_shallow() { return D == 128 ? 2 : 3; }

template <int D, int NS_ = ring_deep<D>()>
struct StreamLayout {
  static constexpr int NP = D / 64;                          // 64-channel panels
  static constexpr uint32_t PANEL = ST_TILE * 128;           // bytes
  static constexpr uint32_t STAGE = NP * PANEL;
  static constexpr int NS = NS_;                             // ring depth
  static constexpr uint32_t BARS = NS * STAGE;               // full[NS], empty[NS]
  static constexpr uint32_t MISC = BARS + 16 * NS;           // abort flag, slot, keys
  static constexpr uint32_t RED = MISC + 64;                 // float2 [8 warps][8 rows]
  static constexpr uint32_t XCH = RED + 8 * ST_RMAX * 8;     // float2 [8 ranks][8 rows], pushed by peers
  static constexpr uint32_t LG = XCH + 8 * ST_RMAX * 8;      // float [G][per + pad]
};

template <int D, int NS = ring_deep<D>()>
size_t stream_smem(int G, int per) {
  return StreamLayout<D, NS>::LG + (size_t)G * (per + ST_LG_PAD) * 4 + 1024;
}

struct StreamArgs {
  const uint16_t* q;   // [B, H, D]: one new query per head
  int B, H, KVH, G;    // G query rows per KV head
  int S;               // slots
  int per;             // slots per CTA (a multiple of 128)
  int split;           // CTAs per (b, kvh) (a cluster when > 1)
  float sl2;           // scale * log2(e)
  float inv_g;
  const uint32_t* live;  // [B*KVH][S/32] live words, or null (every slot live)
  int64_t live_words;
  const int32_t* wslot;  // TOVA: the new token's slot per (b, kvh)
  const uint16_t* knew;  // [B*KVH][D] the new token's key / value rows
  const uint16_t* vnew;
  uint16_t* Kc;          // the cache, written at the new token's slot
  uint16_t* Vc;
  int64_t sb, sh, ss;
  float* out;            // [B*KVH][S]: group-mean probabilities (unless allh_out is given)
  float* allh_out;       // TOVA in one kernel: [B*KVH][S] all-heads mean (cluster = the KVH heads)
  int32_t* allh_slot;    //   and the evicted slot per (b, kvh) (may alias wslot)
  kvc_sh_state shs;      // Scissorhands step (shs.B > 0)
  const int32_t* queue;
  int qm, qpos;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
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
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with the given parity; false: timed out (abort flag raised,
// KVC_ERR_TIMEOUT recorded) or another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > ST_WAIT_NS) {
      *abort_flag = 1;
      set_device_status(KVC_ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtimer();
  while (!mbar_try_wait(bar, parity)) {
    if (gtimer() - t0 > ST_WAIT_NS) return;
  }
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
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
__device__ __forceinline__ uint32_t map_rank(uint32_t local, unsigned int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(local), "r"(rank));
  return ra;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// running (max, sum) of exp2 over a row, updated with two values; the sum is rescaled only
// when the max grows
__device__ __forceinline__ void online2(float& m, float& l, float xa, float xb) {
  const float mx = fmaxf(xa, xb);
  if (mx > m) {
    l = (m == -CUDART_INF_F ? 0.f : l * ex2(m - mx)) + ex2(xa - mx) + ex2(xb - mx);
    m = mx;
  } else if (mx != -CUDART_INF_F) {
    l += ex2(xa - m) + ex2(xb - m);
  }
}
__device__ __forceinline__ void merge2(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn != -CUDART_INF_F) {
    l = l * ex2(m - mn) + l2 * ex2(m2 - mn);
    m = mn;
  }
}

// The cluster = the a.split CTAs of one (b, kvh), each over `per` slots, or (a.allh_out) the
// KVH CTAs of one batch row.
template <int D, int NS = ring_deep<D>()>
__global__ void __launch_bounds__(ST_THREADS, NS == ring_shallow<D>() ? 2 : 1)
    k_scores_stream(const StreamArgs a, const __grid_constant__ CUtensorMap tmK) {
  using L = StreamLayout<D, NS>;
  constexpr int KS = D / 16;
  constexpr int CH = D / 8;  // 16-byte pieces per row
  extern __shared__ unsigned char smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = su32(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  unsigned int cs, cr;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cs));
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(cr));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::MISC);
  int* s_slot = reinterpret_cast<int*>(base + L::MISC + 16);  // [0] the new token's slot, [1] live keys
  float2* red = reinterpret_cast<float2*>(base + L::RED);
  float2* xch = reinterpret_cast<float2*>(base + L::XCH);
  const int lgs = a.per + ST_LG_PAD;
  float* lg = reinterpret_cast<float*>(base + L::LG);  // [G][lgs]
  auto full = [&](int s) { return sbase + L::BARS + 8u * s; };
  auto empty = [&](int s) { return sbase + L::BARS + 8u * (L::NS + s); };

  const int split = a.split;
  const unsigned int sr = split > 1 ? cr : 0u;  // this CTA's slice of the row
  const int64_t bk = blockIdx.x / split;
  const int b = (int)(bk / a.KVH), kvh = (int)(bk % a.KVH);
  const int kbeg = (int)sr * a.per;
  const int kend = min(a.S, kbeg + a.per);
  const int len = kend > kbeg ? kend - kbeg : 0;
  const int ntiles = (len + ST_TILE - 1) / ST_TILE;
  const int R = a.G;

  // the key tensor map's descriptor fetched while the barriers are set up and the previous
  // kernel finishes (it is a launch parameter, not an output of that kernel)
  if (warp == ST_PRODUCER && lane == 0)
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
  if (tid == 0) {
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), ST_CWARPS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  pdl_wait();  // previous kernel on the stream complete and visible

  // the producer fills the ring at once (no stage is in use yet)
  int issued = 0;
  if (warp == ST_PRODUCER && lane == 0) {
    for (; issued < ntiles && issued < L::NS; ++issued) {
      mbar_expect_tx(full(issued), L::STAGE);
      for (int p = 0; p < L::NP; ++p)
        tma_load_4d(sbase + issued * L::STAGE + p * L::PANEL, &tmK, p * 64, kbeg + issued * ST_TILE, kvh, b,
                    full(issued));
    }
  }

  // B operand of the consumer warps: query row g (< R), channels ks*16 + 2t4 (+1) and + 8,
  // loaded before the slot search so that the loads overlap it
  const uint16_t* qg = a.q + ((int64_t)b * a.H + (int64_t)kvh * a.G) * D;  // the group's query rows
  uint32_t bq[KS][2];
  if (warp != ST_PRODUCER) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const bool rv = g < R;
      bq[ks][0] = rv ? __ldg(reinterpret_cast<const uint32_t*>(qg + (int64_t)g * D + ks * 16 + 2 * t4)) : 0u;
      bq[ks][1] = rv ? __ldg(reinterpret_cast<const uint32_t*>(qg + (int64_t)g * D + ks * 16 + 8 + 2 * t4)) : 0u;
    }
  }

  // the new token: its slot (TOVA: given; Scissorhands: the lowest free slot, or the queued
  // one) and, Scissorhands, the live keys once it is in
  if (a.shs.B) {
    __shared__ int s_cnt[ST_THREADS / 32], s_free[ST_THREADS / 32];
    const int nw = a.shs.cap / 32;
    const uint32_t* lwr = a.shs.live + bk * nw;
    int cnt = 0, ff = 0x7fffffff;
    for (int x = tid; x < nw; x += ST_THREADS) {
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
    if (tid == 0) {
      cnt = 0;
      ff = 0x7fffffff;
      for (int q = 0; q < ST_THREADS / 32; ++q) {
        cnt += s_cnt[q];
        ff = min(ff, s_free[q]);
      }
      int f, keys;
      if (a.queue) {
        f = __ldg(a.queue + bk * a.qm + a.qpos);
        if (f >= 0 && f < a.S && !((lwr[f >> 5] >> (f & 31)) & 1u)) f = -1;  // a queued slot must be live
        keys = cnt;
      } else {
        f = ff < a.S ? ff : -1;
        keys = cnt + 1;
      }
      if (f < 0 || f >= a.S) {
        if (sr == 0) set_device_status(KVC_ERR_DEVICE_BOUNDS);
        if (keys > 0 && !a.queue) --keys;  // nothing was inserted
        f = -1;
      }
      s_slot[0] = f;
      s_slot[1] = keys;
    }
  } else if (tid == 0) {
    int f = a.wslot ? __ldg(a.wslot + bk) : -1;
    if (a.wslot && (f < 0 || f >= a.S)) {
      if (sr == 0) set_device_status(KVC_ERR_DEVICE_BOUNDS);
      f = -1;
    }
    s_slot[0] = f;
    s_slot[1] = 0;
  }
  __syncthreads();
  const int fslot = s_slot[0];
  const int keys = s_slot[1];
  const int wf = (fslot >= kbeg && fslot < kend) ? fslot - kbeg : -1;  // slice-relative
  if (wf >= 0 && warp == 0 && lane < CH) {  // the cache rows for later steps
    const int64_t off = (int64_t)b * a.sb + (int64_t)kvh * a.sh + (int64_t)fslot * a.ss + lane * 8;
    *reinterpret_cast<uint4*>(a.Kc + off) = *reinterpret_cast<const uint4*>(a.knew + bk * D + lane * 8);
    if (a.Vc) *reinterpret_cast<uint4*>(a.Vc + off) = *reinterpret_cast<const uint4*>(a.vnew + bk * D + lane * 8);
  }

  // Scissorhands (deep ring, one CTA per SM): the history state of this thread's first NPRE
  // output-pass iterations is loaded now, so its latency runs under the stream instead of
  // stalling the output pass (the kernel writes that state only in the output pass)
  constexpr bool PRE = NS != ring_shallow<D>();
  constexpr int OB = 4, NPRE = PRE ? 2 : 1;
  const int64_t nwl = a.shs.cap / 32;
  uint32_t pre_l[NPRE][OB], pre_h[NPRE][OB];
  int32_t pre_i[NPRE][OB];
  uint32_t pre_w[NPRE][OB];
  if (PRE && a.shs.B) {
    const int64_t plane = ((a.shs.t % a.shs.history) * a.shs.B * a.shs.KVH + bk) * nwl;
#pragma unroll
    for (int it = 0; it < NPRE; ++it)
#pragma unroll
      for (int u = 0; u < OB; ++u) {
        const int j0 = warp * 32 + it * OB * ST_THREADS + u * ST_THREADS;
        pre_l[it][u] = pre_h[it][u] = pre_w[it][u] = 0u;
        pre_i[it][u] = 0;
        if (j0 < len) {
          const int64_t gj = kbeg + j0 + lane;
          const int64_t x = bk * a.shs.cap + gj;
          pre_l[it][u] = a.shs.live[bk * nwl + (gj >> 5)];
          pre_h[it][u] = a.shs.hist[plane + (gj >> 5)];
          pre_i[it][u] = a.shs.insert_step[x];
          pre_w[it][u] = a.shs.low_count[x];
        }
      }
  }

  if (warp == ST_PRODUCER) {
    if (lane == 0) {
      for (int it = issued; it < ntiles; ++it) {
        const int s = it % L::NS;
        if (!wait_bar(empty(s), ((uint32_t)(it / L::NS) & 1u) ^ 1u, abort_flag)) break;
        mbar_expect_tx(full(s), L::STAGE);
        for (int p = 0; p < L::NP; ++p)
          tma_load_4d(sbase + s * L::STAGE + p * L::PANEL, &tmK, p * 64, kbeg + it * ST_TILE, kvh, b, full(s));
        issued = it + 1;
      }
      // copies still in flight when the consumers stopped early are waited for (bounded)
      if (*abort_flag)
        for (int it = (issued > L::NS ? issued - L::NS : 0); it < issued; ++it)
          drain_bar(full(it % L::NS), (uint32_t)(it / L::NS) & 1u);
    }
  } else {
    const int r0 = 2 * t4, r1 = r0 + 1;
    const bool v0 = r0 < R, v1 = r1 < R;
    const uint32_t* lw = a.live ? a.live + bk * a.live_words : nullptr;
    float m0 = -CUDART_INF_F, l0 = 0.f, m1 = -CUDART_INF_F, l1 = 0.f;
    const int rr = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;  // tile row this lane addresses
    // the new token's key, lane l < D/8 holding 16-byte piece l (written over its slot's staged row)
    uint4 knp = make_uint4(0u, 0u, 0u, 0u);
    if (wf >= 0 && lane < CH) knp = __ldg(reinterpret_cast<const uint4*>(a.knew + bk * D) + lane);
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % L::NS;
      const int key0 = it * ST_TILE + warp * 16;  // slice-relative
      const uint32_t word = (lw && key0 < len) ? __ldg(lw + ((kbeg + key0) >> 5)) : 0xffffffffu;
      if (!wait_bar(full(s), (uint32_t)(it / L::NS) & 1u, abort_flag)) break;
      const uint32_t st = sbase + s * L::STAGE;
      const bool has_new = wf >= key0 && wf < key0 + 16;  // warp-uniform
      if (has_new) {
        // the slot's cache row is being rewritten: score k_new instead, staged in its place
        const int rw = wf - it * ST_TILE;  // tile row
        if (lane < CH) {
          const int pnl = lane >> 3, chk = lane & 7;
          const uint32_t dst = st + pnl * L::PANEL + rw * 128 + ((chk ^ (rw & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(knp.x), "r"(knp.y), "r"(knp.z),
                       "r"(knp.w)
                       : "memory");
        }
        __syncwarp();
      }
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t af[4];
        const int chunk = ((ks & 3) << 1) + (lane >> 4);
        ldsm_x4(st + (ks >> 2) * L::PANEL + rr * 128 + ((chunk ^ (rr & 7)) << 4), af);
        mma16816(c, af, bq[ks][0], bq[ks][1]);
      }
      // generic-proxy writes to the stage (k_new) ordered before its next TMA fill
      if (has_new) asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));  // this warp has read the stage
      const int j1 = key0 + g, j2 = j1 + 8;
      const int sh = (kbeg + key0) & 31;
      const bool lv1 = j1 < len && (j1 == wf || ((word >> (sh + g)) & 1u));
      const bool lv2 = j2 < len && (j2 == wf || ((word >> (sh + g + 8)) & 1u));
      const float x00 = lv1 ? c[0] * a.sl2 : -CUDART_INF_F, x01 = lv1 ? c[1] * a.sl2 : -CUDART_INF_F;
      const float x10 = lv2 ? c[2] * a.sl2 : -CUDART_INF_F, x11 = lv2 ? c[3] * a.sl2 : -CUDART_INF_F;
      if (v0) {
        lg[r0 * lgs + j1] = x00;
        lg[r0 * lgs + j2] = x10;
        online2(m0, l0, x00, x10);
      }
      if (v1) {
        lg[r1 * lgs + j1] = x01;
        lg[r1 * lgs + j2] = x11;
        online2(m1, l1, x01, x11);
      }
    }
    // rows 2t4, 2t4 + 1: merge over the 8 lanes with the same t4, then the warps
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      merge2(m0, l0, __shfl_xor_sync(0xffffffffu, m0, o), __shfl_xor_sync(0xffffffffu, l0, o));
      merge2(m1, l1, __shfl_xor_sync(0xffffffffu, m1, o), __shfl_xor_sync(0xffffffffu, l1, o));
    }
    if (g == 0) {
      red[warp * ST_RMAX + r0] = make_float2(m0, l0);
      red[warp * ST_RMAX + r1] = make_float2(m1, l1);
    }
  }
  __syncthreads();
  // the next kernel (the all-heads mean and eviction of a TOVA step) may start launching: it
  // waits for this grid's completion before reading
  pdl_trigger();
  // this CTA's (max, sum) per query row; across the slices of a (b, kvh) through the cluster
  float M = -CUDART_INF_F, Ls = 0.f;
  if (tid < R) {
    for (int q = 0; q < ST_CWARPS; ++q) merge2(M, Ls, red[q * ST_RMAX + tid].x, red[q * ST_RMAX + tid].y);
    if (split > 1) {
      for (unsigned int p = 0; p < cs; ++p) {
        const uint32_t ra = map_rank(su32(&xch[cr * ST_RMAX + tid]), p);
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(ra), "f"(M), "f"(Ls) : "memory");
      }
    }
  }
  if (split > 1) cluster_sync();
  float* crow = reinterpret_cast<float*>(red);  // the merged normalisers (red is no longer read)
  __syncthreads();
  if (tid < R) {
    if (split > 1) {
      M = -CUDART_INF_F;
      Ls = 0.f;
      for (unsigned int p = 0; p < cs; ++p) {
        const float2 o = xch[p * ST_RMAX + tid];
        if (o.y > 0.f) merge2(M, Ls, o.x, o.y);
      }
    }
    crow[tid] = Ls > 0.f ? M + log2f(Ls) : CUDART_INF_F;
  }
  __syncthreads();
  float cv[ST_RMAX];
#pragma unroll
  for (int r = 0; r < ST_RMAX; ++r) cv[r] = r < R ? crow[r] : 0.f;

  // output pass: p = mean over the group's query rows of the probability (whole warps per 32
  // slots: a slice starts at a multiple of 128, and a Scissorhands row is whole live words).
  // The Scissorhands state of OB iterations is loaded before any is used (the loads overlap).
  const float thr = __fdiv_rn(1.0f, (float)(keys > 0 ? keys : 1));  // Scissorhands: float32(1)/float32(keys)
  for (int jb = warp * 32, oit = 0; jb < len; jb += OB * ST_THREADS, ++oit) {
    uint32_t lword[OB], hword[OB];
    int32_t insv[OB];
    uint16_t lowv[OB];
    if (PRE && a.shs.B && oit < NPRE) {
#pragma unroll
      for (int it = 0; it < NPRE; ++it)
        if (it == oit) {
#pragma unroll
          for (int u = 0; u < OB; ++u) {
            lword[u] = pre_l[it][u];
            hword[u] = pre_h[it][u];
            insv[u] = pre_i[it][u];
            lowv[u] = (uint16_t)pre_w[it][u];
          }
        }
    } else if (a.shs.B) {
#pragma unroll
      for (int u = 0; u < OB; ++u) {
        const int j0 = jb + u * ST_THREADS;
        lword[u] = hword[u] = 0u;
        insv[u] = 0;
        lowv[u] = 0;
        if (j0 < len) {
          const int64_t gj = kbeg + j0 + lane;
          const int64_t x = bk * a.shs.cap + gj;
          lword[u] = a.shs.live[bk * nwl + (gj >> 5)];
          hword[u] = a.shs.hist[((a.shs.t % a.shs.history) * a.shs.B * a.shs.KVH + bk) * nwl + (gj >> 5)];
          insv[u] = a.shs.insert_step[x];
          lowv[u] = a.shs.low_count[x];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < OB; ++u) {
      const int j0 = jb + u * ST_THREADS;
      if (j0 >= len) break;  // warp-uniform
      const int j = j0 + lane;
      const bool in = j < len;
      float sc = 0.f;
#pragma unroll
      for (int r = 0; r < ST_RMAX; ++r)
        if (r < R && in) sc += ex2(lg[r * lgs + j] - cv[r]);
      const float p = sc * a.inv_g;
      if (in) {
        if (a.allh_out) lg[j] = p;  // (row 0 of column j: read above by this thread only)
        else a.out[bk * a.S + kbeg + j] = p;
      }
      if (a.shs.B) {
        // record: lane l holds bit l of live word (kbeg + j0) / 32
        const int64_t gj = kbeg + j;
        const bool fresh = j == wf;
        const bool live = in && (fresh || ((lword[u] >> (gj & 31)) & 1u));
        const bool flag = live && p < thr;
        const uint32_t bits = __ballot_sync(0xffffffffu, flag);
        if (live) {
          const int64_t x = bk * a.shs.cap + gj;
          const int64_t ins = fresh ? a.shs.t : (int64_t)insv[u];
          const int oldbit = ((a.shs.t - ins) >= a.shs.history && ((hword[u] >> lane) & 1u)) ? 1 : 0;
          const int lw0 = fresh ? 0 : (int)lowv[u];
          a.shs.low_count[x] = (uint16_t)(lw0 + (flag ? 1 : 0) - oldbit);
          if (fresh) a.shs.insert_step[x] = (int32_t)a.shs.t;
        }
        if (lane == 0 && in)
          a.shs.hist[((a.shs.t % a.shs.history) * a.shs.B * a.shs.KVH + bk) * nwl + ((kbeg + j0) >> 5)] = bits;
      }
    }
  }
  if (a.shs.B && wf >= 0 && tid == 0) {  // the new token's slot is live from the next kernel on
    atomicOr(a.shs.live + bk * nwl + (fslot >> 5), 1u << (fslot & 31));
    a.shs.slot[bk] = fslot;
  }
  if (a.allh_out) {
    // TOVA eviction: slot j's score is the mean over the KV heads of their group-mean
    // probabilities (each head's row 0 of lg, read through the cluster); the evicted slot has
    // the lowest score, then the highest index (composite (~key, slot), largest wins)
    __shared__ unsigned long long wbest[ST_THREADS / 32], cbest[8];
    cluster_sync();  // every head's probabilities are in its CTA
    const int KV = (int)cs;
    const int per2 = (a.S + KV - 1) / KV;
    const int j0 = (int)cr * per2, j1 = min(a.S, j0 + per2);
    const float inv = 1.f / (float)KV;
    const int64_t row0 = (int64_t)b * KV;
    unsigned long long best = 0ull;
    for (int j = j0 + tid; j < j1; j += ST_THREADS) {
      const uint32_t la = su32(lg + j);
      // all heads' loads issued before the first add (KV <= 8), summed in head order
      float v[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        v[h] = 0.f;
        if (h < KV) asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v[h]) : "r"(map_rank(la, (unsigned)h)));
      }
      float sm = 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (h < KV) sm += v[h];
      sm *= inv;
      for (int h = 0; h < KV; ++h) a.allh_out[(row0 + h) * a.S + j] = sm;
      uint32_t u = __float_as_uint(sm);
      if (u == 0x80000000u) u = 0u;  // -0 ranks as +0
      const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      const unsigned long long c = ((unsigned long long)(~key) << 32) | (uint32_t)j;
      best = c > best ? c : best;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y > best ? y : best;
    }
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (tid == 0) {
      for (int q = 1; q < ST_THREADS / 32; ++q) best = wbest[q] > best ? wbest[q] : best;
      asm volatile("st.shared::cluster.u64 [%0], %1;\n" ::"r"(map_rank(su32(&cbest[cr]), 0u)), "l"(best) : "memory");
    }
    cluster_sync();  // (also: no CTA leaves while a peer may still read its probabilities)
    if (cr == 0 && tid < 32) {
      unsigned long long w = 0ull;
      for (int q = 0; q < KV; ++q) w = cbest[q] > w ? cbest[q] : w;
      for (int h = tid; h < KV; h += 32) a.allh_slot[row0 + h] = w ? (int32_t)(uint32_t)w : -1;
    }
  }
  // no remote access follows the last cluster barrier
}

// a.split CTAs per (b, kvh); the cluster is a.split CTAs, or the KVH heads in the TOVA mode
template <int D, int NS = ring_deep<D>()>
cudaError_t launch_stream_t(const StreamArgs& a, const kvc_kv_desc& kv, cudaStream_t st) {
  CUtensorMap tm;
  if (!make_cache_tensor_map(a.Kc, kv, &tm, ST_TILE)) return cudaErrorNotSupported;
  const size_t smem = stream_smem<D, NS>(a.G, a.per);
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(k_scores_stream<D, NS>), (int)ST_SMEM_MAX);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)kv.B * kv.KVH;
  const int cl = a.allh_out ? kv.KVH : a.split;
  cudaLaunchAttribute attrs[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(units * a.split)), dim3(ST_THREADS), smem, st, attrs, cl);
  e = cudaLaunchKernelEx(&cfg, k_scores_stream<D, NS>, a, tm);
  if (e != cudaSuccess) return e;
  return launched(1);
}

// Whether every head cluster of a one-kernel TOVA step is resident at once (clusters of KVH
// CTAs with the shallow ring, up to two CTAs per SM); cached per device and shape.
template <int D>
bool allh_clusters_fit(int KVH, int B, size_t smem) {
  constexpr int NS = ring_shallow<D>();
  struct Entry {
    int dev, KVH;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].KVH == KVH && cache[i].smem == smem) return cache[i].n >= B;
  auto kern = k_scores_stream<D, NS>;
  int n = 0;
  if (func_attrs_once(reinterpret_cast<const void*>(kern), (int)ST_SMEM_MAX) == cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = KVH;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)KVH);
    cfg.blockDim = dim3(ST_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  if (used < 16) cache[used++] = Entry{dev, KVH, smem, n};
  return n >= B;
}

// CTAs per (b, kvh): about one per SM over all rows, at most 8, every slice at least one
// tile, and the slice's logits within shared memory.  0: the shapes do not fit.
int stream_cluster(const kvc_kv_desc& kv, int* per_out) {
  const int G = kv.H / kv.KVH;
  const int64_t units = (int64_t)kv.B * kv.KVH;
  int cs = (int)std::max<int64_t>(1, std::min<int64_t>(8, num_sms() / std::max<int64_t>(1, units)));
  cs = (int)std::min<int64_t>(cs, (kv.S + ST_TILE - 1) / ST_TILE);
  for (;; ++cs) {
    const int per = (int)(((kv.S + cs - 1) / cs + ST_TILE - 1) / ST_TILE * ST_TILE);
    const size_t smem = kv.D == 64 ? stream_smem<64>(G, per) : stream_smem<128>(G, per);
    if (smem <= ST_SMEM_MAX) {
      *per_out = per;
      return cs;
    }
    if (cs >= 8) return 0;
  }
}

StreamArgs base_args(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                     const kvc_kv_desc& kv, float scale) {
  StreamArgs a{};
  a.q = q;
  a.B = kv.B;
  a.H = kv.H;
  a.KVH = kv.KVH;
  a.G = kv.H / kv.KVH;
  a.S = (int)kv.S;
  a.sl2 = scale * 1.4426950408889634f;
  a.inv_g = 1.f / (float)a.G;
  a.knew = knew;
  a.vnew = vnew;
  a.Kc = K;
  a.Vc = V;
  a.sb = kv.stride_b;
  a.sh = kv.stride_h;
  a.ss = kv.stride_s;
  return a;
}

bool stream_shape_ok(const kvc_kv_desc& kv) {
  const int G = kv.H / kv.KVH;
  return G <= ST_RMAX && (kv.D == 64 || kv.D == 128) && kv.S >= 1 && kv.S <= (1 << 24);
}

}  // namespace

cudaError_t launch_decode_scores_stream(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K,
                                        uint16_t* V, const kvc_kv_desc& kv, float scale, const int32_t* free_slot,
                                        float* group_scores, cudaStream_t st) {
  if (!stream_shape_ok(kv)) return cudaErrorNotSupported;
  int per = 0;
  const int cs = stream_cluster(kv, &per);
  if (cs == 0) return cudaErrorNotSupported;
  StreamArgs a = base_args(q, knew, vnew, K, V, kv, scale);
  a.per = per;
  a.split = cs;
  a.wslot = free_slot;
  a.out = group_scores;
  return kv.D == 64 ? launch_stream_t<64>(a, kv, st) : launch_stream_t<128>(a, kv, st);
}

cudaError_t launch_tova_step_stream(const uint16_t* q, const uint16_t* knew, const uint16_t* vnew, uint16_t* K,
                                    uint16_t* V, const kvc_kv_desc& kv, float scale, int32_t* free_slot, float* scores,
                                    cudaStream_t st) {
  if (!stream_shape_ok(kv) || kv.KVH > 8 || kv.KVH < 2) return cudaErrorNotSupported;
  int per = 0;
  if (stream_cluster(kv, &per) != 1) return cudaErrorNotSupported;  // one CTA per (b, kvh) only
  const int G = kv.H / kv.KVH;
  const size_t smem = kv.D == 64 ? stream_smem<64, ring_shallow<64>()>(G, per) : stream_smem<128, ring_shallow<128>()>(G, per);
  if (smem > ST_SMEM_MAX) return cudaErrorNotSupported;
  const bool fits = kv.D == 64 ? allh_clusters_fit<64>(kv.KVH, kv.B, smem) : allh_clusters_fit<128>(kv.KVH, kv.B, smem);
  if (!fits) return cudaErrorNotSupported;
  StreamArgs a = base_args(q, knew, vnew, K, V, kv, scale);
  a.per = per;
  a.split = 1;
  a.wslot = free_slot;
  a.allh_out = scores;
  a.allh_slot = free_slot;
  return kv.D == 64 ? launch_stream_t<64, ring_shallow<64>()>(a, kv, st)
                    : launch_stream_t<128, ring_shallow<128>()>(a, kv, st);
}

cudaError_t launch_sh_update_stream(const kvc_sh_state& sh, const int32_t* queue, int qm, int qpos, const uint16_t* q,
                                    const uint16_t* knew, const uint16_t* vnew, uint16_t* K, uint16_t* V,
                                    const kvc_kv_desc& kv, float scale, float* probs, cudaStream_t st) {
  if (!stream_shape_ok(kv)) return cudaErrorNotSupported;
  int per = 0;
  const int cs = stream_cluster(kv, &per);
  if (cs == 0) return cudaErrorNotSupported;
  StreamArgs a = base_args(q, knew, vnew, K, V, kv, scale);
  a.per = per;
  a.split = cs;
  a.live = sh.live;
  a.live_words = kv.S / 32;
  a.out = probs;
  a.shs = sh;
  a.queue = queue;
  a.qm = qm;
  a.qpos = qpos;
  return kv.D == 64 ? launch_stream_t<64>(a, kv, st) : launch_stream_t<128>(a, kv, st);
}

KVC_TU_STATUS(scores_stream)

}  // namespace kvc
