// Window scores on the 5th-generation tensor cores: the same two-pass computation as the
// mma.sync path in kvc_scores.cu ("Add TOVA press": only the last w attention rows; cold-
// compress PR 11: mean over each KV head's grouped queries), rebuilt around tcgen05.
//
// One CTA per (b, kvh, key range), 10 warps:
//   warp 8  producer: TMA loads of the query group (once) and of 128-key K tiles into a
//           4-stage shared-memory ring (128-byte swizzle), mbarrier-tracked;
//   warp 9  MMA issuer: allocates all 512 TMEM columns (two 256-column accumulators) and
//           issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) from one thread; commits
//           free the K stage and publish the accumulator;
//   warps 0-7 epilogue: tcgen05.ld the accumulator, release it, then do the softmax math.
// pass 1: A = query rows (M = 128 per half), B = K tile (N = 128 keys): each epilogue thread
//         owns one query row, so its running max / sum over keys is thread-local.
// pass 2: A = K tile (M = 128 keys), B = the query group (N = Rpad rows): each thread owns
//         one key and sums exp2(s*log2e - c_r) over its half of the query rows.
// Every mbarrier wait is bounded (%globaltimer); on timeout the kernel records
// KVC_ERR_TIMEOUT, all roles leave their loops, and TMEM is released before exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int TILE = 128;           // keys per tile
constexpr int STAGES = 4;           // K ring depth
constexpr int EPI_WARPS = 16;       // 4 per SM sub-partition
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int THREADS = 576;
constexpr int QROWS_MAX = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s bound on any single wait

__host__ __device__ constexpr uint32_t qpanel_bytes() { return QROWS_MAX * 128; }
__host__ __device__ constexpr uint32_t kpanel_bytes() { return TILE * 128; }

// shared-memory layout behind a 1024-byte aligned base
template <int D>
struct Layout {
  static constexpr int NP = D / 64;  // 64-element (128-byte) panels along head_dim
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + NP * qpanel_bytes();
  static constexpr uint32_t STAGE = NP * kpanel_bytes();
  static constexpr uint32_t BARS = K + STAGES * STAGE;      // 2*STAGES + 5 mbarriers
  static constexpr uint32_t MISC = (BARS + 8 * (2 * STAGES + 5) + 15) / 16 * 16;  // tmem base, abort flag
  static constexpr uint32_t CR = MISC + 16;                 // float[256], 16-byte aligned (float4 reads)
  static constexpr uint32_t LIM = CR + 256 * 4;             // int[256]
  static constexpr uint32_t STAT = LIM + 256 * 4;           // float2[4][256]
  static constexpr uint32_t KSUM = STAT + 4 * 256 * 8;      // float[2][4][128]
  static constexpr uint32_t END = KSUM + 2 * 4 * 128 * 4;
  static constexpr size_t SMEM = END + 1024;                // + alignment slack
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
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
// Bounded wait for the phase with the given parity.  false: timed out (the abort flag is
// raised and KVC_ERR_TIMEOUT recorded) or another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > WAIT_NS) {
      *abort_flag = 1;
      set_device_status(KVC_ERR_TIMEOUT);
      return false;
    }
  }
}
// same, ignoring the abort flag (used only to drain copies already in flight at teardown)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtimer();
  while (!mbar_try_wait(bar, parity)) {
    if (gtimer() - t0 > WAIT_NS) return;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
          "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, bf16 in, fp32 accumulate
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Shared-memory operand descriptor: K-major, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row x 128-byte atoms, consecutive 8-row groups 1024 bytes
// apart.  A K step of 16 bf16 inside a 64-element panel advances the start address by 32 B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                    // leading byte offset (not used by this layout)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset between 8-row groups
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void named_sync_epilogue() { asm volatile("bar.sync 1, 512;\n" ::: "memory"); }

// 16 consecutive 32-bit TMEM columns of this thread's lane, then wait for the load
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit TMEM columns of this thread's lane, then wait for the load
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive 32-bit TMEM columns of this thread's lane, then wait for the load
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive 32-bit TMEM columns of this thread's lane, then wait for the load
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}


template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float* v) {
  if constexpr (NC == 16) {
    tmem_ld16(taddr, v);
  } else if constexpr (NC == 32) {
    tmem_ld32(taddr, v);
  } else if constexpr (NC == 48) {
    tmem_ld32(taddr, v);
    tmem_ld16(taddr + 32, v + 32);
  } else if constexpr (NC == 64) {
    tmem_ld64(taddr, v);
  } else if constexpr (NC == 96) {
    tmem_ld64(taddr, v);
    tmem_ld32(taddr + 64, v + 64);
  } else {
    tmem_ld128(taddr, v);
  }
}

__device__ __forceinline__ int row_limit_i(const ScoresArgs& a, int r) {
  if (r >= a.R) return -1;
  return a.causal ? (int)(a.S - a.w + (r % a.w)) : (int)(a.S - 1);
}

struct Ctx {
  uint8_t* base;
  uint32_t sbase;
  volatile int* abort_flag;
  uint32_t tmem;
  __device__ uint32_t full(int s) const { return sbase + BARS_OFF + 8 * s; }
  __device__ uint32_t empty(int s) const { return sbase + BARS_OFF + 8 * (STAGES + s); }
  __device__ uint32_t tfull(int b) const { return sbase + BARS_OFF + 8 * (2 * STAGES + b); }
  __device__ uint32_t tempty(int b) const { return sbase + BARS_OFF + 8 * (2 * STAGES + 2 + b); }
  __device__ uint32_t qfull() const { return sbase + BARS_OFF + 8 * (2 * STAGES + 4); }
  uint32_t BARS_OFF;
};

// common prologue: barriers, TMEM allocation (warp MMA_WARP)
template <int D>
__device__ __forceinline__ Ctx prologue(unsigned char* smem_raw) {
  using L = Layout<D>;
  Ctx c;
  c.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  c.sbase = su32(c.base);
  c.BARS_OFF = L::BARS;
  c.abort_flag = reinterpret_cast<volatile int*>(c.base + L::MISC + 4);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(c.full(s), 1);
      mbar_init(c.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.tfull(b), 1);
      mbar_init(c.tempty(b), EPI_WARPS);
    }
    mbar_init(c.qfull(), 1);
    *c.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(c.sbase + L::MISC),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *reinterpret_cast<volatile uint32_t*>(c.base + L::MISC);
  return c;
}

template <int D>
__device__ __forceinline__ void teardown(const Ctx& c) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(c.tmem), "r"(TMEM_COLS) : "memory");
  }
}

// producer: query group once, then the K ring
template <int D>
__device__ __forceinline__ void producer(const Ctx& c, const ScoresArgs& a, const CUtensorMap* tmK,
                                         const CUtensorMap* tmQ, int qrows, int kvh, int b, int64_t kbeg,
                                         int ntiles) {
  using L = Layout<D>;
  const int qrow0 = (b * a.H + kvh * a.G) * a.w;
  mbar_expect_tx(c.qfull(), (uint32_t)(L::NP * qrows * 128));
  for (int p = 0; p < L::NP; ++p) tma_load_2d(c.sbase + L::Q + p * qpanel_bytes(), tmQ, p * 64, qrow0, c.qfull());
  int issued = 0;
  for (int it = 0; it < ntiles; ++it) {
    const int s = it % STAGES;
    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
    if (!wait_bar(c.empty(s), ph ^ 1u, c.abort_flag)) break;
    mbar_expect_tx(c.full(s), L::STAGE);
    const int y = (int)(kbeg + (int64_t)it * TILE);
    for (int p = 0; p < L::NP; ++p)
      tma_load_4d(c.sbase + L::K + s * L::STAGE + p * kpanel_bytes(), tmK, p * 64, y, kvh, b, c.full(s));
    issued = it + 1;
  }
  // copies still in flight when the kernel stops early are waited for (bounded) before exit
  if (*c.abort_flag) {
    drain_bar(c.qfull(), 0);
    for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
      drain_bar(c.full(it % STAGES), (uint32_t)(it / STAGES) & 1u);
  }
}

// ----------------------------------------------------------------------------------------
// pass 1
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ float max8(const float* v, int n) {
  float m[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) m[q] = -CUDART_INF_F;
  for (int i = 0; i < n; i += 8) {
#pragma unroll
    for (int q = 0; q < 8; ++q) m[q] = fmaxf(m[q], v[i + q]);
  }
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}
// sum_i exp2(v_i * sl2 - off) with eight independent accumulators
template <int NC>
__device__ __forceinline__ float sum_exp8(const float* v, float sl2, float off) {
  float s[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) s[q] = 0.f;
#pragma unroll
  for (int i = 0; i < NC; i += 8) {
#pragma unroll
    for (int q = 0; q < 8; ++q) s[q] += ex2(fmaf(v[i + q], sl2, -off));
  }
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// Epilogue warp w reads columns [part*NC, part*NC + NC) of accumulator half h for the query
// rows of lane quadrant w%4; the row's (max, sum) is then merged over its NPART warps.
template <int D, int NHALF>
__global__ void __launch_bounds__(THREADS, 1)
    k_pass1_tc(const ScoresArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ) {
  using L = Layout<D>;
  constexpr int KS = D / 16;
  constexpr int NPART = 4 / NHALF;        // warps sharing one query row
  constexpr int NC = TILE / NPART;        // accumulator columns per warp
  extern __shared__ unsigned char smem_raw[];
  const Ctx c = prologue<D>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int bk = b * a.KVH + kvh;
  int64_t kbeg, kend;
  key_range(a, split, &kbeg, &kend);
  const int ntiles = (int)((kend - kbeg + TILE - 1) / TILE);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) producer<D>(c, a, &tmK, &tmQ, NHALF * 128, kvh, b, kbeg, ntiles);
  } else if (warp == MMA_WARP) {
    if (lane == 0 && wait_bar(c.qfull(), 0, c.abort_flag)) {
      int done = 0;
      constexpr uint32_t idesc = idesc_bf16(128, TILE);
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % STAGES, buf = it & 1;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u, bph = (uint32_t)(it >> 1) & 1u;
        if (!wait_bar(c.tempty(buf), bph ^ 1u, c.abort_flag)) break;
        if (!wait_bar(c.full(s), ph, c.abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < NHALF; ++h) {
          const uint32_t d = c.tmem + buf * 256 + h * 128;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t ad = sw128_desc(c.sbase + L::Q + (ks >> 2) * qpanel_bytes() + h * 128 * 128 + koff);
            const uint64_t bd = sw128_desc(c.sbase + L::K + s * L::STAGE + (ks >> 2) * kpanel_bytes() + koff);
            tc_mma(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
        }
        tc_commit(c.empty(s));
        tc_commit(c.tfull(buf));
        done = it + 1;
      }
      // stopped early: let the MMAs already issued finish before TMEM is released
      if (*c.abort_flag && done > 0) drain_bar(c.tfull((done - 1) & 1), (uint32_t)((done - 1) >> 1) & 1u);
    }
    __syncwarp();
  } else {
    // epilogue: one query row per thread and warp-part
    const int qd = warp & 3;
    const int h = NHALF == 2 ? ((warp >> 2) & 1) : 0;
    const int part = NHALF == 2 ? (warp >> 3) : (warp >> 2);
    const int c0 = part * NC;
    const int r = h * 128 + qd * 32 + lane;
    const int lim = row_limit_i(a, r);
    // (m, l): l = sum exp2(s*log2e - m).  m is a reference, not always the exact max: a tile
    // is accumulated against the current m unless its sum shows values more than 2^64 above
    // it, in which case the exact tile max is taken and l rescaled.
    float m = -CUDART_INF_F, l = 0.f;
    float v[NC];
    for (int it = 0; it < ntiles; ++it) {
      const int buf = it & 1;
      const uint32_t bph = (uint32_t)(it >> 1) & 1u;
      if (!wait_bar(c.tfull(buf), bph, c.abort_flag)) break;
      tc_fence_after();
      tmem_load_cols<NC>(c.tmem + ((uint32_t)(qd * 32) << 16) + buf * 256 + h * 128 + c0, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.tempty(buf));
      if (lim < 0) continue;
      const int64_t kt0 = kbeg + (int64_t)it * TILE + c0;
      const bool clean = (kt0 + NC <= kend) && (!a.causal || kt0 + NC - 1 <= (int64_t)lim);
      if (!clean) {
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int64_t j = kt0 + i;
          if (j >= kend || j > lim) v[i] = -CUDART_INF_F;
        }
      }
      if (m != -CUDART_INF_F) {
        const float t = sum_exp8<NC>(v, a.sl2, m);
        if (t <= 0x1p64f) {
          l += t;
          continue;
        }
      }
      const float mx = max8(v, NC);
      if (mx == -CUDART_INF_F) continue;
      const float mn = fmaxf(m, mx * a.sl2);
      l = l * ex2(m - mn) + sum_exp8<NC>(v, a.sl2, mn);
      m = mn;
    }
    // merge the NPART partial (m, l) of each row
    float2* stat = reinterpret_cast<float2*>(c.base + L::STAT);
    stat[part * 256 + r] = make_float2(m, l);
    named_sync_epilogue();
    if (part == 0) {
      float M = -CUDART_INF_F;
#pragma unroll
      for (int q = 0; q < NPART; ++q) {
        const float2 o = stat[q * 256 + r];
        if (o.y > 0.f) M = fmaxf(M, o.x);
      }
      float Lsum = 0.f;
#pragma unroll
      for (int q = 0; q < NPART; ++q) {
        const float2 o = stat[q * 256 + r];
        if (o.y > 0.f) Lsum += o.y * ex2(o.x - M);
      }
      if (r < a.Rpad) a.part[part_index(a, bk, r, split)] = make_float2(M, Lsum);
    }
  }
  teardown<D>(c);
}

// ----------------------------------------------------------------------------------------
// pass 2
// ----------------------------------------------------------------------------------------
// Epilogue warp w reads, for the 32 keys of lane quadrant w%4, the NQ query-row columns
// [(w/4)*NQ, (w/4)*NQ + NQ); the four partial key sums are added after a named barrier.
// The per-row normalisers c_r = M + log2(L) are merged from pass 1's key-range partials in
// the prologue (no separate merge launch).
template <int D, int NQ>
__global__ void __launch_bounds__(THREADS, 1)
    k_pass2_tc(const ScoresArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ) {
  using L = Layout<D>;
  constexpr int KS = D / 16;
  constexpr int N = 4 * NQ;
  extern __shared__ unsigned char smem_raw[];
  const Ctx c = prologue<D>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int bk = b * a.KVH + kvh;
  int64_t kbeg, kend;
  key_range(a, split, &kbeg, &kend);
  const int ntiles = (int)((kend - kbeg + TILE - 1) / TILE);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) producer<D>(c, a, &tmK, &tmQ, N, kvh, b, kbeg, ntiles);
  } else if (warp == MMA_WARP) {
    if (lane == 0 && wait_bar(c.qfull(), 0, c.abort_flag)) {
      int done = 0;
      constexpr uint32_t idesc = idesc_bf16(128, N);
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % STAGES, buf = it & 1;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u, bph = (uint32_t)(it >> 1) & 1u;
        if (!wait_bar(c.tempty(buf), bph ^ 1u, c.abort_flag)) break;
        if (!wait_bar(c.full(s), ph, c.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = c.tmem + buf * 256;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t koff = (ks & 3) * 32;
          const uint64_t ad = sw128_desc(c.sbase + L::K + s * L::STAGE + (ks >> 2) * kpanel_bytes() + koff);
          const uint64_t bd = sw128_desc(c.sbase + L::Q + (ks >> 2) * qpanel_bytes() + koff);
          tc_mma(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        tc_commit(c.empty(s));
        tc_commit(c.tfull(buf));
        done = it + 1;
      }
      if (*c.abort_flag && done > 0) drain_bar(c.tfull((done - 1) & 1), (uint32_t)((done - 1) >> 1) & 1u);
    }
    __syncwarp();
  } else {
    float* cr = reinterpret_cast<float*>(c.base + L::CR);
    int* limr = reinterpret_cast<int*>(c.base + L::LIM);
    float* ksum = reinterpret_cast<float*>(c.base + L::KSUM);
    // merge pass 1's key-range partials: c_r = M + log2(L), +inf when the row sees no key
    for (int r = threadIdx.x; r < N; r += EPI_WARPS * 32) {
      cr[r] = merge_row(a, bk, r);
      limr[r] = row_limit_i(a, r);
    }
    named_sync_epilogue();
    const int qd = warp & 3, cq = warp >> 2;
    const int kr = qd * 32 + lane;
    const float* crq = cr + cq * NQ;
    const int* limq = limr + cq * NQ;
    float* out = a.out + (int64_t)bk * a.S;
    bool dead = false;
    float v[NQ];
    for (int it = 0; it < ntiles; ++it) {
      const int buf = it & 1;
      const uint32_t bph = (uint32_t)(it >> 1) & 1u;
      const int64_t kt0 = kbeg + (int64_t)it * TILE;
      const int64_t j = kt0 + kr;
      float acc = 0.f;
      if (!dead && wait_bar(c.tfull(buf), bph, c.abort_flag)) {
        tc_fence_after();
        tmem_load_cols<NQ>(c.tmem + ((uint32_t)(qd * 32) << 16) + buf * 256 + cq * NQ, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.tempty(buf));
        const bool clean = (kt0 + TILE <= kend) && (!a.causal || kt0 + TILE - 1 <= a.S - a.w);
        float s[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) s[q] = 0.f;
        if (clean) {
#pragma unroll
          for (int i = 0; i < NQ; i += 8) {
            const float4 c4a = *reinterpret_cast<const float4*>(crq + i);
            const float4 c4b = *reinterpret_cast<const float4*>(crq + i + 4);
            s[0] += ex2(fmaf(v[i + 0], a.sl2, -c4a.x));
            s[1] += ex2(fmaf(v[i + 1], a.sl2, -c4a.y));
            s[2] += ex2(fmaf(v[i + 2], a.sl2, -c4a.z));
            s[3] += ex2(fmaf(v[i + 3], a.sl2, -c4a.w));
            s[4] += ex2(fmaf(v[i + 4], a.sl2, -c4b.x));
            s[5] += ex2(fmaf(v[i + 5], a.sl2, -c4b.y));
            s[6] += ex2(fmaf(v[i + 6], a.sl2, -c4b.z));
            s[7] += ex2(fmaf(v[i + 7], a.sl2, -c4b.w));
          }
        } else if (j < kend) {
#pragma unroll
          for (int i = 0; i < NQ; ++i)
            if (j <= limq[i]) s[i & 7] += ex2(fmaf(v[i], a.sl2, -crq[i]));
        }
        acc = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
      } else {
        dead = true;
      }
      ksum[(buf * 4 + cq) * 128 + kr] = acc;
      named_sync_epilogue();
      if (cq == 0 && !dead && j < kend) {
        const float* kb = ksum + buf * 4 * 128 + kr;
        out[j] = ((acc + kb[128]) + (kb[256] + kb[384])) * a.out_mul;
      }
    }
  }
  teardown<D>(c);
}

// ----------------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_k_map(const ScoresArgs& a, int D, CUtensorMap* tmK) {
  auto enc = encode_fn();
  if (!enc) return false;
  if (a.ss <= 0 || (a.KVH > 1 && a.sh <= 0) || (a.B > 1 && a.sb <= 0)) return false;
  const cuuint64_t kdims[4] = {(cuuint64_t)D, (cuuint64_t)a.S, (cuuint64_t)a.KVH, (cuuint64_t)a.B};
  const cuuint64_t kstr[3] = {(cuuint64_t)a.ss * 2, (cuuint64_t)(a.KVH > 1 ? a.sh : a.S * a.ss) * 2,
                              (cuuint64_t)(a.B > 1 ? a.sb : (int64_t)a.KVH * (a.KVH > 1 ? a.sh : a.S * a.ss)) * 2};
  const cuuint32_t kbox[4] = {64, (cuuint32_t)TILE, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.K), kdims, kstr, kbox, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_q_map(const ScoresArgs& a, int D, int qrows, CUtensorMap* tmQ) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t qdims[2] = {(cuuint64_t)D, (cuuint64_t)a.B * a.H * a.w};
  const cuuint64_t qstr[1] = {(cuuint64_t)D * 2};
  const cuuint32_t qbox[2] = {64, (cuuint32_t)qrows};
  const cuuint32_t es[2] = {1, 1};
  return enc(tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.q), qdims, qstr, qbox, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The three tensor maps of one call (K; the query group for pass 1 and for pass 2).  Encoding
// costs host microseconds per map, so the last few sets are kept per host thread, keyed on
// the addresses, shapes and strides they describe.
struct TcMaps {
  CUtensorMap k, q1, q2;
};
struct MapKey {
  const void* K;
  const void* q;
  int64_t S, ss, sh, sb;
  int B, H, KVH, w, D, Rpad;
  bool operator==(const MapKey& o) const {
    return K == o.K && q == o.q && S == o.S && ss == o.ss && sh == o.sh && sb == o.sb && B == o.B && H == o.H &&
           KVH == o.KVH && w == o.w && D == o.D && Rpad == o.Rpad;
  }
};

const TcMaps* tc_maps(const ScoresArgs& a, int D) {
  struct Entry {
    TcMaps maps;
    MapKey key;
    bool valid = false, ok = false;
  };
  thread_local Entry cache[8];
  thread_local int next = 0;
  const MapKey key{a.K, a.q, a.S, a.ss, a.sh, a.sb, a.B, a.H, a.KVH, a.w, D, a.Rpad};
  for (Entry& e : cache)
    if (e.valid && e.key == key) return e.ok ? &e.maps : nullptr;
  Entry& e = cache[next];
  next = (next + 1) % 8;
  e.key = key;
  e.valid = true;
  e.ok = make_k_map(a, D, &e.maps.k) && make_q_map(a, D, a.Rpad > 128 ? 256 : 128, &e.maps.q1) &&
         make_q_map(a, D, a.Rpad, &e.maps.q2);
  return e.ok ? &e.maps : nullptr;
}

template <typename Kern>
cudaError_t set_smem_once(Kern k, size_t bytes, int slot) {
  static bool done[64][16] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev][slot]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev][slot] = true;
  return e;
}

template <int D, int NHALF>
cudaError_t run_pass1(const ScoresArgs& a, cudaStream_t st, int slot) {
  const TcMaps* m = tc_maps(a, D);
  if (!m) return cudaErrorInvalidValue;
  const size_t smem = Layout<D>::SMEM;
  cudaError_t e = set_smem_once(k_pass1_tc<D, NHALF>, smem, slot);
  if (e != cudaSuccess) return e;
  k_pass1_tc<D, NHALF><<<dim3(a.nsplit, a.KVH, a.B), THREADS, smem, st>>>(a, m->k, m->q1);
  return launched(1);
}

template <int D, int NQ>
cudaError_t run_pass2(const ScoresArgs& a, cudaStream_t st, int slot) {
  const TcMaps* m = tc_maps(a, D);
  if (!m) return cudaErrorInvalidValue;
  const size_t smem = Layout<D>::SMEM;
  cudaError_t e = set_smem_once(k_pass2_tc<D, NQ>, smem, slot);
  if (e != cudaSuccess) return e;
  k_pass2_tc<D, NQ><<<dim3(a.nsplit, a.KVH, a.B), THREADS, smem, st>>>(a, m->k, m->q2);
  return launched(1);
}

}  // namespace

bool tc_supported(const ScoresArgs& a, int D) {
  if (D != 64 && D != 128) return false;
  if (a.live != nullptr) return false;
  if (a.Rpad != 64 && a.Rpad != 128 && a.Rpad != 192 && a.Rpad != 256) return false;
  if (a.R <= 32 || a.S < TILE) return false;
  if ((int64_t)a.B * a.H * a.w < (a.Rpad > 128 ? 256 : 128)) return false;
  if (a.nsplit > 65535 || a.KVH > 65535 || a.B > 65535) return false;
  return tc_maps(a, D) != nullptr;
}

cudaError_t launch_pass1_tc(const ScoresArgs& a, int D, cudaStream_t st) {
  const bool two = a.Rpad > 128;
  if (D == 64) return two ? run_pass1<64, 2>(a, st, 0) : run_pass1<64, 1>(a, st, 1);
  return two ? run_pass1<128, 2>(a, st, 2) : run_pass1<128, 1>(a, st, 3);
}

cudaError_t launch_pass2_tc(const ScoresArgs& a, int D, cudaStream_t st) {
  const int nq = a.Rpad / 4;
  if (D == 64) {
    switch (nq) {
      case 16: return run_pass2<64, 16>(a, st, 4);
      case 32: return run_pass2<64, 32>(a, st, 5);
      case 48: return run_pass2<64, 48>(a, st, 6);
      default: return run_pass2<64, 64>(a, st, 7);
    }
  }
  switch (nq) {
    case 16: return run_pass2<128, 16>(a, st, 8);
    case 32: return run_pass2<128, 32>(a, st, 9);
    case 48: return run_pass2<128, 48>(a, st, 10);
    default: return run_pass2<128, 64>(a, st, 11);
  }
}

}  // namespace kvc
