// Window scores on the 5th-generation tensor cores: the same two-pass computation as the
// mma.sync path in kvc_scores.cu ("Add TOVA press": only the last w attention rows; cold-
// compress PR 11: mean over each KV head's grouped queries), rebuilt around tcgen05.
//
// One CTA per (b, kvh, key range), 18 warps:
//   warp 16 producer: TMA loads of the query group (once) and of 256-key K stages into a
//           2-stage (D = 128) or 4-stage (D = 64) shared-memory ring (128-byte swizzle),
//           mbarrier-tracked;
//   warp 17 MMA issuer: allocates all 512 TMEM columns (two 256-column accumulators) and
//           issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) from one thread; commits
//           free the K stage and publish the accumulator;
//   warps 0-15 epilogue: tcgen05.ld the accumulator, release it, then do the softmax math.
// pass 1: A = query rows (M = 128 per half), B = K stage (N = 256 keys): each epilogue thread
//         owns one query row, so its running max / sum over keys is thread-local.
// pass 2: A = K tile (M = 128 keys), B = the query group (N = Rpad rows): each thread owns
//         one key and sums exp2(s*log2e - c_r) over its quarter of the query rows; the three
//         other quarters reach the key's owner warp through shared memory and an mbarrier.
// The passes run as two launches, or fused in one cooperative launch: every CTA is resident,
// a CTA publishes its pass-1 partials and waits for the other key ranges of its (b, kvh),
// while its MMA warp streams the same key range again for pass 2 without a pause.
// Every wait is bounded (%globaltimer); on timeout the kernel records KVC_ERR_TIMEOUT, all
// roles leave their loops, and TMEM is released before exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int TILE = 128;           // keys per accumulator unit of pass 2 (its MMA M)
constexpr int KT = 256;             // keys per K stage: pass 1's MMA N, two pass-2 units
// K bytes over all CTAs that pass 1 marks to stay in L2 for pass 2 (of the 126 MB L2; the
// rest holds what is streamed through once, the partials and the scores)
constexpr int64_t L2_KEEP_BYTES = 80ll << 20;
// the range's K stage that pass 2 reads i-th: the stages in reverse order, so that it starts
// with those pass 1 read last
__device__ __forceinline__ int pass2_stage(int ntiles, int i) { return ntiles - 1 - i; }
constexpr int MAX_STAGES = 4;       // K ring depth: 2 stages of 64 KiB (D = 128), 4 of 32 KiB (D = 64)
template <int D>
__host__ __device__ constexpr int ring_stages() { return D == 128 ? 2 : 4; }
constexpr int EPI_WARPS = 16;       // 4 per SM sub-partition
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int THREADS = 576;
constexpr int QROWS_MAX = 256;
constexpr uint32_t TMEM_COLS = 512;
// Every wait is bounded by ScoresArgs::wait_ns (2 s; 1 ms under kvc_debug_inject_timeout).
constexpr int KSLOTS = 4;           // pass-2 key-sum exchange slots per group and quadrant
// K ring full/empty, two accumulator full/empty pairs, query group, key-sum slots per quadrant
constexpr int NBARS = 2 * MAX_STAGES + 5 + 2 * 4 * KSLOTS;

__host__ __device__ constexpr uint32_t qpanel_bytes() { return QROWS_MAX * 128; }
__host__ __device__ constexpr uint32_t kpanel_bytes() { return KT * 128; }

// shared-memory layout behind a 1024-byte aligned base
template <int D>
struct Layout {
  static constexpr int NP = D / 64;  // 64-element (128-byte) panels along head_dim
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + NP * qpanel_bytes();
  static constexpr int ST = ring_stages<D>();
  static constexpr uint32_t STAGE = NP * kpanel_bytes();
  static constexpr uint32_t BARS = K + ST * STAGE;          // NBARS mbarriers
  static constexpr uint32_t MISC = (BARS + 8 * NBARS + 15) / 16 * 16;  // tmem base, abort flag
  static constexpr uint32_t CR = MISC + 16;                 // float[256], 16-byte aligned (float4 reads)
  static constexpr uint32_t LIM = CR + 256 * 4;             // int[256]
  static constexpr uint32_t STAT = LIM + 256 * 4;           // float2[4][256]
  static constexpr uint32_t KSUM = STAT + 4 * 256 * 8;      // float[2][KSLOTS][128]
  static constexpr uint32_t END = KSUM + 2 * KSLOTS * 128 * 4;
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
// non-blocking test of the phase with the given parity
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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
// Bounded wait (limit ns) for the phase with the given parity.  false: timed out (the abort
// flag is raised and KVC_ERR_TIMEOUT recorded) or another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > limit) {
      *abort_flag = 1;
      set_device_status(KVC_ERR_TIMEOUT);
      return false;
    }
  }
}
// same, ignoring the abort flag (used only to drain copies already in flight at teardown)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = gtimer();
  while (!mbar_try_wait(bar, parity)) {
    if (gtimer() - t0 > limit) return;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
          "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// one K box with an L2 eviction policy (createpolicy below)
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
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
  uint64_t wait_ns;  // bound on any single wait
  __device__ uint32_t full(int s) const { return sbase + BARS_OFF + 8 * s; }
  __device__ uint32_t empty(int s) const { return sbase + BARS_OFF + 8 * (MAX_STAGES + s); }
  __device__ uint32_t tfull(int b) const { return sbase + BARS_OFF + 8 * (2 * MAX_STAGES + b); }
  __device__ uint32_t tempty(int b) const { return sbase + BARS_OFF + 8 * (2 * MAX_STAGES + 2 + b); }
  __device__ uint32_t qfull() const { return sbase + BARS_OFF + 8 * (2 * MAX_STAGES + 4); }
  __device__ uint32_t kready(int g, int qd, int slot) const {
    return sbase + BARS_OFF + 8 * (2 * MAX_STAGES + 5 + (g * 4 + qd) * KSLOTS + slot);
  }
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
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(c.full(s), 1);
      mbar_init(c.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.tfull(b), 1);
      mbar_init(c.tempty(b), EPI_WARPS / 2);
    }
    mbar_init(c.qfull(), 1);
    for (int g = 0; g < 2; ++g)
      for (int q = 0; q < 4; ++q)
        for (int k = 0; k < KSLOTS; ++k) mbar_init(c.kready(g, q, k), 32);
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

// producer: query group once, then the K ring: `total` stages of KT keys, the key range's
// `ntiles` stages once per pass
template <int D>
__device__ __forceinline__ void producer(const Ctx& c, const ScoresArgs& a, const CUtensorMap* tmK,
                                         const CUtensorMap* tmQ, int qrows, int kvh, int b, int64_t kbeg,
                                         int ntiles, int nt1, int total) {
  using L = Layout<D>;
  const int qrow0 = (b * a.H + kvh * a.G) * a.w;
  mbar_expect_tx(c.qfull(), (uint32_t)(L::NP * qrows * 128));
  for (int p = 0; p < L::NP; ++p) tma_load_2d(c.sbase + L::Q + p * qpanel_bytes(), tmQ, p * 64, qrow0, c.qfull());
  // Pass 1 reads the range's stages in order, pass 2 in reverse (pass2_stage).  The last
  // `keep` stages of pass 1, the first that pass 2 reads, are loaded with the L2 evict-last
  // policy, all other loads with evict-first: where K is larger than L2, the part of it that
  // L2 can hold is still there when pass 2 starts instead of the part read longest ago.
  const int64_t ctas = (int64_t)gridDim.x * gridDim.y * gridDim.z;
  const int64_t fit = L2_KEEP_BYTES / (ctas * (int64_t)L::STAGE);
  const int keep = fit < ntiles ? (int)fit : ntiles;
  const uint64_t pol_keep = l2_evict_last(), pol_once = l2_evict_first();
  int issued = 0;
  for (int it = 0; it < total; ++it) {
    const int s = it % L::ST;
    const uint32_t ph = (uint32_t)(it / L::ST) & 1u;
    if (!wait_bar(c.empty(s), ph ^ 1u, c.abort_flag, c.wait_ns)) break;
    mbar_expect_tx(c.full(s), L::STAGE);
    const bool p2 = it >= nt1;
    const int t = p2 ? pass2_stage(ntiles, it - nt1) : it;
    const int y = (int)(kbeg + (int64_t)t * KT);
    const uint64_t pol = !p2 && t >= ntiles - keep ? pol_keep : pol_once;
    for (int p = 0; p < L::NP; ++p)
      tma_load_4d(c.sbase + L::K + s * L::STAGE + p * kpanel_bytes(), tmK, p * 64, y, kvh, b, c.full(s), pol);
    issued = it + 1;
  }
  // copies still in flight when the kernel stops early are waited for (bounded) before exit
  if (*c.abort_flag) {
    drain_bar(c.qfull(), 0, c.wait_ns);
    for (int it = (issued > L::ST ? issued - L::ST : 0); it < issued; ++it)
      drain_bar(c.full(it % L::ST), (uint32_t)(it / L::ST) & 1u, c.wait_ns);
  }
}

// ----------------------------------------------------------------------------------------
// softmax helpers
// ----------------------------------------------------------------------------------------
// Packed pairs of fp32 (fma.rn.f32x2 / add.rn.f32x2 issue once for two lanes of work).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t ex2x2(uint64_t y) {
  float lo, hi;
  upk2(y, lo, hi);
  return pk2(ex2(lo), ex2(hi));
}
__device__ __forceinline__ float hsum4(const uint64_t* acc) {
  float lo, hi;
  upk2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), lo, hi);
  return lo + hi;
}
// sum_i exp2(v_i * sl2 - off) over NC values (NC a multiple of 8), four packed accumulators
template <int NC>
__device__ __forceinline__ float sum_exp2x(const float* v, float sl2, float off) {
  const uint64_t SL = pk2(sl2, sl2), OF = pk2(-off, -off);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < NC; i += 8) {
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = add2(acc[q], ex2x2(fma2(pk2(v[i + 2 * q], v[i + 2 * q + 1]), SL, OF)));
  }
  return hsum4(acc);
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// max of 32 values with three-input max: 16 instructions, depth 4
__device__ __forceinline__ float max32(const float* v) {
  float a[12];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = v[30];
  a[11] = v[31];
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]), b2 = max3f(a[6], a[7], a[8]),
              b3 = max3f(a[9], a[10], a[11]);
  return fmaxf(max3f(b0, b1, b2), b3);
}
// sum_i exp2(v_i * sl2 + nc_i) over NC values with per-column offsets nc (16-byte aligned)
template <int NC>
__device__ __forceinline__ float sum_exp2x_cols(const float* v, float sl2, const float* nc) {
  const uint64_t SL = pk2(sl2, sl2);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < NC; i += 8) {
    const float4 ca = *reinterpret_cast<const float4*>(nc + i);
    const float4 cb = *reinterpret_cast<const float4*>(nc + i + 4);
    acc[0] = add2(acc[0], ex2x2(fma2(pk2(v[i + 0], v[i + 1]), SL, pk2(ca.x, ca.y))));
    acc[1] = add2(acc[1], ex2x2(fma2(pk2(v[i + 2], v[i + 3]), SL, pk2(ca.z, ca.w))));
    acc[2] = add2(acc[2], ex2x2(fma2(pk2(v[i + 4], v[i + 5]), SL, pk2(cb.x, cb.y))));
    acc[3] = add2(acc[3], ex2x2(fma2(pk2(v[i + 6], v[i + 7]), SL, pk2(cb.z, cb.w))));
  }
  return hsum4(acc);
}

// ----------------------------------------------------------------------------------------
// key-range barrier of the fused launch
// ----------------------------------------------------------------------------------------
// Workspace words: sync[0] holds an epoch E that advances by one per launch; CTA (b, kvh,
// split) sets sync[1 + (b*KVH + kvh)*nsplit + split] to tag(E + 1) once its pass-1 partials
// are stored.  tag() is the splitmix64 output mix (Steele, Lea & Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014): leftover words from any earlier use of the
// memory equal the current tag only by a 2^-64 chance, so the words need no initialisation.
__device__ __forceinline__ uint64_t epoch_tag(uint64_t e) {
  uint64_t z = e + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;\n" ::: "memory"); }
// One warp waits (bounded) until words [0, n) of `w` all equal `tag`.  With a non-null
// abort flag the wait also ends when another role of the CTA has given up.
__device__ __forceinline__ bool warp_wait_tags(const unsigned long long* w, int64_t n, uint64_t tag,
                                               volatile int* abort_flag, uint64_t limit) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  const uint64_t t0 = gtimer();
  for (int64_t i = lane; i < n && ok; i += 32) {
    while (ld_relaxed_u64(w + i) != tag) {
      if (abort_flag != nullptr && *abort_flag) {
        ok = false;
        break;
      }
      if (gtimer() - t0 > limit) {
        if (abort_flag != nullptr) *abort_flag = 1;
        set_device_status(KVC_ERR_TIMEOUT);
        ok = false;
        break;
      }
      __nanosleep(32);
    }
  }
  fence_acq_rel_gpu();  // what the tag writers stored before their release is now visible
  return __all_sync(0xffffffffu, ok);
}

// (M, L) <- the log2-domain sum of (M, L) and (m2, l2); an empty side has L = 0
__device__ __forceinline__ void lse2_merge(float& M, float& L, float m2, float l2) {
  if (!(l2 > 0.f)) return;
  if (!(L > 0.f)) {
    M = m2;
    L = l2;
  } else if (m2 > M) {
    L = L * ex2(M - m2) + l2;
    M = m2;
  } else {
    L += l2 * ex2(m2 - M);
  }
}
// Pass-2 prologue: nc[r] = -log2(sum over the nsplit key ranges of 2^lse) for row r (-inf
// when the row sees no key) and the row's causal limit, for r < N2.  A thread takes four
// adjacent rows (one 16-byte load per key range: a range's rows are contiguous, so a warp's
// loads are whole sectors) and every TPR-th range, all its loads in flight at once (up to 8);
// the TPR threads of a row quad then combine with shuffles.  Every CTA of a (b, kvh) reads
// the same partials at the same moment, so the bytes per partial matter: one float each.
template <int N2>
__device__ __forceinline__ void merge_rows(const ScoresArgs& a, int bk, float* nc, int* lim) {
  constexpr int NQD = N2 / 4;  // row quads
  constexpr int TPR = NQD >= 64 ? 8 : (NQD >= 48 ? 8 : (NQD >= 32 ? 16 : 32));
  constexpr int BATCH = 8;
  static_assert(NQD * TPR <= EPI_WARPS * 32, "row quads x threads per quad fit the epilogue");
  const int rq = threadIdx.x / TPR, sub = threadIdx.x % TPR;
  float M[4], L[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    M[i] = -CUDART_INF_F;
    L[i] = 0.f;
  }
  if (rq < NQD) {
    for (int s0 = sub; s0 < a.nsplit; s0 += BATCH * TPR) {
      float4 o[BATCH];
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        const int sidx = s0 + q * TPR;
        o[q] = sidx < a.nsplit ? __ldcg(reinterpret_cast<const float4*>(a.part + part_index(a, bk, 4 * rq, sidx)))
                               : make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
      }
      float mx[4] = {M[0], M[1], M[2], M[3]};
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        mx[0] = fmaxf(mx[0], o[q].x);
        mx[1] = fmaxf(mx[1], o[q].y);
        mx[2] = fmaxf(mx[2], o[q].z);
        mx[3] = fmaxf(mx[3], o[q].w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (mx[i] == -CUDART_INF_F) continue;
        float sum = L[i] > 0.f ? L[i] * ex2(M[i] - mx[i]) : 0.f;
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          const float v = i == 0 ? o[q].x : (i == 1 ? o[q].y : (i == 2 ? o[q].z : o[q].w));
          sum += ex2(v - mx[i]);  // 2^-inf = 0 for a range without keys
        }
        M[i] = mx[i];
        L[i] = sum;
      }
    }
  }
#pragma unroll
  for (int off = 1; off < TPR; off <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      lse2_merge(M[i], L[i], __shfl_xor_sync(0xffffffffu, M[i], off), __shfl_xor_sync(0xffffffffu, L[i], off));
  if (rq < NQD && sub < 4) {
    const int r = 4 * rq + sub;
    const float Mr = sub == 0 ? M[0] : (sub == 1 ? M[1] : (sub == 2 ? M[2] : M[3]));
    const float Lr = sub == 0 ? L[0] : (sub == 1 ? L[1] : (sub == 2 ? L[2] : L[3]));
    nc[r] = Lr > 0.f ? -(Mr + log2f(Lr)) * a.pw : -CUDART_INF_F;
    lim[r] = row_limit_i(a, r);
  }
}

// Pass-2 chunk: W query-row columns of this thread's key from TMEM (the accumulator is
// released after the call's last chunk is loaded), masked columns set to -inf, then
// sum exp2(s*log2e - c_r) with nc = -c_r.
template <int W>
__device__ __forceinline__ float pass2_chunk(const Ctx& c, int buf, uint32_t taddr, bool release, const float* nc,
                                             const int* lim, float sl2, bool clean, int64_t j, int64_t kend) {
  float v[W];
  tmem_load_cols<W>(taddr, v);
  if (release) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(c.tempty(buf));
  }
  if (!clean) {
    // limits are loaded unconditionally and applied with selects (a short-circuit test
    // around the load would make every column a divergent branch)
    const bool in = j < kend;
#pragma unroll
    for (int i = 0; i < W; i += 4) {
      const int4 l4 = *reinterpret_cast<const int4*>(lim + i);
      v[i + 0] = (in & (j <= l4.x)) ? v[i + 0] : -CUDART_INF_F;
      v[i + 1] = (in & (j <= l4.y)) ? v[i + 1] : -CUDART_INF_F;
      v[i + 2] = (in & (j <= l4.z)) ? v[i + 2] : -CUDART_INF_F;
      v[i + 3] = (in & (j <= l4.w)) ? v[i + 3] : -CUDART_INF_F;
    }
  }
  return sum_exp2x_cols<W>(v, sl2, nc);
}

// ----------------------------------------------------------------------------------------
// the scoring kernel
// ----------------------------------------------------------------------------------------
// MODE 1: pass 1 only (key-range partials (m, l) of every query row to a.part);
// MODE 2: pass 2 only (c_r merged from a.part, column sums to a.out);
// MODE 3: both, one cooperative launch, with the key-range barrier between them.
// The epilogue runs as two groups that alternate tiles: warps 0-7 take the tiles landing in
// accumulator 0, warps 8-15 those in accumulator 1, so one group computes while the other
// waits for its next tile.  A warp w only reads TMEM lanes of quadrant w%4.
// Pass 1: warp (g, w8) reads, for the query rows of quadrant w8%4 in half h, NC1 key columns
// of its group's tiles; a row's (max, sum) is then merged over its NPART1 warps.
// Pass 2: warp (g, w8) reads, for the 32 keys of quadrant w8%4, the query-row columns
// [hf*NW, hf*NW + NW) with hf = w8/4; the hf = 1 warp hands its key sums to the hf = 0 warp
// through a shared-memory slot and an mbarrier, and that warp adds them and stores.
template <int D, int NHALF, int NQ, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    k_scores_tc(const ScoresArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ) {
  using L = Layout<D>;
  constexpr int KS = D / 16;
  constexpr bool P1 = (MODE & 1) != 0, P2 = (MODE & 2) != 0;
  constexpr int N2 = 4 * NQ;                     // pass-2 MMA N: padded query rows
  constexpr int QROWS = P1 ? NHALF * 128 : N2;   // query rows staged in shared memory
  constexpr int NPART1 = NHALF == 2 ? 2 : 4;     // pass 1: warps sharing one query row
  constexpr int NC1 = KT / 2;                    // pass 1: key columns per warp and unit
  constexpr int UPT1 = NHALF;                    // pass-1 units per K stage (one per query half)
  constexpr int NW = N2 / 2;                     // pass 2: query-row columns per warp and tile
  extern __shared__ unsigned char smem_raw[];
  // both tensor maps' descriptors fetched during the prologue and the wait for the previous
  // kernel (they are launch parameters, not outputs of that kernel)
  if (threadIdx.x == PRODUCER_WARP * 32) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
  }
  Ctx cx = prologue<D>(smem_raw);  // shared memory and TMEM only
  cx.wait_ns = a.wait_ns;
  const Ctx& c = cx;
  pdl_wait();  // previous kernel on the stream complete and visible
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int bk = b * a.KVH + kvh;
  int64_t kbeg, kend;
  key_range(a, split, &kbeg, &kend);
  // Work comes in units, one accumulator (256 TMEM columns) each, alternating between the two
  // buffers and the two epilogue groups: pass 1 has UPT1 units per K stage (query half h, all
  // KT keys), pass 2 two (the stage's 128-key halves on M).
  const int ntiles = (int)((kend - kbeg + KT - 1) / KT);
  const int n1 = P1 ? ntiles * UPT1 : 0;
  const int total = n1 + (P2 ? 2 * ntiles : 0);
  const int nt1 = P1 ? ntiles : 0;  // K stages of pass 1
  auto unit_stage = [&](int u) -> int { return u < n1 ? u / UPT1 : nt1 + ((u - n1) >> 1); };
  auto first_of_stage = [&](int u) -> bool { return u < n1 ? (u % UPT1) == 0 : ((u - n1) & 1) == 0; };
  auto last_of_stage = [&](int u) -> bool { return u < n1 ? (u % UPT1) == UPT1 - 1 : ((u - n1) & 1) == 1; };

  if (warp == PRODUCER_WARP) {
    if (lane == 0) producer<D>(c, a, &tmK, &tmQ, QROWS, kvh, b, kbeg, ntiles, nt1, nt1 + (P2 ? ntiles : 0));
  } else if (warp == MMA_WARP) {
    if (lane == 0 && wait_bar(c.qfull(), 0, c.abort_flag, c.wait_ns)) {
      int done = 0;
      // Unit it+1's barriers are tested (without blocking) halfway through unit it's MMAs;
      // only if they were not yet complete does the thread wait after the commits.  Either
      // way no MMA of unit it waits on the epilogue.
      auto ready = [&](int t) -> bool {
        const int st = unit_stage(t);
        return wait_bar(c.tempty(t & 1), ((uint32_t)(t >> 1) & 1u) ^ 1u, c.abort_flag, c.wait_ns) &&
               (!first_of_stage(t) ||
                wait_bar(c.full(st % L::ST), (uint32_t)(st / L::ST) & 1u, c.abort_flag, c.wait_ns));
      };
      auto ready_now = [&](int t) -> bool {
        const int st = unit_stage(t);
        return mbar_test(c.tempty(t & 1), ((uint32_t)(t >> 1) & 1u) ^ 1u) &&
               (!first_of_stage(t) || mbar_test(c.full(st % L::ST), (uint32_t)(st / L::ST) & 1u));
      };
      // descriptor start addresses advance in 16-byte units (no carry: shared memory < 256 KB)
      const uint64_t qdesc = sw128_desc(c.sbase + L::Q), kdesc0 = sw128_desc(c.sbase + L::K);
      bool ok = total > 0 && ready(0);
      bool next_ready = false;
      for (int it = 0; ok && it < total; ++it) {
        const int s = unit_stage(it) % L::ST, buf = it & 1;
        tc_fence_after();
        const uint64_t kdesc = kdesc0 + (uint64_t)((s * L::STAGE) >> 4);
        const uint32_t d = c.tmem + buf * 256;
        if (it < n1) {
          // query half h (M = 128 rows) against all KT keys of the stage (N = 256)
          constexpr uint32_t idesc = idesc_bf16(128, KT);
          const int h = NHALF == 2 ? (it & 1) : 0;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            if (ks == KS / 2) next_ready = it + 1 < total && ready_now(it + 1);
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t ad = qdesc + (uint64_t)(((ks >> 2) * qpanel_bytes() + h * 128 * 128 + koff) >> 4);
            const uint64_t bd = kdesc + (uint64_t)(((ks >> 2) * kpanel_bytes() + koff) >> 4);
            tc_mma(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
        } else {
          // the stage's 128-key half kh on M against the query group (N = N2)
          constexpr uint32_t idesc = idesc_bf16(128, N2);
          const int kh = (it - n1) & 1;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            if (ks == KS / 2) next_ready = it + 1 < total && ready_now(it + 1);
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t ad = kdesc + (uint64_t)(((ks >> 2) * kpanel_bytes() + kh * TILE * 128 + koff) >> 4);
            const uint64_t bd = qdesc + (uint64_t)(((ks >> 2) * qpanel_bytes() + koff) >> 4);
            tc_mma(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
        }
        if (last_of_stage(it)) tc_commit(c.empty(s));
        tc_commit(c.tfull(buf));
        done = it + 1;
        if (it + 1 < total && !next_ready) ok = ready(it + 1);
      }
      // stopped early: let the MMAs already issued finish before TMEM is released
      if (*c.abort_flag && done > 0)
        drain_bar(c.tfull((done - 1) & 1), (uint32_t)((done - 1) >> 1) & 1u, c.wait_ns);
    }
    __syncwarp();
  } else {
    const int qd = warp & 3;
    const int g = warp >> 3, w8 = warp & 7;  // tile group (= accumulator buffer), warp in group
    uint64_t epoch = 0;
    if constexpr (MODE == 3) {
      if (warp == 0) epoch = ld_relaxed_u64(a.sync);
    }
    if constexpr (P1) {
      // one query row per thread; the group's units (query half g when NHALF == 2), each
      // warp taking one half of the KT key columns, read in 32-column chunks
      const int h = NHALF == 2 ? g : 0;
      const int part = NHALF == 2 ? (w8 >> 2) : g * 2 + (w8 >> 2);
      const int c0 = (w8 >> 2) * NC1;
      const int r = h * 128 + qd * 32 + lane;
      const int lim = row_limit_i(a, r);
      // (m, l): l = sum exp2(s*log2e - m), m the running max, updated every 32-column chunk
      // (three-input max tree, one rescale of l).  No chunk waits on the previous chunk's
      // sum, so the next chunk's TMEM load and max overlap this chunk's exponentials.
      float m = -CUDART_INF_F, l = 0.f;
      float v[32];
      for (int it = g; it < n1; it += 2) {
        const uint32_t bph = (uint32_t)(it >> 1) & 1u;
        if (!wait_bar(c.tfull(g), bph, c.abort_flag, c.wait_ns)) break;
        tc_fence_after();
        const uint32_t taddr = c.tmem + ((uint32_t)(qd * 32) << 16) + g * 256 + c0;
        // last visible column of the unit for this row (rows without keys: lim < 0, none)
        const int64_t jlast =
            (kend - 1 < (int64_t)lim ? kend - 1 : (int64_t)lim) - (kbeg + (int64_t)(it / UPT1) * KT + c0);
#pragma unroll
        for (int ch = 0; ch < NC1 / 32; ++ch) {
          tmem_ld32(taddr + ch * 32, v);
          if (ch == NC1 / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(c.tempty(g));
          }
          const int64_t jmax = jlast - ch * 32;
          if (jmax < 31) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (i <= jmax) ? v[i] : -CUDART_INF_F;
          }
          const float mn = fmaxf(m, max32(v) * a.sl2);
          const float mref = mn == -CUDART_INF_F ? 0.f : mn;  // all masked so far: sums stay 0
          l = l * ex2(m - mref) + sum_exp2x<32>(v, a.sl2, mref);
          m = mn;
        }
      }
      // merge the NPART1 partial (m, l) of each row
      float2* stat = reinterpret_cast<float2*>(c.base + L::STAT);
      stat[part * 256 + r] = make_float2(m, l);
      named_sync_epilogue();
      if (part == 0) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int q = 0; q < NPART1; ++q) {
          const float2 o = stat[q * 256 + r];
          if (o.y > 0.f) M = fmaxf(M, o.x);
        }
        float Lsum = 0.f;
#pragma unroll
        for (int q = 0; q < NPART1; ++q) {
          const float2 o = stat[q * 256 + r];
          if (o.y > 0.f) Lsum += o.y * ex2(o.x - M);
        }
        if (r < a.Rpad) a.part[part_index(a, bk, r, split)] = range_lse(M, Lsum);
      }
    }
    if constexpr (MODE == 3) {
      // publish this key range's partials, then wait for the other ranges of (b, kvh)
      named_sync_epilogue();
      if (warp == 0) {
        unsigned long long* tags = a.sync + 1 + (int64_t)bk * a.nsplit;
        const uint64_t tag = epoch_tag(epoch + 1);
        // (a.withhold: a test of the timeout path names one CTA whose arrival is left out)
        if (lane == 0 && (int64_t)bk * a.nsplit + split != a.withhold) {
          fence_acq_rel_gpu();  // release: the CTA's partials (ordered by the barrier above)
          st_relaxed_u64(tags + split, tag);
        }
        __syncwarp();
        warp_wait_tags(tags, a.nsplit, tag, c.abort_flag, c.wait_ns);
      }
      named_sync_epilogue();
      pdl_trigger();  // the next kernel may begin launching; it waits for this grid's end
    }
    if constexpr (P2) {
      float* ncr = reinterpret_cast<float*>(c.base + L::CR);
      int* limr = reinterpret_cast<int*>(c.base + L::LIM);
      merge_rows<N2>(a, bk, ncr, limr);
      named_sync_epilogue();
      const int hf = w8 >> 2;
      const int kr = qd * 32 + lane;
      const float* ncq = ncr + hf * NW;
      const int* limq = limr + hf * NW;
      float* out = a.out + (int64_t)bk * a.S;
      bool dead = false;
      const int first = n1 + ((g - n1) & 1);  // this group's first pass-2 tile
      for (int it = first; it < total; it += 2) {
        const int u = (it - first) >> 1;       // this group's pass-2 tile count
        const int64_t kt0 = kbeg + (int64_t)pass2_stage(ntiles, (it - n1) >> 1) * KT + ((it - n1) & 1) * TILE;
        const int64_t j = kt0 + kr;
        float acc = 0.f;
        if (!dead && wait_bar(c.tfull(g), (uint32_t)(it >> 1) & 1u, c.abort_flag, c.wait_ns)) {
          tc_fence_after();
          const uint32_t taddr = c.tmem + ((uint32_t)(qd * 32) << 16) + g * 256 + hf * NW;
          const bool clean = (kt0 + TILE <= kend) && (!a.causal || kt0 + TILE - 1 <= a.S - a.w);
#pragma unroll
          for (int ch = 0; ch < NW / 32; ++ch)
            acc += pass2_chunk<32>(c, g, taddr + ch * 32, ch == NW / 32 - 1, ncq + ch * 32, limq + ch * 32,
                                   a.sl2 * a.pw, clean, j, kend);
        } else {
          dead = true;
        }
        // Slot u % KSLOTS is written again only KSLOTS group tiles later, after the reader has
        // released the accumulator of the group's tile u + KSLOTS - 1 (so has read tile u).
        const int slot = u % KSLOTS;
        const uint32_t kb = c.kready(g, qd, slot);
        float* ks = reinterpret_cast<float*>(c.base + L::KSUM) + (g * KSLOTS + slot) * 128 + kr;
        if (hf != 0) {
          *ks = acc;
          mbar_arrive(kb);
        } else if (wait_bar(kb, (uint32_t)(u / KSLOTS) & 1u, c.abort_flag, c.wait_ns) && !dead && j < kend) {
          out[j] = (acc + *ks) * a.out_mul;
        }
      }
    }
    if constexpr (MODE == 3) {
      // CTA 0 advances the epoch once every CTA has published (so has read the epoch)
      if (warp == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
        warp_wait_tags(a.sync + 1, (int64_t)a.B * a.KVH * a.nsplit, epoch_tag(epoch + 1), nullptr, c.wait_ns);
        if (lane == 0) st_relaxed_u64(a.sync, epoch + 1);
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
  const cuuint32_t kbox[4] = {64, (cuuint32_t)KT, 1, 1};
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

// Armed by kvc_debug_inject_timeout: the next fused launch waits at most 1 ms and leaves out
// the key-range arrival of its first CTA, so its other CTAs time out (a test of that path).
std::atomic<int> g_inject_timeout{0};

// one launch of the scoring kernel in the given mode; the fused mode is cooperative
template <int D, int NHALF, int NQ, int MODE>
cudaError_t run_tc(const ScoresArgs& a_in, cudaStream_t st) {
  ScoresArgs a = a_in;
  if (MODE == 3 && g_inject_timeout.exchange(0) != 0) {
    a.wait_ns = 1000000ull;
    a.withhold = 0;
  }
  const TcMaps* m = tc_maps(a, D);
  if (!m) return cudaErrorInvalidValue;
  auto kern = k_scores_tc<D, NHALF, NQ, MODE>;
  const size_t smem = Layout<D>::SMEM;
  cudaError_t e = func_attrs_once(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.nsplit, a.KVH, a.B);
  if constexpr (MODE != 3) {
    e = launch_pdl(kern, grid, dim3(THREADS), smem, st, a, m->k, MODE == 2 ? m->q2 : m->q1);
    if (e != cudaSuccess) return e;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // cooperative (every CTA resident: the key-range barrier) and programmatic stream
    // serialisation (the prologue overlaps the previous kernel's tail)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, a, m->k, m->q1);
    if (e != cudaSuccess) return e;
  }
  return launched(1);
}

// Whether every CTA of the fused launch can be resident at once (cached per device).
template <int D, int NHALF, int NQ>
bool fused_fits(const ScoresArgs& a) {
  static int occ_cache[64] = {0};  // 0: not yet known, -1: not usable
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (occ_cache[dev] == 0) {
    auto kern = k_scores_tc<D, NHALF, NQ, 3>;
    const size_t smem = Layout<D>::SMEM;
    int occ = 0, coop = 0;
    if (func_attrs_once(reinterpret_cast<const void*>(kern), (int)smem) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, smem) != cudaSuccess || !coop ||
        occ < 1) {
      cudaGetLastError();
      occ = -1;
    }
    occ_cache[dev] = occ;
  }
  return occ_cache[dev] > 0 && (int64_t)a.nsplit * a.KVH * a.B <= (int64_t)occ_cache[dev] * num_sms();
}

template <int D, int NHALF, int NQ>
cudaError_t run_scores(const ScoresArgs& a, cudaStream_t st) {
  if (a.sync != nullptr && fused_fits<D, NHALF, NQ>(a)) return run_tc<D, NHALF, NQ, 3>(a, st);
  // pass 1 does not depend on NQ, pass 2 not on NHALF
  const cudaError_t e = run_tc<D, NHALF, 16, 1>(a, st);
  if (e != cudaSuccess) return e;
  return run_tc<D, 1, NQ, 2>(a, st);
}

template <int D>
cudaError_t run_scores_d(const ScoresArgs& a, cudaStream_t st) {
  switch (a.Rpad) {
    case 64: return run_scores<D, 1, 16>(a, st);
    case 128: return run_scores<D, 1, 32>(a, st);
    case 192: return run_scores<D, 2, 48>(a, st);
    default: return run_scores<D, 2, 64>(a, st);
  }
}

}  // namespace

bool tc_supported(const ScoresArgs& a, int D) {
  if (D != 64 && D != 128) return false;
  if (a.live != nullptr) return false;
  if (a.Rpad != 64 && a.Rpad != 128 && a.Rpad != 192 && a.Rpad != 256) return false;
  if (a.R <= 32 || a.S < KT) return false;
  if ((int64_t)a.B * a.H * a.w < (a.Rpad > 128 ? 256 : 128)) return false;
  if (a.nsplit > 65535 || a.KVH > 65535 || a.B > 65535) return false;
  return tc_maps(a, D) != nullptr;
}

void inject_scores_timeout(int armed) { g_inject_timeout.store(armed ? 1 : 0); }

bool make_cache_tensor_map(const uint16_t* K, const kvc_kv_desc& kv, CUtensorMap* tm, int box_rows) {
  auto enc = encode_fn();
  if (!enc || box_rows < 1 || box_rows > 256) return false;
  if (kv.stride_s <= 0 || (kv.KVH > 1 && kv.stride_h <= 0) || (kv.B > 1 && kv.stride_b <= 0)) return false;
  const int64_t sh = kv.KVH > 1 ? kv.stride_h : kv.S * kv.stride_s;
  const int64_t sb = kv.B > 1 ? kv.stride_b : (int64_t)kv.KVH * sh;
  const cuuint64_t dims[4] = {(cuuint64_t)kv.D, (cuuint64_t)kv.S, (cuuint64_t)kv.KVH, (cuuint64_t)kv.B};
  const cuuint64_t str[3] = {(cuuint64_t)kv.stride_s * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(K), dims, str, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_scores_tc(const ScoresArgs& a, int D, cudaStream_t st) {
  return D == 64 ? run_scores_d<64>(a, st) : run_scores_d<128>(a, st);
}

KVC_TU_STATUS(scores_tc)

}  // namespace kvc
