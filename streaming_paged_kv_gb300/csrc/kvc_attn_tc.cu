// Tensor-core paged attention for sm_103a: TMA gathers of K/V page tiles
// through the page table, tcgen05 MMAs with TMEM accumulators, fp32 online
// softmax.
//
// What it computes ([KVC] "Kernel-Level Execution Flow": causal=False,
// pos_encoding_mode="NONE", as many KV heads as query heads):
//     O[t,h,:] = sum_j softmax_j(Q[t,h,:].K[j,h,:] * sm_scale) V[j,h,:]
// over the visible tokens j, which the plan lists as KV tiles of 128 rows
// (scale pages, live window, then the special pages; a page's rows beyond its
// valid count never enter the softmax, so exact page sizes such as 999 need no
// padding -- [PERF] "Page-Size Handling for FA2 vs FA3").  A tile holds rows of
// one page, or -- packed -- a page's last rows rounded up to a multiple of 8
// and the next page's first rows, gathered as boxes of 8 to 64 rows into the
// 1024-byte swizzle atoms of the stage, so that a 999-row page costs 7.8
// tiles, not 8.
//
// Pages cited by tag: [KVC] "How LingBot-Map Implements the KV Cache Mechanism
// for Streaming Inference with FlashInfer Integration"; [PERF] "How to Improve
// Streaming Inference Performance with FlashInfer KV Cache Backend".
//
// A launch serves up to kTcMaxBatch independent requests (streams); a CTA =
// two 128-row query tiles (Q0, Q1) of one request x one head x one KV split;
// each K/V tile is loaded once and serves both query tiles.  Warps:
//   0-3   softmax + epilogue of Q0, 4-7 softmax + epilogue of Q1: one thread
//         per query row (warp w owns TMEM lanes [32(w%4), +32)), holding the
//         row's 128 scores of a tile in registers
//   8     TMA producer (one lane): Q0/Q1, then K/V tiles into a 5-stage ring
//   9     P V issuer (one lane): O_i += P V with P read from TMEM
//   10    S issuer (one lane): S = Q_i K^T into TMEM
// Score tiles are numbered in issue order k = j * nq + i (KV tile j, query
// tile i) and rotate through three 128-column TMEM buffers, b = k mod 3.  A
// softmax thread reads its whole row of S(k), writes P(k) as 16-bit pairs over
// the first 64 columns of the same buffer, and the P V product reads it there.
// S(k+3) may enter buffer b once P(k) V has completed, so while one query
// tile's warps exponentiate, the other tile's next scores are already being
// computed.  TMEM (512 columns): buffers [0,128) [128,256) [256,384),
// O0 [384,448), O1 [448,512).  A CTA with a single query tile may run in dual
// mode (below): then both warp groups share Q0, taking alternate KV tiles.
// Q and K/V tiles use the 128-byte swizzle that both TMA and the tensor core
// understand.  Scores live in the log2 domain (scaled by sm_scale * log2 e).
// Each row keeps a reference m_ref, starting at 0, and takes P against it.
// The reference moves (to the tile's row max; O and the row sum are rescaled,
// O only after the previous P V product has completed) only when a tile's row
// sum would exceed 2^64 (or, on the first tile, fall below 2^-64): the
// relative precision of P, O and the sums does not depend on the reference,
// only their range does, so most tiles need no row max at all; that rare
// path is a separate, non-inlined function, which keeps its registers out of
// the softmax loop.
//
// K/V tiles are loaded with an L2 evict-first policy, so that the split-KV
// partials stay in L2 for the merge kernel.  The epilogue stages each query
// tile's normalised rows in shared memory (the tile's own Q area) and writes
// them with TMA stores: the bf16 / f16 output, or the fp32 partials (their
// log2-sum-exp goes out with plain stores).
//
// Every mbarrier wait is bounded: when a wait runs out, the thread records
// the fact in the status word, raises a CTA-wide abort flag, and every role
// skips its remaining work, drains its own in-flight copies / MMAs (again
// with a bound), frees TMEM and returns.  The flag, the status pointer and
// the budget live in shared memory, read only by the out-of-line slow path
// of a wait.

#include "kvc_internal.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <cstring>
#include <new>
#include <type_traits>

namespace kvc {

struct TcMaps {
  CUtensorMap cache;     // 3D view of the whole cache: {H*D, page_size, blocks*pages*2}, 128-row boxes
  CUtensorMap cache_u[4];  // the same view with boxes of 8, 16, 32 and 64 rows (packed tiles)
  int dtype;
  int num_heads;
  int head_dim;
};

namespace {

constexpr int BM = 128;           // query rows per query tile
constexpr int QT = 2;             // query tiles per CTA
constexpr int BN = 128;           // KV rows per tile
constexpr int HD = 64;            // head dim of this kernel
constexpr int STAGES = 5;         // K/V ring depth
constexpr int NBUF = 3;           // rotating S / P buffers in TMEM
constexpr int NUM_THREADS = 352;
// Register budget: the register file is split over the four SM sub-partitions
// and warp w runs on sub-partition w % 4, so with eleven warps three
// sub-partitions hold three warps each: 16384 / (3 * 32) = 170, rounded down
// to 168.
constexpr int REG_BOUND_THREADS = 384;
constexpr int PRODUCER_WARP = 8, PV_WARP = 9, S_WARP = 10;
constexpr int GROUP_THREADS = BM;                    // softmax threads per query tile
constexpr uint32_t TILE_BYTES = BN * HD * 2;         // 16 KB: one K or V tile
constexpr uint32_t Q_BYTES = BM * HD * 2;            // 16 KB per query tile
constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t buf_col(int b) { return b * BN; }
__host__ __device__ constexpr uint32_t o_col(int i) { return NBUF * BN + i * HD; }
static_assert(o_col(QT) <= TMEM_COLS, "TMEM budget");
constexpr long long kDrainBudget = 1LL << 26;        // cycles for draining after an abort

// Shared memory map (offsets from a 1024-aligned base).
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + QT * Q_BYTES;
constexpr uint32_t OFF_V = OFF_K + STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + STAGES * TILE_BYTES;
// Dual-mode hand-off from softmax group 1 to group 0: [128 rows][max, sum, flag].
constexpr uint32_t OFF_XCH = OFF_BAR + 256;
constexpr uint32_t OFF_STATE = OFF_XCH + BM * 3 * 4;            // CtaState
constexpr uint32_t SMEM_BYTES = OFF_STATE + 32 + 1024;  // + alignment slack

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// CTA state of the bounded waits, in shared memory: the abort flag, the status
// word of the CTA's request and the wait budget.  A wait passes only its
// barrier; the slow path (rare) reads the rest from here.
struct CtaState {
  int abort_flag;
  int pad;
  int32_t* status;
  long long budget;
};

__device__ __forceinline__ CtaState* cta_state() {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  return reinterpret_cast<CtaState*>(smem + OFF_STATE);
}

__device__ __noinline__ void raise_abort(int where) {
  CtaState* cs = cta_state();
  *reinterpret_cast<volatile int*>(&cs->abort_flag) = 1;
  if (atomicCAS(cs->status, 0, 1) == 0) {
    cs->status[1] = where;
    cs->status[2] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  }
  __threadfence();
}

// Checked builds: a tile outside its cache records the failure (code, where,
// value) and aborts the CTA through the same path as a timed-out wait.
__device__ __noinline__ void raise_bounds(int where, int value) {
  CtaState* cs = cta_state();
  *reinterpret_cast<volatile int*>(&cs->abort_flag) = 1;
  record_bounds(cs->status, where, value);
}

// Bounded wait.  Returns false when the CTA is (or becomes) aborted.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, int where) {
  CtaState* cs = cta_state();
  const long long t0 = clock64();
  while (true) {
    if (*reinterpret_cast<volatile int*>(&cs->abort_flag)) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > cs->budget) {
      raise_abort(where);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, where);
}

// Bounded wait whose outcome is the same for all 32 lanes of the warp (the
// warp-collective tcgen05.ld / st that follow need a converged warp).
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, int where) {
  const bool ok = wait_bar(bar, parity, where);
  return __all_sync(0xffffffffu, ok);
}

// Wait with a fixed budget, ignoring the abort flag (used to drain).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kDrainBudget) {
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tile load with an L2 cache policy (createpolicy) for the copied lines.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy that makes the lines it touches the first to be evicted.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Tile stores from shared memory (bulk-group completion).  Rows outside the
// tensor are not written.  The source may be reused once wait_group.read has
// returned; the writes themselves are complete when the grid is.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the copy engine.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One lane of a converged warp (elect.sync), the same lane every time.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(pred));
  return pred != 0;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format:
// start>>4 in [0,14), LBO>>4 in [16,30), SBO>>4 in [32,46), version 1 at 46,
// swizzle mode 2 = 128B at [61,64)).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A and B both
// bf16 (or both f16), A K-major, B K-major or MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
      "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
      "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Named barrier over the eight softmax warps.
__device__ __forceinline__ void softmax_sync(int id) {
  asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory");
}

// Named barrier over one softmax group's four warps (ids 3 and 4); the
// second form also returns whether `pred` holds in all 128 threads.
__device__ __forceinline__ void group_sync(int qi) {
  asm volatile("bar.sync %0, 128;" ::"r"(3 + qi) : "memory");
}
__device__ __forceinline__ bool group_all(bool pred, int qi) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(3 + qi)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr), "r"(v)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Ties the registers to a point after tcgen05.wait::ld so that no use of them
// is scheduled before the wait.
__device__ __forceinline__ void reg_fence(uint32_t (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[i])::"memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
  } else {
    __half2 t = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
  }
}

// MMA with A read from TMEM (two 16-bit elements per column, row m in lane m).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// Two fp32 FMAs / adds in one instruction.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ------------------------------------------------------------------ kernel
template <int OFF, int N>
__device__ __forceinline__ void tmem_st16_at(uint32_t taddr, const uint32_t (&v)[N]);

// Rare path of a score tile whose row sum left [2^-64, 2^64] (or is not a
// number): S is still intact in TMEM.  Rereads it, moves the reference of the
// overflowing rows to their max, stores the redone P over S's first 64
// columns, and rescales O once the previous P V product has completed.
// Returns false when that wait gave up.
template <bool BF16>
__device__ __noinline__ bool rescue_tile(uint32_t S_, uint32_t O_, float sl2, bool moved, int j,
                                         uint64_t* prev_done, uint32_t prev_parity, float* m_ref_io, uint64_t* ta_out,
                                         uint64_t* tb_out, float* alpha_out) {
  uint32_t v[BN];
  tmem_ld32(S_, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
  tmem_ld32(S_ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
  tmem_ld32(S_ + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
  tmem_ld32(S_ + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < BN; ++c) asm volatile("" : "+r"(v[c])::"memory");
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < BN; c += 8) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      m4[u] = fmax3(m4[u], __uint_as_float(v[c + 2 * u]), __uint_as_float(v[c + 2 * u + 1]));
  }
  const float m_ref = *m_ref_io;
  const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
  const float m_new = moved ? mt : m_ref;
  const float alpha = j > 0 ? ex2(m_ref - m_new) : 0.f;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const uint64_t negm2 = f2_pack(-m_new, -m_new);
  uint32_t pk[BN / 2];
  uint64_t ta = 0, tb = 0;
#pragma unroll
  for (int t = 0; t < BN / 2; ++t) {
    const uint64_t x = ffma2(f2_pack(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1])), sl2x2, negm2);
    const float p0 = ex2(f2_lo(x)), p1 = ex2(f2_hi(x));
    if (t & 1) tb = fadd2(tb, f2_pack(p0, p1));
    else ta = fadd2(ta, f2_pack(p0, p1));
    pk[t] = pack2<BF16>(p0, p1);
  }
  tmem_st16_at<0>(S_, pk);
  tmem_st16_at<16>(S_ + 16, pk);
  tmem_st16_at<32>(S_ + 32, pk);
  tmem_st16_at<48>(S_ + 48, pk);
  bool ok = true;
  if (j > 0) {
    ok = wait_bar_warp(prev_done, prev_parity, 8);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < HD / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(O_ + cc * 32, o);
        tmem_wait_ld();
        reg_fence(o);
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
        tmem_st32(O_ + cc * 32, o);
      }
    }
  }
  *m_ref_io = m_new;
  *ta_out = ta;
  *tb_out = tb;
  *alpha_out = alpha;
  return ok;
}

template <int OFF, int N>
__device__ __forceinline__ void tmem_st16_at(uint32_t taddr, const uint32_t (&v)[N]) {
  static_assert(OFF + 16 <= N, "range");
  tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(&v[OFF]));
}

// 32 consecutive TMEM columns of this thread's lane into v[off, off + 32).
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(OFF + 32 <= N, "range");
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[OFF]));
}

// One launch serves up to kTcMaxBatch independent requests (streams, each with
// its own cache, plan and split-KV partials).  Everything a CTA needs is in the
// launch parameters; the grid is one-dimensional and request r owns CTAs
// [cta0, cta0 + q_blocks * H * n_splits), ordered query block fastest, then
// head, then split.
struct TcRequest {
  const KvTile* tiles;
  float* part_o;           // [n_splits][n_q][H][D] (n_splits > 1)
  float* part_lse;         // [n_splits][n_q][H]
  int32_t* status;
  int32_t n_tiles, n_splits, q_row0, n_q, page_base, cta0, q_blocks, max_pages, page_size;
};
// MAXB: requests the parameter block has room for -- 1 for single-stream
// launches, which then pass about 0.9 KB of parameters instead of 11.6 KB.
template <int MAXB>
struct TcLaunch {
  CUtensorMap q_map;       // [rows, H * D] over every request's query rows
  CUtensorMap cache_map[MAXB];    // 3D view of each request's whole cache
  CUtensorMap cache_map_u[MAXB][4];  // the same with 8-, 16-, 32- and 64-row boxes
  CUtensorMap out_map[MAXB];      // one split: the request's output rows [n_q, H * D], 128 x 64 boxes
  CUtensorMap part_map[MAXB];     // several splits: its partials [n_splits][n_q][H * D] fp32, 128 x 32 boxes
  void* out;               // [rows, H, D]
  int32_t count, num_heads, stall_test;
  int32_t allow_dual;      // single-query-tile CTAs may use dual mode (three or more waves of CTAs)
  int32_t q_rows_cta;      // query rows per CTA: 256 (two tiles) or 128 (one tile)
  float sm_scale_log2;
  long long wait_budget;
  TcRequest req[MAXB];
};
// Above the classic 4 KB: kernel parameters may take up to 32764 bytes on
// every architecture this file builds for (CUDA 12.1 and later).
static_assert(sizeof(TcLaunch<kTcMaxBatch>) <= 32764, "kernel parameter space");

template <bool BF16, int MAXB>
__global__ void __launch_bounds__(REG_BOUND_THREADS, 1)
attn_tc_kernel(const __grid_constant__ TcLaunch<MAXB> P) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                   // [STAGES]
  uint64_t* kv_empty = kv_full + STAGES;          // [STAGES]
  uint64_t* s_full = kv_empty + STAGES;           // [NBUF] S(k) written by the tensor core
  uint64_t* p_full = s_full + NBUF;               // [NBUF] P(k) written (and O rescaled)
  uint64_t* buf_free = p_full + NBUF;             // [NBUF] P(k) V done: the buffer may take S(k+3)
  // [QT][3] O_i += P_i(j) V(j) done, on barrier [i][j % 3].  Rotating over
  // three barriers keeps every parity wait unambiguous: when a softmax
  // thread waits for product j of its accumulator, product j - 3 (the
  // barrier's previous phase) has completed -- S of the thread's current
  // tile waited for the P V product three score tiles back -- and product
  // j + 3 cannot have been issued, so the barrier it polls is either one
  // phase short of the target or at it.
  uint64_t* o_done = buf_free + NBUF;
  uint64_t* drain = o_done + 3 * QT;               // [2] one per MMA-issuing warp
  uint64_t* never = drain + 2;                    // signalled by nothing (timeout test)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  CtaState* cstate = reinterpret_cast<CtaState*>(smem + OFF_STATE);
  volatile int* abort_flag = &cstate->abort_flag;
  static_assert((1 + 2 * STAGES + 3 * NBUF + 3 * QT + 3) * 8 + 8 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Which request, query block, head and split this CTA serves.
  int rq = 0;
  while (rq + 1 < P.count && (int)blockIdx.x >= P.req[rq + 1].cta0) ++rq;
  const TcRequest& R = P.req[rq];
  const int local = (int)blockIdx.x - R.cta0;
  const int qblock = local % R.q_blocks;
  const int h = (local / R.q_blocks) % P.num_heads;
  const int split = local / (R.q_blocks * P.num_heads);
  const int q0 = qblock * P.q_rows_cta;           // first query row within the request
  const bool has_q1 = P.q_rows_cta > BM && q0 + BM < R.n_q;
  const int nq = has_q1 ? 2 : 1;
  const int t0 = (int)(((int64_t)split * R.n_tiles) / R.n_splits);
  const int t1 = (int)(((int64_t)(split + 1) * R.n_tiles) / R.n_splits);
  const int n = t1 - t0;
  // Dual mode: a CTA with a single query tile lets both softmax groups work
  // on it, each on every other KV tile and with its own O accumulator; group
  // 0 combines the two halves at the end.  Measured, it pays when CTAs queue
  // for SMs in three or more waves, and costs a few percent in one or two.
  const bool dual = P.allow_dual && !has_q1 && n >= 2;
  const int groups = (has_q1 || dual) ? 2 : 1;    // active softmax groups
  const int per_tile = dual ? 1 : nq;             // score tiles per KV tile
  const int n_s = n * per_tile;                   // score tiles of this CTA
  const KvTile* tiles = R.tiles;
  const CUtensorMap* cache_map = &P.cache_map[rq];
  const CUtensorMap* maps_u = P.cache_map_u[rq];

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);                 // the S and the P V issuer
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], GROUP_THREADS);
      mbar_init(&buf_free[b], 1);
    }
    for (int i = 0; i < 3 * QT; ++i) mbar_init(&o_done[i], 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    cstate->status = R.status;
    cstate->budget = P.wait_budget;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Barriers and TMEM are set up while the previous kernel of the stream may
  // still drain; nothing below runs before it has completed.
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------ TMA producer
    // The whole warp runs the loop and its waits; one elected lane issues.
    if (n > 0) {
      const bool leader = elect_one();
      // K/V lines are read by the CTAs of one head and split at about the
      // same time and never again in this launch, so they are loaded
      // evict-first: the split-KV partials written meanwhile stay in L2 for
      // the merge instead of going out to HBM and back.
      const uint64_t kv_policy = policy_evict_first();
      int issued = 0;
      if (leader) {
        mbar_expect_tx(q_full, nq * Q_BYTES);
        tma_load_2d(sQ, &P.q_map, h * HD, R.q_row0 + q0, q_full);
        if (has_q1) tma_load_2d(sQ + Q_BYTES, &P.q_map, h * HD, R.q_row0 + q0 + BM, q_full);
      }
      for (int j = 0; j < n; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES && !wait_bar_warp(&kv_empty[st], ((j / STAGES) + 1) & 1, 1)) break;
        const KvTile tile = tiles[t0 + j];
        const int plane = (R.page_base + tile.page) * 2;
        const int units1 = (tile.rows + 7) >> 3;        // 8-row units of the first segment
        if (KVC_CHECKED &&
            (tile.page < 0 || tile.page >= R.max_pages || tile.row0 < 0 || tile.rows < 1 || tile.rows > BN ||
             tile.row0 + tile.rows > R.page_size || h >= P.num_heads ||
             (tile.page2 < 0 ? tile.rows2 != 0
                             : (tile.page2 >= R.max_pages || tile.row0_2 < 0 || tile.rows2 < 1 ||
                                units1 * 8 + tile.rows2 > BN || tile.row0_2 + tile.rows2 > R.page_size)))) {
          if (leader) raise_bounds(401, t0 + j);
          __syncwarp();
          break;
        }
        if (leader) {
          mbar_expect_tx(&kv_full[st], 2 * TILE_BYTES);
          if (tile.page2 < 0) {
            tma_load_3d_hint(sK + st * TILE_BYTES, cache_map, h * HD, tile.row0, plane, &kv_full[st], kv_policy);
            tma_load_3d_hint(sV + st * TILE_BYTES, cache_map, h * HD, tile.row0, plane + 1, &kv_full[st], kv_policy);
          } else {
            // Packed tile: the first segment's units (8 rows each) at units
            // [0, units1) of the stage, then the second page's from its row0_2
            // at units [units1, 16).  Each segment (1 to 15 units) is copied as
            // boxes of 8, 4, 2 and 1 units, largest first, every box starting on
            // a 1024-byte swizzle atom.  Units past the second segment's rows
            // read rows past its valid count (masked in S; past the page end the
            // copy fills zeros), so every byte of the stage is written.
            auto load_units = [&](int unit, int count, int row, int pl) {
#pragma unroll
              for (int m = 3; m >= 0; --m) {
                if (count & (1 << m)) {
                  const uint32_t off = st * TILE_BYTES + unit * 1024;
                  tma_load_3d_hint(sK + off, &maps_u[m], h * HD, row, pl, &kv_full[st], kv_policy);
                  tma_load_3d_hint(sV + off, &maps_u[m], h * HD, row, pl + 1, &kv_full[st], kv_policy);
                  unit += 1 << m;
                  row += 8 << m;
                }
              }
            };
            load_units(0, units1, tile.row0, plane);
            load_units(units1, BN / 8 - units1, tile.row0_2, (R.page_base + tile.page2) * 2);
          }
        }
        issued = j + 1;
      }
      if (*abort_flag && leader) {
        // Let every copy this warp started land before the CTA exits.
        drain_bar(q_full, 0);
        for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
          drain_bar(&kv_full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == S_WARP || warp == PV_WARP) {
    // ------------------------------------------------------ MMA issuers
    // Two warps feed the tensor core: one issues the S MMAs, the other the
    // P V MMAs, so that each one's barrier waits overlap the other's issue.
    // Each runs its loop and waits with the whole warp (warp-uniform values);
    // one elected lane issues the MMAs and the commits.  Indices and barrier
    // phases advance incrementally.
    if (n > 0) {
      const bool leader = elect_one();
      // Descriptors are built once; a step along K or to another stage only
      // adds to the start-address field (address >> 4, 14 bits, no carry for
      // shared-memory addresses below 256 KB), so each MMA costs one add.
      constexpr uint64_t STAGE_STEP = TILE_BYTES >> 4;     // next K/V stage
      constexpr uint64_t K16_STEP = 32 >> 4;               // 16 bf16 along K inside a 128-byte row
      constexpr uint64_t V16_STEP = (16 * 128) >> 4;       // 16 rows of V
      constexpr uint64_t Q_STEP = Q_BYTES >> 4;            // second query tile
      int i = 0, b = 0, st = 0;
      uint32_t kv_par = 0, buf_par = 0;                    // one parity bit per stage / buffer
      bool ok = true;
      if (warp == S_WARP) {
        // S(k) = Q_i K(j)^T into buffer k mod 3, once K(j) has landed and the
        // P V product that last read the buffer has completed.
        constexpr uint32_t IDESC_S = idesc_f16(BM, BN, BF16, false);
        const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
        ok = wait_bar_warp(q_full, 0, 2);
        for (int k = 0; ok && k < n_s; ++k) {
          if (i == 0) {
            ok = wait_bar_warp(&kv_full[st], (kv_par >> st) & 1, 3);
            kv_par ^= 1u << st;
          }
          if (ok && k >= NBUF) {
            ok = wait_bar_warp(&buf_free[b], (buf_par >> b) & 1, 4);
            buf_par ^= 1u << b;
          }
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK = dK0 + (uint64_t)st * STAGE_STEP;
          const uint64_t dQ = dQ0 + (uint64_t)(dual ? 0 : i) * Q_STEP;
          const uint32_t d = tmem + buf_col(b);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
              umma(d, dQ + kk * K16_STEP, dK + kk * K16_STEP, IDESC_S, kk > 0);
            umma_commit(&s_full[b]);
            if (i == per_tile - 1) umma_commit(&kv_empty[st]);
          }
          __syncwarp();
          b = b == NBUF - 1 ? 0 : b + 1;
          if (++i == per_tile) {
            i = 0;
            st = st == STAGES - 1 ? 0 : st + 1;
          }
        }
      } else {
        // O_i += P(k) V(j), P read from the first 64 columns of buffer k mod 3.
        // Timeout test: a wait that nothing ends, so the bound runs out and the
        // whole CTA takes the abort path.
        constexpr uint32_t IDESC_O = idesc_f16(BM, HD, BF16, true);
        const uint64_t dV0 = sdesc_sw128(smem_u32(sV), BN * 128, 1024);
        uint32_t p_par = 0;
        ok = !P.stall_test || wait_bar_warp(never, 0, 12);
        for (int k = 0, j = 0; ok && k < n_s; ++k) {
          if (i == 0) {
            // V(j) landed (already true in practice: S(k) needed K(j) of the same copy).
            ok = wait_bar_warp(&kv_full[st], (kv_par >> st) & 1, 3);
            kv_par ^= 1u << st;
          }
          if (ok) {
            ok = wait_bar_warp(&p_full[b], (p_par >> b) & 1, 5);
            p_par ^= 1u << b;
          }
          if (!ok) break;
          tc_fence_after();
          const uint64_t dV = dV0 + (uint64_t)st * STAGE_STEP;
          // The O accumulator this score tile goes to, and how many tiles
          // that accumulator has taken before.
          const int grp = dual ? (k & 1) : i;
          const int jg = dual ? (k >> 1) : j;
          const uint32_t o = tmem + o_col(grp), pa = tmem + buf_col(b);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              umma_ts(o, pa + kk * 8, dV + kk * V16_STEP, IDESC_O, (jg > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&buf_free[b]);
            umma_commit(&o_done[3 * grp + jg % 3]);
            if (i == per_tile - 1) umma_commit(&kv_empty[st]);
          }
          __syncwarp();
          b = b == NBUF - 1 ? 0 : b + 1;
          if (++i == per_tile) {
            i = 0;
            ++j;
            st = st == STAGES - 1 ? 0 : st + 1;
          }
        }
      }
      // Every MMA this warp issued has completed once its drain barrier flips.
      uint64_t* my_drain = warp == S_WARP ? drain : drain + 1;
      if (leader) {
        umma_commit(my_drain);
        drain_bar(my_drain, 0);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ softmax + epilogue
    const int qi = warp >> 2;                        // query tile of this warp
    const int quarter = warp & 3;                    // TMEM lanes [32 quarter, +32)
    const int r = quarter * 32 + lane;               // query row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t O_ = lane_base + o_col(qi);
    const float sl2 = P.sm_scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    // Starting reference: any finite value within a few tens of the scores
    // (log2 units) works, so ordinary first tiles need no row max either.
    float m_ref = 0.f;
    uint64_t la = 0, lb = 0;                         // row-sum partials (two fp32 pairs)
    bool ok = n > 0 && qi < groups;                  // warp-uniform
    // This group's tiles: j counts them; in dual mode the group takes KV
    // tiles qi, qi + 2, ..., otherwise every KV tile.
    const int n_g = dual ? (n - qi + 1) / 2 : n;

    // Valid rows of a tile: {rows, rows2} -- the first segment's rows, then
    // (packed tiles) the second's from row ceil(rows / 8) * 8.
    // Both (at most 128) travel in one register: rows | rows2 << 8.
    auto tile_rows = [&](int t) {
      const int2 r = *reinterpret_cast<const int2*>(&tiles[t].rows);
      return r.x | (r.y << 8);
    };
    int rows_next = ok ? tile_rows(t0 + (dual ? qi : 0)) : 0;
    for (int j = 0; ok && j < n_g; ++j) {
      const int k = j * groups + qi, b = k % NBUF;
      const int rows_valid = rows_next;
      if (j + 1 < n_g) rows_next = tile_rows(t0 + (dual ? k + 2 : j + 1));   // prefetch for the next tile
      ok = wait_bar_warp(&s_full[b], (k / NBUF) & 1, 6);
      if (!ok) break;
      tc_fence_after();
      const uint32_t S_ = lane_base + buf_col(b);
      const int rows1 = rows_valid & 0xff, rows2 = rows_valid >> 8;
      if (rows1 + rows2 < BN) {
        // Rows of the tile that hold no visible token never enter the softmax:
        // their scores are overwritten with -inf in TMEM before the row is
        // read (short loops keep this rare case out of the unrolled hot path).
        // They are [rows, ceil8(rows)) and [ceil8(rows) + rows2, BN).
        const uint32_t ninf = __float_as_uint(-INFINITY);
        const int a8 = (rows1 + 7) & ~7;
        int c = rows1;
        for (; c < a8; ++c) tmem_st1(S_ + c, ninf);
        c = a8 + rows2;
        for (; (c & 7) != 0; ++c) tmem_st1(S_ + c, ninf);
        for (; c < BN; c += 8) tmem_st8(S_ + c, ninf);
        tmem_wait_st();
      }
      // The row's 128 scores: the first half is waited for, the second half's
      // loads are in flight while the first half is exponentiated.
      uint32_t v[BN];
      tmem_ld32_at<0>(S_, v);
      tmem_ld32_at<32>(S_ + 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) asm volatile("" : "+r"(v[c])::"memory");
      tmem_ld32_at<64>(S_ + 64, v);
      tmem_ld32_at<96>(S_ + 96, v);
      // P = 2^(s * scale - m_ref) against the running reference, held in
      // registers until the row sum shows that it is usable.  The reference
      // only has to keep P and the sums finite -- their relative precision
      // does not depend on it -- so a tile's own max is needed only when its
      // row sum exceeds 2^64 or is not a number (after a jump of about 57 or
      // more in log2 units), or -- on the first tile -- falls below 2^-64.
      uint32_t pk[BN / 2];
      uint64_t ta = 0, tb = 0;
      {
        const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
#pragma unroll
        for (int t = 0; t < BN / 2; ++t) {
          if (t == BN / 4) {
            tmem_wait_ld();                            // the second half of the scores
#pragma unroll
            for (int c = BN / 2; c < BN; ++c) asm volatile("" : "+r"(v[c])::"memory");
          }
          const uint64_t x = ffma2(f2_pack(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1])), sl2x2, negm2);
          const float p0 = ex2(f2_lo(x)), p1 = ex2(f2_hi(x));
          if (t & 1) tb = fadd2(tb, f2_pack(p0, p1));
          else ta = fadd2(ta, f2_pack(p0, p1));
          pk[t] = pack2<BF16>(p0, p1);
        }
      }
      const float tsum = (f2_lo(ta) + f2_hi(ta)) + (f2_lo(tb) + f2_hi(tb));
      // The first tile also moves the reference when its sum underflows.
      const bool moved = !(tsum <= 0x1p64f) || (j == 0 && !(tsum >= 0x1p-64f));
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, moved)) {
        // Rare (out of line, to keep its registers out of this loop): the
        // previous product into this accumulator is j - 1 (waited for only
        // when j > 0).
        ok = rescue_tile<BF16>(S_, O_, sl2, moved, j, &o_done[3 * qi + (j + 2) % 3], ((j - 1) / 3) & 1, &m_ref, &ta,
                               &tb, &alpha);
        if (!ok) break;
      } else {
        // P as 16-bit pairs over S's first 64 columns.
        tmem_st16_at<0>(S_, pk);
        tmem_st16_at<16>(S_ + 16, pk);
        tmem_st16_at<32>(S_ + 32, pk);
        tmem_st16_at<48>(S_ + 48, pk);
      }
      const uint64_t alpha2 = f2_pack(alpha, alpha);
      la = ffma2(la, alpha2, ta);
      lb = ffma2(lb, alpha2, tb);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[b]);                       // P(k) is in TMEM (and O_i rescaled)
    }
    if (n > 0 && qi < groups) {
      // Epilogue: wait for this group's last P V product, normalise, write
      // the row.  In dual mode group 1 hands its row max and sum to group 0
      // through shared memory, and group 0 combines both halves (group 1's O
      // sits in the same TMEM lanes) before writing.
      bool good = ok && wait_bar_warp(&o_done[3 * qi + (n_g - 1) % 3], ((n_g - 1) / 3) & 1, 9);
      float l = (f2_lo(la) + f2_hi(la)) + (f2_lo(lb) + f2_hi(lb));
      float m_fin = m_ref, w0 = 1.f, w1 = 0.f;
      if (dual) {
        float* xr = reinterpret_cast<float*>(smem + OFF_XCH) + 3 * r;
        if (qi == 1) {
          xr[0] = m_ref;
          xr[1] = l;
          xr[2] = good ? 0.f : 1.f;
        }
        softmax_sync(2);
        if (qi == 1) {
          good = false;                              // group 0 writes the row
        } else if (good && xr[2] == 0.f) {
          const int n_g1 = n / 2;                    // group 1's tiles
          good = wait_bar_warp(&o_done[3 + (n_g1 - 1) % 3], ((n_g1 - 1) / 3) & 1, 9);
          const float m1 = xr[0], l1 = xr[1];
          m_fin = fmaxf(m_ref, m1);
          w0 = ex2(m_ref - m_fin);
          w1 = ex2(m1 - m_fin);
          l = w0 * l + w1 * l1;
        } else {
          good = false;
        }
      }
      // Output: the group's 128 rows are staged in shared memory -- its own Q
      // tile, free once its last S product has completed (in dual mode group
      // 0 writes, after both groups' S products) -- in the 128-byte swizzle,
      // and leave as TMA stores of whole row segments (the copy clips rows
      // past n_q), instead of 16-byte stores scattered over 128 rows.  The
      // group's four warps first agree that all of them got here in order.
      if (group_all(good, qi)) {
        tc_fence_after();
        uint32_t v[HD];
        tmem_ld32_at<0>(O_, v);
        tmem_ld32_at<32>(O_ + 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < HD; ++c) asm volatile("" : "+r"(v[c])::"memory");
        if (dual) {
          uint32_t v1[HD];
          const uint32_t O1 = lane_base + o_col(1);
          tmem_ld32_at<0>(O1, v1);
          tmem_ld32_at<32>(O1 + 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HD; ++c)
            v[c] = __float_as_uint(fmaf(w1, __uint_as_float(v1[c]), w0 * __uint_as_float(v[c])));
        }
        const int row = q0 + qi * BM + r;             // within the request
        const float inv = 1.f / l;
        uint8_t* stage = sQ + qi * Q_BYTES;           // 128 rows x 128 bytes
        const uint32_t srow = smem_u32(stage) + r * 128;
        const bool issuer = (warp & 3) == 0 && lane == 0;
        if (R.n_splits == 1) {
          // 64 16-bit values per row: eight 16-byte chunks, chunk c at c ^ (r mod 8).
#pragma unroll
          for (int c = 0; c < HD / 8; ++c) {
            const float* o = reinterpret_cast<const float*>(&v[8 * c]);
            st_shared16(srow + ((c ^ (r & 7)) << 4), pack2<BF16>(o[0] * inv, o[1] * inv),
                        pack2<BF16>(o[2] * inv, o[3] * inv), pack2<BF16>(o[4] * inv, o[5] * inv),
                        pack2<BF16>(o[6] * inv, o[7] * inv));
          }
          fence_proxy_async();
          group_sync(qi);
          if (issuer) {
            tma_store_2d(&P.out_map[rq], stage, h * HD, q0 + qi * BM);
            bulk_commit();
            bulk_wait_read();
          }
        } else {
          if (row < R.n_q) R.part_lse[((int64_t)split * R.n_q + row) * P.num_heads + h] = m_fin + __log2f(l);
          // 64 fp32 values per row: two halves of 32 (128 bytes), one copy each.
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (half) group_sync(qi);                 // the first copy has read the stage
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* o = &v[32 * half + 4 * c];
              st_shared16(srow + ((c ^ (r & 7)) << 4), __float_as_uint(__uint_as_float(o[0]) * inv),
                          __float_as_uint(__uint_as_float(o[1]) * inv), __float_as_uint(__uint_as_float(o[2]) * inv),
                          __float_as_uint(__uint_as_float(o[3]) * inv));
            }
            fence_proxy_async();
            group_sync(qi);
            if (issuer) {
              tma_store_3d(&P.part_map[rq], stage, h * HD + 32 * half, q0 + qi * BM, split);
              bulk_commit();
              bulk_wait_read();                       // before the stage is reused or goes away
            }
          }
        }
      }
    }
    __syncwarp();
    tmem_wait_ld();                                  // nothing of ours in flight on the way out
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool configured_smem[4] = {false, false, false, false};

}  // namespace

bool tc_supported(int dtype, int head_dim, int num_heads, int page_size) {
  return (dtype == 0 || dtype == 1) && head_dim == HD && num_heads >= 1 && page_size >= 1;
}

TcMaps* tc_create_maps(void* cache, int dtype, int num_blocks, int max_pages, int page_size, int num_heads,
                       int head_dim, cudaError_t* err) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !tc_supported(dtype, head_dim, num_heads, page_size)) {
    if (err) *err = cudaErrorNotSupported;
    return nullptr;
  }
  TcMaps* m = new (std::nothrow) TcMaps();
  if (!m) {
    if (err) *err = cudaErrorMemoryAllocation;
    return nullptr;
  }
  m->dtype = dtype;
  m->num_heads = num_heads;
  m->head_dim = head_dim;
  const cuuint64_t row_bytes = (cuuint64_t)num_heads * head_dim * 2;
  cuuint64_t dims[3] = {(cuuint64_t)num_heads * head_dim, (cuuint64_t)page_size,
                        (cuuint64_t)num_blocks * max_pages * 2};
  cuuint64_t strides[2] = {row_bytes, row_bytes * page_size};
  cuuint32_t box[3] = {HD, BN, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty = dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&m->cache, ty, 3, cache, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  for (int u = 0; u < 4 && r == CUDA_SUCCESS; ++u) {
    cuuint32_t box_u[3] = {HD, (cuuint32_t)(8 << u), 1};
    r = enc(&m->cache_u[u], ty, 3, cache, dims, strides, box_u, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    delete m;
    if (err) *err = cudaErrorInvalidValue;
    return nullptr;
  }
  return m;
}

void tc_destroy_maps(TcMaps* m) { delete m; }

namespace {

template <int MAXB>
cudaError_t launch_impl(const TcBatchArgs& b, EncodeTiledFn enc, cudaStream_t stream) {
  TcLaunch<MAXB> P;
  std::memset(&P, 0, sizeof(P));
  const cuuint64_t row_bytes = (cuuint64_t)b.num_heads * HD * 2;
  cuuint64_t dims[2] = {(cuuint64_t)b.num_heads * HD, (cuuint64_t)b.rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {HD, BM};
  cuuint32_t estr[2] = {1, 1};
  CUresult cr = enc(&P.q_map, b.dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(b.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  P.out = b.out;
  P.count = b.count;
  P.num_heads = b.num_heads;
  P.stall_test = b.stall_test;
  P.sm_scale_log2 = b.sm_scale_log2;
  P.wait_budget = b.wait_budget;
  P.q_rows_cta = b.q_tiles * BM;
  int64_t ctas = 0;
  for (int r = 0; r < b.count; ++r) {
    const TcRequestDesc& d = b.req[r];
    if (!d.maps || d.n_q < 0 || d.n_splits < 1 || d.q_row0 < 0 || d.q_row0 + d.n_q > b.rows)
      return cudaErrorInvalidValue;
    TcRequest& q = P.req[r];
    if (d.n_q > 0) {
      // Output tile maps: one split writes bf16 / f16 rows of `out`; several
      // write fp32 partials [n_splits][n_q][H * D].  Both use 128-byte rows
      // in the 128-byte swizzle, as staged by the epilogue.
      CUresult mr;
      if (d.n_splits == 1) {
        cuuint64_t odims[2] = {(cuuint64_t)b.num_heads * HD, (cuuint64_t)d.n_q};
        cuuint64_t ostr[1] = {row_bytes};
        cuuint32_t obox[2] = {HD, BM};
        mr = enc(&P.out_map[r], b.dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                 static_cast<char*>(b.out) + (size_t)d.q_row0 * row_bytes, odims, ostr, obox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      } else {
        const cuuint64_t prow = (cuuint64_t)b.num_heads * HD * 4;
        cuuint64_t pdims[3] = {(cuuint64_t)b.num_heads * HD, (cuuint64_t)d.n_q, (cuuint64_t)d.n_splits};
        cuuint64_t pstr[2] = {prow, prow * (cuuint64_t)d.n_q};
        cuuint32_t pbox[3] = {32, BM, 1};
        cuuint32_t pestr[3] = {1, 1, 1};
        mr = enc(&P.part_map[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, d.part_o, pdims, pstr, pbox, pestr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      }
      if (mr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    P.cache_map[r] = d.maps->cache;
    for (int u = 0; u < 4; ++u) P.cache_map_u[r][u] = d.maps->cache_u[u];
    q.tiles = d.tiles;
    q.part_o = d.part_o;
    q.part_lse = d.part_lse;
    q.status = d.status;
    q.n_tiles = d.n_tiles;
    q.n_splits = d.n_splits;
    q.q_row0 = d.q_row0;
    q.n_q = d.n_q;
    q.page_base = d.block * d.max_pages;
    q.max_pages = d.max_pages;
    q.page_size = d.page_size;
    q.q_blocks = (d.n_q + P.q_rows_cta - 1) / P.q_rows_cta;
    q.cta0 = (int32_t)ctas;
    ctas += (int64_t)q.q_blocks * b.num_heads * d.n_splits;
  }
  if (ctas == 0) return cudaSuccess;
  // Two-tile CTAs: dual mode for their single-tile tail only from about three
  // waves on (measured).  One-tile CTAs always run in dual mode.
  P.allow_dual = (b.q_tiles == 1 || ctas > 2 * (int64_t)b.num_sms) ? 1 : 0;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  const int which = (b.dtype == 0 ? 0 : 1) + (MAXB == 1 ? 0 : 2);
  auto kernel = b.dtype == 0 ? attn_tc_kernel<true, MAXB> : attn_tc_kernel<false, MAXB>;
  if (!configured_smem[which]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_smem[which] = true;
  }
  return launch_kernel(kernel, dim3((unsigned)ctas), dim3(NUM_THREADS), SMEM_BYTES, stream, b.pdl != 0, P);
}

}  // namespace

cudaError_t launch_attn_tc(const TcBatchArgs& b, cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || b.count < 1 || b.count > kTcMaxBatch || b.head_dim != HD) return cudaErrorNotSupported;
  if (b.q_tiles != 1 && b.q_tiles != QT) return cudaErrorInvalidValue;
  return b.count == 1 ? launch_impl<1>(b, enc, stream) : launch_impl<kTcMaxBatch>(b, enc, stream);
}

}  // namespace kvc
