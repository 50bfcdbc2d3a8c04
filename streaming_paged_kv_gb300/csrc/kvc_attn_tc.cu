// Tensor-core paged attention for sm_103a: TMA gathers of K/V page tiles
// through the page table, tcgen05 MMAs with TMEM accumulators, fp32 online
// softmax.
//
// What it computes ([KVC] "Kernel-Level Execution Flow": causal=False,
// pos_encoding_mode="NONE", as many KV heads as query heads):
//     O[t,h,:] = sum_j softmax_j(Q[t,h,:].K[j,h,:] * sm_scale) V[j,h,:]
// over the visible tokens j, which the plan lists as KV tiles of at most 128
// rows of one page (scale pages, live window, then the special pages; a
// page's rows beyond its valid count never enter the softmax, so exact page
// sizes such as 999 need no padding -- [PERF] "Page-Size Handling for FA2 vs
// FA3").
//
// Pages cited by tag: [KVC] "How LingBot-Map Implements the KV Cache Mechanism
// for Streaming Inference with FlashInfer Integration"; [PERF] "How to Improve
// Streaming Inference Performance with FlashInfer KV Cache Backend".
//
// CTA = two 128-row query tiles (Q0, Q1) x one head x one KV split; each K/V
// tile is loaded once and serves both query tiles.  Warps:
//   0-7   softmax + epilogue of Q0, 8-15 softmax + epilogue of Q1.  Within a
//         query tile, warp w owns TMEM lanes [32(w%4), +32) (query rows) and
//         columns [64 h, +64) of each S tile, h = (w/4)%2: two warps share
//         every row, each holding half of its scores
//   16    TMA producer (one lane): Q0/Q1, then K/V tiles into a 4-stage ring
//   17    MMA issuer (one lane): S_i = Q_i K^T into TMEM, O_i += P_i V with P_i
//         read from TMEM
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
// P0 [384,448) P1 [448,512); P holds two 16-bit values per column.
// Q and K/V tiles use the 128-byte swizzle that both TMA and the tensor core
// understand.  Scores live in the log2 domain (scaled by sm_scale * log2 e).
// Each warp exponentiates its half of the row against the running reference
// max m_ref of the row.  The reference moves only when a score exceeds it by
// more than 8 (a factor 256): then the two warps of the row agree on the new
// reference through shared memory, recompute that tile's P from S and rescale
// O and the row sums.  Otherwise P is taken against the stale reference, which
// fp32 accumulation absorbs.
//
// Every mbarrier wait is bounded: when a wait runs out, the thread records
// the fact in the status word, raises a CTA-wide abort flag, and every role
// skips its remaining work, drains its own in-flight copies / MMAs (again
// with a bound), frees TMEM and returns.

#include "kvc_internal.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <new>
#include <type_traits>

namespace kvc {

struct TcMaps {
  CUtensorMap cache;     // 3D view of the whole cache: {H*D, page_size, blocks*pages*2}
  int dtype;
  int num_heads;
  int head_dim;
};

namespace {

constexpr int BM = 128;           // query rows per query tile
constexpr int QT = 2;             // query tiles per CTA
constexpr int BN = 128;           // KV rows per tile
constexpr int HD = 64;            // head dim of this kernel
constexpr int STAGES = 4;
constexpr int NUM_THREADS = 576;
constexpr int PRODUCER_WARP = 16, MMA_WARP = 17;
constexpr int SOFTMAX_THREADS = 2 * BM;              // per query tile: two warps per row
constexpr uint32_t TILE_BYTES = BN * HD * 2;         // 16 KB: one K or V tile
constexpr uint32_t Q_BYTES = BM * HD * 2;            // 16 KB per query tile
constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t s_col(int i) { return i * BN; }
__host__ __device__ constexpr uint32_t o_col(int i) { return 2 * BN + i * HD; }
__host__ __device__ constexpr uint32_t p_col(int i) { return 2 * BN + 2 * HD + i * (BN / 2); }
constexpr float RESCALE_THRESHOLD = 8.0f;            // log2 units
constexpr long long kDrainBudget = 1LL << 26;        // cycles for draining after an abort

// Shared memory map (offsets from a 1024-aligned base).
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + QT * Q_BYTES;
constexpr uint32_t OFF_V = OFF_K + STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + STAGES * TILE_BYTES;
// Row exchange between the two warps of a row: [pair][warp half][slot][33 floats].
constexpr uint32_t OFF_XCH = OFF_BAR + 256;
constexpr uint32_t XCH_BYTES = 8 * 2 * 2 * 33 * 4;
constexpr uint32_t SMEM_BYTES = OFF_XCH + XCH_BYTES + 1024;  // + alignment slack

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

// Bounded wait.  Returns false when the CTA is (or becomes) aborted.
struct Guard {
  volatile int* abort_flag;   // shared
  int32_t* status;            // global
  long long budget;
};

__device__ __noinline__ void raise_abort(const Guard& g, int where) {
  *g.abort_flag = 1;
  if (atomicCAS(g.status, 0, 1) == 0) {
    g.status[1] = where;
    g.status[2] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  }
  __threadfence();
}

__device__ __forceinline__ bool wait_bar(const Guard& g, uint64_t* bar, uint32_t parity, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*g.abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > g.budget) {
      raise_abort(g, where);
      return false;
    }
  }
}

// Bounded wait whose outcome is the same for all 32 lanes of the warp (the
// warp-collective tcgen05.ld / st that follow need a converged warp).
__device__ __forceinline__ bool wait_bar_warp(const Guard& g, uint64_t* bar, uint32_t parity, int where) {
  const bool ok = wait_bar(g, bar, parity, where);
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

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
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

// Named barrier over `count` threads (the two warps of a row pair).
__device__ __forceinline__ void pair_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
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

template <bool BF16>
__device__ __forceinline__ uint32_t scale_pair(uint32_t packed, float alpha) {
  if constexpr (BF16) {
    __nv_bfloat162 t = *reinterpret_cast<__nv_bfloat162*>(&packed);
    return pack2<true>(__low2float(t) * alpha, __high2float(t) * alpha);
  } else {
    __half2 t = *reinterpret_cast<__half2*>(&packed);
    return pack2<false>(__low2float(t) * alpha, __high2float(t) * alpha);
  }
}

template <bool BF16>
__device__ __forceinline__ void store_row(void* dst, const float* o, float inv) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    uint4 u;
    u.x = pack2<BF16>(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
    u.y = pack2<BF16>(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
    u.z = pack2<BF16>(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
    u.w = pack2<BF16>(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
    d[i] = u;
  }
}

// ------------------------------------------------------------------ kernel
template <bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap cache_map,
               const __grid_constant__ CUtensorMap q_map, int32_t page_base) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                 // [STAGES]
  uint64_t* kv_empty = bars + 1 + STAGES;       // [STAGES]
  uint64_t* s_full = bars + 1 + 2 * STAGES;     // [QT] S_i written by the tensor core
  uint64_t* s_free = bars + 3 + 2 * STAGES;     // [QT] S_i copied out by its warpgroup
  uint64_t* p_full = bars + 5 + 2 * STAGES;     // [QT] P_i written (and O_i rescaled)
  uint64_t* p_free = bars + 7 + 2 * STAGES;     // [QT] P_i V product done
  uint64_t* drain = bars + 9 + 2 * STAGES;
  uint64_t* never = bars + 10 + 2 * STAGES;     // signalled by nothing (timeout test)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11 + 2 * STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y, split = blockIdx.z;
  const int q0 = blockIdx.x * (QT * BM);
  const bool has_q1 = q0 + BM < a.n_q;
  const int nq_tiles = has_q1 ? 2 : 1;
  const int t0 = (int)(((int64_t)split * a.n_tiles) / a.n_splits);
  const int t1 = (int)(((int64_t)(split + 1) * a.n_tiles) / a.n_splits);
  const int n = t1 - t0;
  Guard g{abort_flag, a.status, a.wait_budget};

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < QT; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], SOFTMAX_THREADS);
      mbar_init(&p_full[i], SOFTMAX_THREADS);
      mbar_init(&p_free[i], 1);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------ TMA producer
    // The whole warp runs the loop and its waits; one elected lane issues.
    if (n > 0) {
      const bool leader = elect_one();
      int issued = 0;
      if (leader) {
        mbar_expect_tx(q_full, nq_tiles * Q_BYTES);
        tma_load_2d(sQ, &q_map, h * HD, q0, q_full);
        if (has_q1) tma_load_2d(sQ + Q_BYTES, &q_map, h * HD, q0 + BM, q_full);
      }
      for (int j = 0; j < n; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES && !wait_bar_warp(g, &kv_empty[st], ((j / STAGES) + 1) & 1, 1)) break;
        const KvTile tile = a.tiles[t0 + j];
        const int plane = (page_base + tile.page) * 2;
        if (leader) {
          mbar_expect_tx(&kv_full[st], 2 * TILE_BYTES);
          tma_load_3d(sK + st * TILE_BYTES, &cache_map, h * HD, tile.row0, plane, &kv_full[st]);
          tma_load_3d(sV + st * TILE_BYTES, &cache_map, h * HD, tile.row0, plane + 1, &kv_full[st]);
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
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and its waits with warp-uniform values;
    // one elected lane issues the MMAs and the commits.
    if (n > 0) {
      const bool leader = elect_one();
      constexpr uint32_t IDESC_S = idesc_f16(BM, BN, BF16, false);
      constexpr uint32_t IDESC_O = idesc_f16(BM, HD, BF16, true);
      // Descriptors are built once; a step along K or to another stage only
      // adds to the start-address field (address >> 4, 14 bits, no carry for
      // shared-memory addresses below 256 KB), so each MMA costs one add.
      const uint64_t dQ[QT] = {sdesc_sw128(smem_u32(sQ), 16, 1024), sdesc_sw128(smem_u32(sQ) + Q_BYTES, 16, 1024)};
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), BN * 128, 1024);
      constexpr uint64_t STAGE_STEP = TILE_BYTES >> 4;     // next K/V stage
      constexpr uint64_t K16_STEP = 32 >> 4;               // 16 bf16 along K inside a 128-byte row
      constexpr uint64_t V16_STEP = (16 * 128) >> 4;       // 16 rows of V
      auto issue_s = [&](int i, int j) {
        const uint64_t dK = dK0 + (uint64_t)(j % STAGES) * STAGE_STEP;
        const uint32_t d = tmem + s_col(i);
        if (leader) {
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma(d, dQ[i] + k * K16_STEP, dK + k * K16_STEP, IDESC_S, k > 0);
          umma_commit(&s_full[i]);
        }
        __syncwarp();
      };
      // Timeout test: a wait that nothing ends, so the bound runs out and the
      // whole CTA takes the abort path.
      bool ok = !a.stall_test || wait_bar_warp(g, never, 0, 12);
      ok = ok && wait_bar_warp(g, q_full, 0, 2) && wait_bar_warp(g, &kv_full[0], 0, 3);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < nq_tiles; ++i) issue_s(i, 0);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % STAGES;
        if (j + 1 < n) ok = wait_bar_warp(g, &kv_full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1, 3);
        // Per query tile: its next S as soon as its warps have copied S out,
        // then its P V product once P is in TMEM.
        for (int i = 0; ok && i < nq_tiles; ++i) {
          if (j + 1 < n) {
            ok = wait_bar_warp(g, &s_free[i], j & 1, 4);
            if (!ok) break;
            tc_fence_after();
            issue_s(i, j + 1);
          }
          ok = wait_bar_warp(g, &p_full[i], j & 1, 5);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dV = dV0 + (uint64_t)st * STAGE_STEP;
          const uint32_t o = tmem + o_col(i), pa = tmem + p_col(i);
          if (leader) {
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
              umma_ts(o, pa + k * 8, dV + k * V16_STEP, IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
            umma_commit(&p_free[i]);
          }
          __syncwarp();
        }
        if (ok && leader) umma_commit(&kv_empty[st]);
        __syncwarp();
      }
      // Every MMA this warp issued has completed once `drain` flips.
      if (leader) {
        umma_commit(drain);
        drain_bar(drain, 0);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ softmax + epilogue
    const int qi = warp >> 3;                        // query tile of this warp
    const int half = (warp >> 2) & 1;                // which 64 columns of each S tile
    const int quarter = warp & 3;                    // TMEM lanes [32 quarter, +32)
    const int pair = qi * 4 + quarter;               // the two warps sharing these rows
    const int r = quarter * 32 + lane;               // query row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t S_ = lane_base + s_col(qi) + half * 64;
    const uint32_t P_ = lane_base + p_col(qi) + half * 32;
    const uint32_t O_ = lane_base + o_col(qi);
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);
    float* mine = xch + (pair * 2 + half) * 66;      // two slots of 33
    float* theirs = xch + (pair * 2 + (half ^ 1)) * 66;
    const int bar_id = 1 + pair;
    const int col0 = half * 64;
    const float sl2 = a.sm_scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    float m_ref = -INFINITY;
    uint64_t la = 0, lb = 0;                         // row-sum partials over this warp's columns
    bool ok = n > 0 && qi < nq_tiles;                // the same for both warps of a pair

    // P for this warp's 64 columns of tile S into TMEM, against reference m:
    // returns the partial sums; clamps the exponent so that a stale reference
    // can never produce inf (such tiles are recomputed).
    auto make_p = [&](int rows_valid, float m, uint64_t& ta, uint64_t& tb, float* smax) {
      const uint64_t negx2 = f2_pack(-m, -m);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t v[32];
        tmem_ld32(S_ + u * 32, v);
        tmem_wait_ld();
        reg_fence(v);
        if (rows_valid < col0 + 64) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + u * 32 + i >= rows_valid) v[i] = __float_as_uint(-INFINITY);
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float s0 = __uint_as_float(v[2 * i]), s1 = __uint_as_float(v[2 * i + 1]);
          if (smax) *smax = fmax3(*smax, s0, s1);
          const uint64_t x = ffma2(f2_pack(s0, s1), sl2x2, negx2);
          const float p0 = ex2(fminf(f2_lo(x), 120.f)), p1 = ex2(fminf(f2_hi(x), 120.f));
          if (i & 1) tb = fadd2(tb, f2_pack(p0, p1));
          else ta = fadd2(ta, f2_pack(p0, p1));
          pk[i] = pack2<BF16>(p0, p1);
        }
        tmem_st16(P_ + u * 16, pk);
      }
    };

    int rows_next = ok ? a.tiles[t0].rows : 0;
    for (int j = 0; ok && j < n; ++j) {
      const int rows_valid = rows_next;
      if (j + 1 < n) rows_next = a.tiles[t0 + j + 1].rows;   // prefetch for the next tile
      bool good = wait_bar_warp(g, &s_full[qi], j & 1, 6);
      // P_i is free (and O_i stable) once the P V product of the previous tile has completed.
      if (good && j > 0) good = wait_bar_warp(g, &p_free[qi], (j - 1) & 1, 8);
      uint64_t ta = 0, tb = 0;
      float smax = -INFINITY;
      if (good) {
        tc_fence_after();
        make_p(rows_valid, m_ref, ta, tb, &smax);
      }
      // Tell the other warp of these rows whether the reference has to move
      // (or whether this warp gave up), and this row's score max.
      const float mx = smax * sl2;
      const bool need = __any_sync(0xffffffffu, good && mx > m_ref + RESCALE_THRESHOLD);
      float* my_slot = mine + (j & 1) * 33;
      float* their_slot = theirs + (j & 1) * 33;
      my_slot[lane] = mx;
      if (lane == 0) my_slot[32] = __int_as_float((need ? 1 : 0) | (good ? 0 : 2));
      pair_sync(bar_id, 64);
      const int their_flags = __float_as_int(their_slot[32]);
      const float their_mx = their_slot[lane];
      if (!good || (their_flags & 2)) { ok = false; break; }
      if (need || (their_flags & 1)) {
        // Rare: move the reference of the rows whose max grew too far, then
        // recompute this tile's P (S is still in TMEM) and rescale O and l.
        const float row_mx = fmaxf(mx, their_mx);
        const float m_new = row_mx > m_ref + RESCALE_THRESHOLD ? row_mx : m_ref;
        const float alpha = ex2(m_ref - m_new);      // 0 while nothing has been accumulated
        tmem_wait_st();
        ta = tb = 0;
        make_p(rows_valid, m_new, ta, tb, nullptr);
        if (half == 0 && j > 0) {
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(O_ + cc * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(O_ + cc * 32, o);
          }
        }
        la = f2_pack(f2_lo(la) * alpha, f2_hi(la) * alpha);
        lb = f2_pack(f2_lo(lb) * alpha, f2_hi(lb) * alpha);
        m_ref = m_new;
      }
      la = fadd2(la, ta);
      lb = fadd2(lb, tb);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s_free[qi]);                      // the tensor core may overwrite S now
      mbar_arrive(&p_full[qi]);
    }
    if (n > 0 && qi < nq_tiles) {
      // Epilogue: combine the two warps' row sums, then each warp normalises
      // and writes its half of the head dimension.
      bool good = ok && wait_bar_warp(g, &p_free[qi], (n - 1) & 1, 9);
      const float l_mine = (f2_lo(la) + f2_hi(la)) + (f2_lo(lb) + f2_hi(lb));
      float* my_slot = mine + (n & 1) * 33;
      float* their_slot = theirs + (n & 1) * 33;
      my_slot[lane] = l_mine;
      if (lane == 0) my_slot[32] = __int_as_float(good ? 0 : 2);
      if (ok) pair_sync(bar_id, 64);                 // both warps of a pair left the loop alike
      if (ok && good && !(__float_as_int(their_slot[32]) & 2)) {
        const float l = l_mine + their_slot[lane];
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(O_ + half * 32, v);
        tmem_wait_ld();
        reg_fence(v);
        const int row = q0 + qi * BM + r;
        if (row < a.n_q) {
          const float inv = 1.f / l;
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]) * inv;
          if (a.n_splits == 1) {
            using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.out) +
                                                  ((int64_t)row * a.num_heads + h) * HD + half * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 u;
              u.x = pack2<BF16>(o[8 * i + 0], o[8 * i + 1]);
              u.y = pack2<BF16>(o[8 * i + 2], o[8 * i + 3]);
              u.z = pack2<BF16>(o[8 * i + 4], o[8 * i + 5]);
              u.w = pack2<BF16>(o[8 * i + 6], o[8 * i + 7]);
              dst[i] = u;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(
                a.part_o + (((int64_t)split * a.n_q + row) * a.num_heads + h) * HD + half * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            if (half == 0) a.part_lse[((int64_t)split * a.n_q + row) * a.num_heads + h] = m_ref + __log2f(l);
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

bool configured_smem[2] = {false, false};

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
  CUresult r = enc(&m->cache, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   cache, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    delete m;
    if (err) *err = cudaErrorInvalidValue;
    return nullptr;
  }
  return m;
}

void tc_destroy_maps(TcMaps* m) { delete m; }

cudaError_t launch_attn_tc(const AttnArgs& a, TcMaps* maps, int block, int max_pages, int dtype,
                           cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !maps || a.head_dim != HD) return cudaErrorNotSupported;
  CUtensorMap qmap;
  const cuuint64_t row_bytes = (cuuint64_t)a.num_heads * HD * 2;
  cuuint64_t dims[2] = {(cuuint64_t)a.num_heads * HD, (cuuint64_t)a.n_q};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {HD, BM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&qmap, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(a.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  dim3 grid((a.n_q + QT * BM - 1) / (QT * BM), a.num_heads, a.n_splits);
  const int page_base = block * max_pages;
  if (dtype == 0) {
    if (!configured_smem[0]) {
      cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      configured_smem[0] = true;
    }
    attn_tc_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(a, maps->cache, qmap, page_base);
  } else {
    if (!configured_smem[1]) {
      cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
      configured_smem[1] = true;
    }
    attn_tc_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(a, maps->cache, qmap, page_base);
  }
  return cudaGetLastError();
}

}  // namespace kvc
