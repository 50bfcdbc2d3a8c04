// Internal interfaces between the host bookkeeping (kvc_host.cpp) and the
// CUDA kernels (kvc_kernels.cu, kvc_attn_tc.cu).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#ifdef __CUDACC__
#define KVC_HD __host__ __device__
#else
#define KVC_HD
#endif

// KVC_CHECKED=1 builds (a separate library, libkvc_checked.so) add device-side
// bounds checks on page ids, slots, tile rows and TMA coordinates; a failed
// check records kStatusBounds, where and the bad value in the status word and
// skips the access -- it never traps.
#ifndef KVC_CHECKED
#define KVC_CHECKED 0
#endif

namespace kvc {

constexpr int kNumSpecial = 6;
constexpr int32_t kStatusTimeout = 1;   // status[0]: a bounded wait ran out
constexpr int32_t kStatusBounds = 2;    // status[0]: a bounds check failed (checked builds)

#ifdef __CUDACC__
// First failure wins: status = {code, where, value}.
__device__ inline void record_bounds(int32_t* status, int32_t where, int32_t value) {
  if (atomicCAS(status, 0, kStatusBounds) == 0) {
    status[1] = where;
    status[2] = value;
  }
  __threadfence();
}
#endif
#ifdef __CUDACC__
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream drains:
// pdl_wait() returns once that kernel has completed and its memory operations
// are visible (at once for a kernel launched the ordinary way), and
// pdl_trigger() lets the next kernel of the stream be launched early.  Every
// kernel of the library calls pdl_wait() before it touches global memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` on `st`, with programmatic stream serialization when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

constexpr int kMaxPatchPages = 1024;   // bound on P (the patch pool), kernel-argument sized

// Device plan written by the plan kernel into the workspace.
struct DevPlanHeader {
  int32_t n_pages;
  int32_t last_page_len;
  int32_t n_tiles;
  int32_t n_tokens;
};

// One KV tile: rows [row0, row0 + rows) of page `page`, and in a packed tile
// (tensor-core plans, page2 >= 0) rows [row0_2, row0_2 + rows2) of page2 after
// them, from tile row ceil(rows / 8) * 8 on; rows2 = 0 and page2 = -1 otherwise.
struct alignas(16) KvTile {
  int32_t page;
  int32_t row0;
  int32_t rows;
  int32_t rows2;   // next to rows: the softmax reads both with one 8-byte load
  int32_t page2;
  int32_t row0_2;
  int32_t token0;  // position of the tile's first token in the visible sequence
  int32_t pad;
};
static_assert(sizeof(KvTile) == 32, "KvTile layout");

// Packed tiles are built from units of 8 rows (the 128-byte swizzle atom of a
// 64-wide bf16 row): a visible entry of v rows takes ceil(v / 8) units, and
// tile t covers units [16 t, 16 t + 16) of the concatenated entries.  A tile
// then spans at most two entries when every entry but the last has at least
// kPackMinUnits units.
constexpr int kPackUnitRows = 8;
constexpr int kPackMinUnits = 15;

// Workspace layout (byte offsets from the workspace base).
struct WorkspaceLayout {
  size_t status;       // int32[64]: [0] error flag, [1] where, [2] cta
  size_t header;       // DevPlanHeader
  size_t page_ids;     // int32[max_pages]
  size_t page_valid;   // int32[max_pages]
  size_t page_row0;    // int32[max_pages]: first visible row of each visible page
  size_t tiles;        // KvTile[max_tiles]
  size_t part_o;       // float[max_splits][max_q][H][D]
  size_t part_lse;     // float[max_splits][max_q][H]
  size_t total;
  int32_t max_pages;
  int32_t max_tiles;
};

// A run of consecutive positions [a, b) of an append-only stream whose page
// p (id page0 + p) holds positions [p * per_page, (p + 1) * per_page), `tok`
// rows each: the special stream (6 rows per frame) or the camera stream (one
// row per frame).  A run covers pages floor(a / per_page) ..
// ceil(b / per_page) - 1; its first and last page may be partial.
struct PlanRun {
  int32_t page0, per_page, tok, a, b;
};

KVC_HD inline int32_t run_pages(const PlanRun& r) {
  return r.b > r.a ? (r.b + r.per_page - 1) / r.per_page - r.a / r.per_page : 0;
}
// Page id, first row and row count of page e of the run.
KVC_HD inline void run_entry(const PlanRun& r, int32_t e, int32_t* page, int32_t* row0, int32_t* rows) {
  const int32_t p = r.a / r.per_page + e;
  const int32_t lo = r.a > p * r.per_page ? r.a : p * r.per_page;
  const int32_t hi = r.b < (p + 1) * r.per_page ? r.b : (p + 1) * r.per_page;
  *page = r.page0 + p;
  *row0 = r.tok * (lo - p * r.per_page);
  *rows = r.tok * (hi - lo);
}

constexpr int kMaxRuns = 3;

// Arguments of the plan kernel, passed by value (no host->device copy).
// Visible entries: the n_patch patch pages (all rows), then every page of
// each run in order.
struct PlanArgs {
  int32_t n_patch;                  // visible patch pages (scale + live)
  int32_t n_runs;                   // special / camera runs
  PlanRun runs[kMaxRuns];
  int32_t page_size;
  int32_t tile_rows;                // rows per KV tile of the attention kernel
  int32_t pack;                     // 1: packed tiles of tile_rows rows in 8-row units
  int32_t max_pages;                // pages of one block's cache (bounds checks)
  int32_t patch_ids[kMaxPatchPages];
};

struct AttnArgs {
  const void* q;          // [n_q, H, D]
  void* out;              // [n_q, H, D]
  const void* cache;      // block base: [max_pages][2][ps][H][D]
  const KvTile* tiles;
  float* part_o;          // [splits][n_q][H][D]
  float* part_lse;        // [splits][n_q][H], log2 domain
  int32_t* status;
  int32_t n_q;
  int32_t num_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t n_tiles;
  int32_t n_splits;
  int32_t max_pages;      // pages of one block's cache (bounds checks)
  float sm_scale_log2;    // sm_scale * log2(e)
  long long wait_budget;  // clock cycles per bounded wait
  int32_t stall_test;     // 1: wait once on a barrier nothing signals (timeout test)
  int32_t pdl;            // launch with programmatic stream serialization
};

// kvc_kernels.cu
cudaError_t launch_append(void* cache_block, const void* K, const void* V, int32_t page,
                          int32_t special_page, int32_t special_slot, int32_t camera_page,
                          int32_t camera_slot, int32_t page_size, int64_t row_bytes, int32_t max_pages,
                          int32_t* status, cudaStream_t stream, bool pdl);
cudaError_t launch_plan(const PlanArgs& a, void* workspace, const WorkspaceLayout& L,
                        cudaStream_t stream, bool pdl);
cudaError_t launch_attn_simt(const AttnArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_merge(const AttnArgs& a, int dtype, cudaStream_t stream);
int simt_tile_rows(int head_dim);

// kvc_attn_tc.cu
bool tc_supported(int dtype, int head_dim, int num_heads, int page_size);
constexpr int kTcTileRows = 128;
constexpr int kTcQRows = 256;   // most query rows per CTA of the tensor-core kernel
struct TcMaps;   // opaque: TMA descriptors of the cache (per handle)
TcMaps* tc_create_maps(void* cache, int dtype, int num_blocks, int max_pages, int page_size,
                       int num_heads, int head_dim, cudaError_t* err);
void tc_destroy_maps(TcMaps* m);
// One tensor-core launch over up to kTcMaxBatch requests (independent streams,
// each with its own cache, plan and partials).  Q and out are one ragged
// tensor [rows, H, D]; request r owns rows [q_row0, q_row0 + n_q).
constexpr int kTcMaxBatch = 16;
struct TcRequestDesc {
  TcMaps* maps;
  int32_t block, max_pages, page_size;
  const KvTile* tiles;
  float* part_o;          // [n_splits][n_q][H][D] (n_splits > 1)
  float* part_lse;        // [n_splits][n_q][H]
  int32_t* status;
  int32_t n_tiles, n_splits, q_row0, n_q;
};
struct TcBatchArgs {
  const void* q;
  void* out;
  int32_t rows, num_heads, head_dim, dtype, stall_test, count;
  int32_t num_sms;        // of the device: decides whether a launch has several waves
  int32_t q_tiles;        // 128-row query tiles per CTA: 2, or 1 (both softmax groups on one tile)
  int32_t pdl;            // launch with programmatic stream serialization
  float sm_scale_log2;
  long long wait_budget;
  TcRequestDesc req[kTcMaxBatch];
};
cudaError_t launch_attn_tc(const TcBatchArgs& b, cudaStream_t stream);

}  // namespace kvc
