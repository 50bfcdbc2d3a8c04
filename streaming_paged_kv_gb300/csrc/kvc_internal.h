// Internal interfaces between the host bookkeeping (kvc_host.cpp) and the
// CUDA kernels (kvc_kernels.cu, kvc_attn_tc.cu).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvc {

constexpr int kNumSpecial = 6;
constexpr int kMaxPatchPages = 1024;   // bound on P (the patch pool), kernel-argument sized

// Device plan written by the plan kernel into the workspace.
struct DevPlanHeader {
  int32_t n_pages;
  int32_t last_page_len;
  int32_t n_tiles;
  int32_t n_tokens;
};

// One KV tile of a visible page: rows [row0, row0 + rows) of page `page`.
struct KvTile {
  int32_t page;
  int32_t row0;
  int32_t rows;
  int32_t token0;  // position of the tile's first token in the visible sequence
};

// Workspace layout (byte offsets from the workspace base).
struct WorkspaceLayout {
  size_t status;       // int32[64]: [0] error flag, [1] where, [2] cta
  size_t header;       // DevPlanHeader
  size_t page_ids;     // int32[max_pages]
  size_t page_valid;   // int32[max_pages]
  size_t tiles;        // KvTile[max_tiles]
  size_t part_o;       // float[max_splits][max_q][H][D]
  size_t part_lse;     // float[max_splits][max_q][H]
  size_t total;
  int32_t max_pages;
  int32_t max_tiles;
};

// Arguments of the plan kernel, passed by value (no host->device copy).
struct PlanArgs {
  int32_t n_patch;                  // visible patch pages (scale + live)
  int32_t n_special;                // visible special pages
  int32_t first_special;            // page id of the first special page (= P)
  int32_t full_special_len;         // valid tokens of a non-last special page (6*fpp)
  int32_t last_page_len;            // valid tokens of the last special page
  int32_t page_size;
  int32_t tile_rows;                // rows per KV tile of the attention kernel
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
  float sm_scale_log2;    // sm_scale * log2(e)
  long long wait_budget;  // clock cycles per bounded wait
  int32_t stall_test;     // 1: wait once on a barrier nothing signals (timeout test)
};

// kvc_kernels.cu
cudaError_t launch_append(void* cache_block, const void* K, const void* V, int32_t page,
                          int32_t special_page, int32_t special_slot, int32_t page_size,
                          int64_t row_bytes, cudaStream_t stream);
cudaError_t launch_plan(const PlanArgs& a, void* workspace, const WorkspaceLayout& L,
                        cudaStream_t stream);
cudaError_t launch_attn_simt(const AttnArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_merge(const AttnArgs& a, int dtype, cudaStream_t stream);
int simt_tile_rows(int head_dim);

// kvc_attn_tc.cu
bool tc_supported(int dtype, int head_dim, int num_heads, int page_size);
constexpr int kTcTileRows = 128;
constexpr int kTcQRows = 256;   // query rows per CTA of the tensor-core kernel
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
  int32_t block, max_pages;
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
  float sm_scale_log2;
  long long wait_budget;
  TcRequestDesc req[kTcMaxBatch];
};
cudaError_t launch_attn_tc(const TcBatchArgs& b, cudaStream_t stream);

}  // namespace kvc
