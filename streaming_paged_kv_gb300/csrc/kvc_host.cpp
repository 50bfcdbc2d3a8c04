// Host side of libkvc.so: the page allocator (scale / live / free deques of
// patch page IDs per block), the special-stream counters, the undo stack for
// rollback, plan construction and the C ABI declared in include/kvc.h.
//
// Pages cited by tag, then section:
//   [KVC]   "How LingBot-Map Implements the KV Cache Mechanism for Streaming
//           Inference with FlashInfer Integration"
//   [PERF]  "How to Improve Streaming Inference Performance with FlashInfer KV
//           Cache Backend"
//   [SLOTS] "LingBot-Map KV缓存机制深度揭秘：scale frames与keyframes如何占用slot"
//
// Every buffer the handle uses is allocated in kvc_create; no call after it
// allocates host or device memory ([PERF] "Two-Stream Page Pool
// Architecture": pages only move between deques after construction).

#include "kvc.h"
#include "kvc_internal.h"

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

using kvc::kNumSpecial;

namespace {

// Fixed-capacity ring deque of page IDs.
struct Ring {
  int32_t* buf = nullptr;
  int32_t cap = 0, head = 0, size = 0;
  void bind(int32_t* storage, int32_t c) { buf = storage; cap = c; head = 0; size = 0; }
  void clear() { head = 0; size = 0; }
  int32_t at(int32_t i) const { return buf[(head + i) % cap]; }
  int32_t back() const { return buf[(head + size - 1) % cap]; }
  void push_back(int32_t v) { buf[(head + size) % cap] = v; ++size; }
  void push_front(int32_t v) { head = (head + cap - 1) % cap; buf[head] = v; ++size; }
  int32_t pop_front() { int32_t v = buf[head]; head = (head + 1) % cap; --size; return v; }
  int32_t pop_back() { int32_t v = back(); --size; return v; }
};

struct Undo {
  int32_t page;
  int32_t to_scale;
};

struct Block {
  Ring scale, live, free_list;
  int32_t special_frames = 0;  // frames in the special stream
  int32_t frame_count = 0;
  Undo* undo = nullptr;        // uncommitted appends, newest last
  int32_t n_undo = 0;

  // Construction state: all patch pages free, in ID order.
  void reset(int32_t P) {
    scale.clear();
    live.clear();
    free_list.clear();
    for (int32_t i = 0; i < P; ++i) free_list.push_back(i);
    special_frames = 0;
    frame_count = 0;
    n_undo = 0;
  }
};

constexpr int kEventPairs = 4096;
constexpr int kDefaultSplits = 32;

int64_t elem_bytes(int dtype) { return dtype == KVC_F32 ? 4 : 2; }

// Validate cfg and fill defaults.  Returns KVC_OK or INVALID_ARG.
int resolve(const kvc_config* in, kvc_config* out) {
  if (!in || !out) return KVC_ERR_INVALID_ARG;
  kvc_config c = *in;
  if (c.num_special_tokens == 0) c.num_special_tokens = kNumSpecial;
  if (c.max_kv_splits == 0) c.max_kv_splits = kDefaultSplits;
  if (c.max_query_tokens == 0) c.max_query_tokens = kNumSpecial + c.page_size;
  if (c.sm_scale == 0.0f && c.head_dim > 0) c.sm_scale = 1.0f / std::sqrt((float)c.head_dim);
  if (c.num_blocks < 1 || c.num_heads < 1 || c.num_heads > 4096) return KVC_ERR_INVALID_ARG;
  if (c.head_dim != 32 && c.head_dim != 64 && c.head_dim != 128) return KVC_ERR_INVALID_ARG;
  if (c.dtype < KVC_BF16 || c.dtype > KVC_F32) return KVC_ERR_INVALID_ARG;
  if (c.num_special_tokens != kNumSpecial) return KVC_ERR_INVALID_ARG;
  if (c.page_size < kNumSpecial || c.page_size > (1 << 16)) return KVC_ERR_INVALID_ARG;
  if (c.scale_frames < 0 || c.sliding_window < 0 || c.headroom < 0) return KVC_ERR_INVALID_ARG;
  int64_t P = (int64_t)c.scale_frames + c.sliding_window + c.headroom;
  if (P < 1 || P > kvc::kMaxPatchPages) return KVC_ERR_INVALID_ARG;
  if (c.max_total_frames < 1 || c.max_total_frames > (1 << 24)) return KVC_ERR_INVALID_ARG;
  if (c.max_query_tokens < 1 || c.max_query_tokens > (1 << 20)) return KVC_ERR_INVALID_ARG;
  if (c.max_kv_splits < 1 || c.max_kv_splits > 256) return KVC_ERR_INVALID_ARG;
  if (!(c.sm_scale > 0.0f) || !std::isfinite(c.sm_scale)) return KVC_ERR_INVALID_ARG;
  if (((int64_t)c.num_heads * c.head_dim * elem_bytes(c.dtype)) % 16 != 0) return KVC_ERR_INVALID_ARG;
  if (c.special_policy < 0 || c.special_policy > (KVC_SPECIAL_NO_CROSS_FRAME | KVC_SPECIAL_CAMERA_ONLY))
    return KVC_ERR_INVALID_ARG;
  *out = c;
  return KVC_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Evicted frames keep only their camera token visible (needs the camera stream).
bool camera_stream(const kvc_config& c) { return c.special_policy == KVC_SPECIAL_CAMERA_ONLY; }
bool cross_frame(const kvc_config& c) { return (c.special_policy & KVC_SPECIAL_NO_CROSS_FRAME) == 0; }

struct Geometry {
  int32_t P, fpp, n_special_pages, n_camera_pages, first_camera, max_pages, max_entries, T;
  int64_t row_bytes, page_bytes, block_bytes;
  size_t cache_bytes;
  kvc::WorkspaceLayout L;
};

void geometry(const kvc_config& c, Geometry* g) {
  g->P = c.scale_frames + c.sliding_window + c.headroom;
  g->fpp = c.page_size / kNumSpecial;                      // floor(page_size / 6)
  g->n_special_pages = (c.max_total_frames + g->fpp - 1) / g->fpp;
  // Camera stream: page_size camera tokens per page, after the special pages.
  g->n_camera_pages = camera_stream(c) ? (c.max_total_frames + c.page_size - 1) / c.page_size : 0;
  g->first_camera = g->P + g->n_special_pages;
  g->max_pages = g->P + g->n_special_pages + g->n_camera_pages;
  // Visible entries: every page at most once, except that the two special
  // runs of a policy without cross-frame specials may share a page each end.
  g->max_entries = g->max_pages + 2;
  g->T = kNumSpecial + c.page_size;
  g->row_bytes = (int64_t)c.num_heads * c.head_dim * elem_bytes(c.dtype);
  g->page_bytes = 2 * (int64_t)c.page_size * g->row_bytes;  // K and V of one page
  g->block_bytes = (int64_t)g->max_pages * g->page_bytes;
  g->cache_bytes = (size_t)g->block_bytes * c.num_blocks;
  // The smallest tile any attention kernel uses bounds the tile count.
  const int min_rows = 32;
  int64_t max_tiles = (int64_t)g->max_entries * ((c.page_size + min_rows - 1) / min_rows);
  kvc::WorkspaceLayout& L = g->L;
  size_t off = 0;
  L.status = off;   off += 256;
  L.header = off;   off += 256;
  L.page_ids = off; off = align_up(off + 4 * (size_t)g->max_entries, 256);
  L.page_valid = off; off = align_up(off + 4 * (size_t)g->max_entries, 256);
  L.page_row0 = off; off = align_up(off + 4 * (size_t)g->max_entries, 256);
  L.tiles = off;    off = align_up(off + sizeof(kvc::KvTile) * (size_t)max_tiles, 256);
  L.part_o = off;
  off = align_up(off + 4 * (size_t)c.max_kv_splits * c.max_query_tokens * c.num_heads * c.head_dim, 256);
  L.part_lse = off;
  off = align_up(off + 4 * (size_t)c.max_kv_splits * c.max_query_tokens * c.num_heads, 256);
  L.total = off;
  L.max_pages = g->max_entries;
  L.max_tiles = (int32_t)max_tiles;
}

}  // namespace

struct kvc_handle {
  kvc_config cfg;
  Geometry g;
  char* cache = nullptr;      // borrowed device buffers
  char* ws = nullptr;
  bool device = false;
  int num_sms = 0;
  Block* blocks = nullptr;
  int32_t* ring_storage = nullptr;
  Undo* undo_storage = nullptr;
  bool defer = false;
  // Plan (host copy + the state it was made from).
  bool has_plan = false;
  int32_t plan_n_pages = 0, plan_lpl = 0, plan_n_tiles = 0, plan_tile_rows = 0, plan_kernel = 0;
  bool plan_packed = false;
  int32_t plan_n_scale = 0, plan_n_live = 0, plan_special_frames = 0;
  int32_t* plan_ids = nullptr;      // [max_entries]
  int32_t* plan_row0 = nullptr;     // [max_entries]
  int32_t* plan_valid = nullptr;    // [max_entries]
  int32_t* plan_snapshot = nullptr; // [P]: scale then live
  kvc::PlanArgs* plan_args = nullptr;
  // Options.
  int opt_kernel = 0;
  int opt_splits = 0;
  int opt_qtiles = 0;
  bool opt_pack = true;
  bool opt_pdl = true;
  long long wait_budget = 0;
  bool timing = false;
  int32_t timing_every = 1;         // time one attention launch in every timing_every
  int64_t timing_count = 0;         // attention launches since timing was set
  int stall_test = 0;
  // Counters.
  int64_t launches = 0, attn_launches = 0;
  int32_t last_qt = 0, last_splits = 0;   // shape of the latest attention launch (0: CUDA-core kernel)
  double attn_ms = 0.0;
  cudaEvent_t* ev = nullptr;        // [2 * kEventPairs] when timing
  bool* ev_used = nullptr;
  int ev_next = 0;
  kvc::TcMaps* maps = nullptr;
};

namespace {

// NVTX range over a call (header-only NVTX 3: costs nothing unless a
// profiler is attached), so that timelines show append / plan / run.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

int check_block(const kvc_handle* h, int32_t block) {
  if (!h || block < 0 || block >= h->cfg.num_blocks) return KVC_ERR_INVALID_ARG;
  return KVC_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Move live pages to the free list until at most `window` remain; an eviction
// that moves a page commits the block's pending frames.
int32_t evict_to(Block& b, int32_t window, bool commit_always) {
  int32_t moved = 0;
  while (b.live.size > window) {
    b.free_list.push_back(b.live.pop_front());
    ++moved;
  }
  if (moved || commit_always) b.n_undo = 0;
  return moved;
}

int attn_kernel_for(const kvc_handle* h) {
  const kvc_config& c = h->cfg;
  bool tc = h->maps != nullptr && kvc::tc_supported(c.dtype, c.head_dim, c.num_heads, c.page_size);
  if (h->opt_kernel == 1) return 1;
  if (h->opt_kernel == 2) return tc ? 2 : -1;
  return tc ? 2 : 1;
}

// Launch shape of an attention launch: 128-row query tiles per CTA of the
// tensor-core kernel and the number of KV splits.
struct Shape {
  int qt, splits;
};

// Cost model of the tensor-core kernel in microseconds, fitted to GB300
// measurements at 518x378 full context (one CTA per SM; CTAs run in waves):
// a CTA costs fixed + tiles * per_tile, with per_tile 0.985 us and fixed
// 6.2 us for two query tiles per CTA, 0.522 us and 4.9 us for one (both
// softmax groups on it); the merge reads splits * rows * H * (D + 1) fp32 at
// about 5 TB/s after a 2 us launch.  base_ctas(qt) = CTAs of one split.
double tc_cost_us(int qt, int s, int64_t base_ctas, int64_t max_tiles, int64_t merge_elems, int num_sms) {
  const double per_tile = qt == 2 ? 0.985 : 0.522, fixed = qt == 2 ? 6.2 : 4.9;
  const int64_t sms = num_sms > 0 ? num_sms : 1;
  const int64_t waves = (base_ctas * s + sms - 1) / sms;
  const double cta = fixed + per_tile * (double)((max_tiles + s - 1) / s);
  const double merge = s > 1 ? 2.0 + (double)s * (double)merge_elems * 4.0 / 5.0e6 : 0.0;
  return (double)waves * cta + merge;
}

// Best shape over qt in {2, 1} and splits in [1, max_s]; one tile per CTA
// must win by 3% (the model is a fit).  rows_blocks(qt) = sum over requests of
// ceil(n_q / (128 qt)).  Options force either choice.
Shape choose_tc_shape(const kvc_handle* h, int max_s, int64_t blocks2, int64_t blocks1, int64_t max_tiles,
                      int64_t rows_total) {
  const int64_t H = h->cfg.num_heads;
  const int64_t merge_elems = rows_total * H * (h->cfg.head_dim + 1);
  Shape best{2, 1};
  double best_cost = 1e300;
  for (int qt = 2; qt >= 1; --qt) {
    if (h->opt_qtiles > 0 && qt != h->opt_qtiles) continue;
    const int64_t base = (qt == 2 ? blocks2 : blocks1) * H;
    for (int sp = 1; sp <= max_s; ++sp) {
      if (h->opt_splits > 0 && sp != (h->opt_splits < max_s ? h->opt_splits : max_s)) continue;
      double c = tc_cost_us(qt, sp, base, max_tiles, merge_elems, h->num_sms);
      if (qt == 1) c *= 1.03;
      if (c < best_cost - 1e-9) { best_cost = c; best = Shape{qt, sp}; }
    }
  }
  return best;
}

int tile_rows_for(const kvc_handle* h, int kernel) {
  return kernel == 2 ? kvc::kTcTileRows : kvc::simt_tile_rows(h->cfg.head_dim);
}

// Launch shape of one request.  Tensor-core kernel: the cost model above.
// CUDA-core kernel (128-row query blocks, two CTAs per SM): balance waves of
// CTAs against work per split, with a small charge per split for the merge.
Shape choose_shape(const kvc_handle* h, int kernel, int32_t n_q) {
  int max_s = h->cfg.max_kv_splits;
  if (max_s > h->plan_n_tiles) max_s = h->plan_n_tiles;
  if (max_s < 1) max_s = 1;
  if (kernel == 2)
    return choose_tc_shape(h, max_s, (n_q + 255) / 256, (n_q + 127) / 128, h->plan_n_tiles, n_q);
  if (h->opt_splits > 0) return Shape{1, h->opt_splits < max_s ? h->opt_splits : max_s};
  int64_t base = (int64_t)((n_q + 127) / 128) * h->cfg.num_heads;
  int64_t slots = (int64_t)h->num_sms * 2;
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= max_s; ++s) {
    int64_t waves = (base * s + slots - 1) / slots;
    int64_t per = (h->plan_n_tiles + s - 1) / s;
    double cost = (double)waves * per * (1.0 + (s > 1 ? 0.02 * s : 0.0));
    if (cost < best - 1e-9) { best = cost; best_s = s; }
  }
  return Shape{1, best_s};
}

// Whether the attention launch about to be made is a timed one: with timing
// set to N, the (N / 2)-th launch of every group of N since it was set.
bool timed_launch(kvc_handle* h) {
  if (!h->timing) return false;
  const int64_t i = h->timing_count++;
  return i % h->timing_every == h->timing_every / 2;
}

void record_timing(kvc_handle* h, int which, cudaStream_t st) {
  // which 0: start, 1: stop of the current pair.
  int i = h->ev_next;
  if (which == 0 && h->ev_used[i]) {
    float ms = 0.f;
    cudaEventSynchronize(h->ev[2 * i + 1]);
    if (cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]) == cudaSuccess)
      h->attn_ms += (double)ms * h->timing_every;
    h->ev_used[i] = false;
  }
  cudaEventRecord(h->ev[2 * i + which], st);
  if (which == 1) {
    h->ev_used[i] = true;
    h->ev_next = (i + 1) % kEventPairs;
  }
}

void drain_timing(kvc_handle* h) {
  if (!h->ev) return;
  for (int i = 0; i < kEventPairs; ++i) {
    if (!h->ev_used[i]) continue;
    float ms = 0.f;
    cudaEventSynchronize(h->ev[2 * i + 1]);
    if (cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]) == cudaSuccess)
      h->attn_ms += (double)ms * h->timing_every;
    h->ev_used[i] = false;
  }
}

}  // namespace

// Preconditions of a run: a device handle, a plan, this block's pages equal
// to the planned ones, n_q within limits, aligned buffers.
int check_run(const kvc_handle* h, int32_t block, const void* Q, const void* out, int32_t n_q) {
  int rc = check_block(h, block);
  if (rc) return rc;
  if (!h->device) return KVC_ERR_NO_DEVICE;
  if (!h->has_plan) return KVC_ERR_NO_PLAN;
  if (n_q < 0 || n_q > h->cfg.max_query_tokens) return KVC_ERR_INVALID_ARG;
  if (n_q > 0 && (!Q || !out || !aligned16(Q) || !aligned16(out))) return KVC_ERR_INVALID_ARG;
  // The plan is valid for this block only if its pages are the planned ones.
  const Block& b = h->blocks[block];
  if (b.scale.size != h->plan_n_scale || b.live.size != h->plan_n_live ||
      b.special_frames != h->plan_special_frames)
    return KVC_ERR_STALE_PLAN;
  for (int32_t i = 0; i < b.scale.size; ++i)
    if (b.scale.at(i) != h->plan_snapshot[i]) return KVC_ERR_STALE_PLAN;
  for (int32_t i = 0; i < b.live.size; ++i)
    if (b.live.at(i) != h->plan_snapshot[b.scale.size + i]) return KVC_ERR_STALE_PLAN;
  return KVC_OK;
}

kvc::AttnArgs attn_args(const kvc_handle* h, int32_t block, const void* Q, void* out, int32_t n_q, int splits) {
  kvc::AttnArgs a;
  a.pdl = h->opt_pdl ? 1 : 0;
  a.q = Q;
  a.out = out;
  a.cache = h->cache + (size_t)block * h->g.block_bytes;
  a.tiles = (const kvc::KvTile*)(h->ws + h->g.L.tiles);
  a.part_o = (float*)(h->ws + h->g.L.part_o);
  a.part_lse = (float*)(h->ws + h->g.L.part_lse);
  a.status = (int32_t*)(h->ws + h->g.L.status);
  a.n_q = n_q;
  a.num_heads = h->cfg.num_heads;
  a.head_dim = h->cfg.head_dim;
  a.page_size = h->cfg.page_size;
  a.n_tiles = h->plan_n_tiles;
  a.n_splits = splits;
  a.max_pages = h->g.max_pages;
  a.sm_scale_log2 = h->cfg.sm_scale * 1.4426950408889634f;
  a.wait_budget = h->wait_budget > 0 ? h->wait_budget : 4000000000LL;
  a.stall_test = h->stall_test;
  return a;
}

kvc::TcBatchArgs tc_batch_header(const kvc_handle* h, const void* Q, void* out, int32_t rows) {
  kvc::TcBatchArgs tb;
  std::memset(&tb, 0, sizeof(tb));
  tb.pdl = h->opt_pdl ? 1 : 0;
  tb.q = Q;
  tb.out = out;
  tb.rows = rows;
  tb.num_heads = h->cfg.num_heads;
  tb.head_dim = h->cfg.head_dim;
  tb.dtype = h->cfg.dtype;
  tb.stall_test = h->stall_test;
  tb.num_sms = h->num_sms;
  tb.q_tiles = 2;
  tb.sm_scale_log2 = h->cfg.sm_scale * 1.4426950408889634f;
  tb.wait_budget = h->wait_budget > 0 ? h->wait_budget : 4000000000LL;
  return tb;
}

kvc::TcRequestDesc tc_request(const kvc_handle* h, int32_t block, int32_t q_row0, int32_t n_q, int splits) {
  kvc::TcRequestDesc d;
  d.maps = h->maps;
  d.block = block;
  d.max_pages = h->g.max_pages;
  d.page_size = h->cfg.page_size;
  d.tiles = (const kvc::KvTile*)(h->ws + h->g.L.tiles);
  d.part_o = (float*)(h->ws + h->g.L.part_o);
  d.part_lse = (float*)(h->ws + h->g.L.part_lse);
  d.status = (int32_t*)(h->ws + h->g.L.status);
  d.n_tiles = h->plan_n_tiles;
  d.n_splits = splits;
  d.q_row0 = q_row0;
  d.n_q = n_q;
  return d;
}

extern "C" {

int kvc_get_geometry(const kvc_config* cfg, kvc_geometry* out) {
  kvc_config c;
  int rc = resolve(cfg, &c);
  if (rc) return rc;
  if (!out) return KVC_ERR_INVALID_ARG;
  Geometry g;
  geometry(c, &g);
  out->num_patch_pages = g.P;
  out->frames_per_special_page = g.fpp;
  out->num_special_pages = g.n_special_pages;
  out->num_camera_pages = g.n_camera_pages;
  out->max_num_pages = g.max_pages;
  out->tokens_per_frame = g.T;
  out->page_bytes = g.page_bytes;
  out->block_bytes = g.block_bytes;
  return KVC_OK;
}

int kvc_required_bytes(const kvc_config* cfg, size_t* cache_bytes, size_t* workspace_bytes) {
  kvc_config c;
  int rc = resolve(cfg, &c);
  if (rc) return rc;
  Geometry g;
  geometry(c, &g);
  if (cache_bytes) *cache_bytes = g.cache_bytes;
  if (workspace_bytes) *workspace_bytes = g.L.total;
  return KVC_OK;
}

int kvc_create(const kvc_config* cfg, void* cache_dev, void* workspace_dev, kvc_stream stream,
               kvc_handle** out) {
  if (!out) return KVC_ERR_INVALID_ARG;
  *out = nullptr;
  kvc_config c;
  int rc = resolve(cfg, &c);
  if (rc) return rc;
  if ((cache_dev == nullptr) != (workspace_dev == nullptr)) return KVC_ERR_INVALID_ARG;
  if (((uintptr_t)cache_dev & 255u) || ((uintptr_t)workspace_dev & 255u)) return KVC_ERR_INVALID_ARG;
  kvc_handle* h = new (std::nothrow) kvc_handle();
  if (!h) return KVC_ERR_INVALID_ARG;
  h->cfg = c;
  geometry(c, &h->g);
  const int32_t P = h->g.P;
  h->blocks = new (std::nothrow) Block[c.num_blocks];
  h->ring_storage = (int32_t*)std::calloc((size_t)c.num_blocks * 3 * P, sizeof(int32_t));
  h->undo_storage = (Undo*)std::calloc((size_t)c.num_blocks * P, sizeof(Undo));
  h->plan_ids = (int32_t*)std::calloc((size_t)h->g.max_entries, sizeof(int32_t));
  h->plan_row0 = (int32_t*)std::calloc((size_t)h->g.max_entries, sizeof(int32_t));
  h->plan_valid = (int32_t*)std::calloc((size_t)h->g.max_entries, sizeof(int32_t));
  h->plan_snapshot = (int32_t*)std::calloc((size_t)P, sizeof(int32_t));
  h->plan_args = (kvc::PlanArgs*)std::calloc(1, sizeof(kvc::PlanArgs));
  if (!h->blocks || !h->ring_storage || !h->undo_storage || !h->plan_ids || !h->plan_row0 ||
      !h->plan_valid || !h->plan_snapshot || !h->plan_args) {
    kvc_destroy(h);
    return KVC_ERR_INVALID_ARG;
  }
  for (int b = 0; b < c.num_blocks; ++b) {
    Block& B = h->blocks[b];
    int32_t* base = h->ring_storage + (size_t)b * 3 * P;
    B.scale.bind(base, P);
    B.live.bind(base + P, P);
    B.free_list.bind(base + 2 * P, P);
    B.undo = h->undo_storage + (size_t)b * P;
    B.reset(P);
  }
  if (cache_dev) {
    h->device = true;
    h->cache = (char*)cache_dev;
    h->ws = (char*)workspace_dev;
    int dev = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaMemsetAsync(h->cache, 0, h->g.cache_bytes, st) != cudaSuccess ||
        cudaMemsetAsync(h->ws, 0, h->g.L.part_o, st) != cudaSuccess) {
      kvc_destroy(h);
      return KVC_ERR_CUDA;
    }
    if (kvc::tc_supported(c.dtype, c.head_dim, c.num_heads, c.page_size)) {
      cudaError_t err = cudaSuccess;
      h->maps = kvc::tc_create_maps(h->cache, c.dtype, c.num_blocks, h->g.max_pages, c.page_size,
                                    c.num_heads, c.head_dim, &err);
      if (!h->maps) {
        kvc_destroy(h);
        return KVC_ERR_CUDA;
      }
    }
  }
  *out = h;
  return KVC_OK;
}

int kvc_destroy(kvc_handle* h) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (h->ev) {
    for (int i = 0; i < 2 * kEventPairs; ++i)
      if (h->ev[i]) cudaEventDestroy(h->ev[i]);
    std::free(h->ev);
  }
  std::free(h->ev_used);
  if (h->maps) kvc::tc_destroy_maps(h->maps);
  delete[] h->blocks;
  std::free(h->ring_storage);
  std::free(h->undo_storage);
  std::free(h->plan_ids);
  std::free(h->plan_row0);
  std::free(h->plan_valid);
  std::free(h->plan_snapshot);
  std::free(h->plan_args);
  delete h;
  return KVC_OK;
}

int kvc_append_frame(kvc_handle* h, int32_t block, const void* K, const void* V, kvc_stream stream) {
  NvtxRange range("kvc_append_frame");
  int rc = check_block(h, block);
  if (rc) return rc;
  if (h->device ? (!K || !V || !aligned16(K) || !aligned16(V)) : (K || V)) return KVC_ERR_INVALID_ARG;
  Block& b = h->blocks[block];
  if (b.special_frames >= h->cfg.max_total_frames) return KVC_ERR_SPECIAL_POOL_FULL;
  if (b.free_list.size == 0) return KVC_ERR_NO_FREE_PAGE;
  // Where this frame's tokens go.
  const int32_t page = b.free_list.at(0);
  const int32_t s = b.special_frames;
  const int32_t sp_page = h->g.P + s / h->g.fpp;
  const int32_t sp_slot = kNumSpecial * (s % h->g.fpp);
  // Camera stream: the camera token (row 0) also goes to camera position s.
  const int32_t cam_page = camera_stream(h->cfg) ? h->g.first_camera + s / h->cfg.page_size : -1;
  const int32_t cam_slot = s % h->cfg.page_size;
  if (h->device) {
    char* cache_block = h->cache + (size_t)block * h->g.block_bytes;
    cudaError_t err = kvc::launch_append(cache_block, K, V, page, sp_page, sp_slot, cam_page, cam_slot,
                                         h->cfg.page_size, h->g.row_bytes, h->g.max_pages,
                                         (int32_t*)(h->ws + h->g.L.status), (cudaStream_t)stream, h->opt_pdl);
    if (err != cudaSuccess) return KVC_ERR_CUDA;
    ++h->launches;
  }
  // Commit the bookkeeping only once the copy is enqueued.
  b.free_list.pop_front();
  const bool to_scale = b.scale.size < h->cfg.scale_frames;   // _write_patch_page routing
  if (to_scale) b.scale.push_back(page); else b.live.push_back(page);
  b.undo[b.n_undo++] = Undo{page, to_scale ? 1 : 0};
  b.special_frames = s + 1;
  b.frame_count += 1;
  return KVC_OK;
}

int kvc_evict_frames(kvc_handle* h, int32_t block, int32_t scale_frames, int32_t sliding_window) {
  int rc = check_block(h, block);
  if (rc) return rc;
  if (scale_frames != h->cfg.scale_frames || sliding_window < 0) return KVC_ERR_INVALID_ARG;
  if (h->defer) return KVC_OK;
  evict_to(h->blocks[block], sliding_window, false);
  return KVC_OK;
}

int kvc_evict_frames_ex(kvc_handle* h, int32_t block, int32_t scale_frames, int32_t sliding_window,
                        int32_t cross_frame_special, int32_t camera_only) {
  int rc = check_block(h, block);
  if (rc) return rc;
  // The options are the cache's (kvc_config.special_policy), like scale_frames.
  if ((cross_frame_special != 0) != cross_frame(h->cfg) ||
      (camera_only != 0) != ((h->cfg.special_policy & KVC_SPECIAL_CAMERA_ONLY) != 0))
    return KVC_ERR_INVALID_ARG;
  return kvc_evict_frames(h, block, scale_frames, sliding_window);
}

int kvc_set_defer_eviction(kvc_handle* h, int32_t on) {
  if (!h) return KVC_ERR_INVALID_ARG;
  h->defer = on != 0;
  return KVC_OK;
}

int kvc_execute_deferred_eviction(kvc_handle* h, int32_t block, int32_t scale_frames,
                                  int32_t sliding_window) {
  int rc = check_block(h, block);
  if (rc) return rc;
  if (scale_frames != h->cfg.scale_frames || sliding_window < 0) return KVC_ERR_INVALID_ARG;
  evict_to(h->blocks[block], sliding_window, true);
  return KVC_OK;
}

int kvc_rollback_last_frame(kvc_handle* h, int32_t block) {
  int rc = check_block(h, block);
  if (rc) return rc;
  Block& b = h->blocks[block];
  if (b.n_undo == 0) return KVC_ERR_NOTHING_TO_ROLLBACK;
  const Undo u = b.undo[b.n_undo - 1];
  Ring& region = u.to_scale ? b.scale : b.live;
  if (region.size == 0 || region.back() != u.page) return KVC_ERR_ROLLBACK_AFTER_EVICT;
  region.pop_back();
  b.free_list.push_front(u.page);
  b.n_undo -= 1;
  b.special_frames -= 1;
  b.frame_count -= 1;
  return KVC_OK;
}

int kvc_clean(kvc_handle* h) {
  if (!h) return KVC_ERR_INVALID_ARG;
  for (int b = 0; b < h->cfg.num_blocks; ++b) h->blocks[b].reset(h->g.P);
  h->defer = false;
  h->has_plan = false;
  return KVC_OK;
}

int kvc_plan(kvc_handle* h, kvc_stream stream) {
  NvtxRange range("kvc_plan");
  if (!h) return KVC_ERR_INVALID_ARG;
  const Block& b = h->blocks[0];
  const int32_t fpp = h->g.fpp;
  const int32_t s = b.special_frames;
  const int32_t n_scale = b.scale.size, n_live = b.live.size;
  const int32_t n_patch = n_scale + n_live;
  // Special-stream runs in frame positions: the frames of the scale pages are
  // positions [0, n_scale) and the live frames [s - n_live, s), since frames
  // enter the special stream in append order, eviction takes the oldest live
  // frame and rollback the newest.  The default policy keeps every frame's
  // specials; without cross-frame specials only those two runs are visible;
  // camera_only adds the evicted frames' camera tokens, camera positions
  // [n_scale, s - n_live).
  kvc::PlanArgs& a = *h->plan_args;
  a.n_runs = 0;
  const int32_t evicted_lo = n_scale, evicted_hi = s - n_live;
  if (h->cfg.special_policy == 0 || evicted_lo >= evicted_hi) {
    a.runs[a.n_runs++] = kvc::PlanRun{h->g.P, fpp, kNumSpecial, 0, s};
  } else {
    a.runs[a.n_runs++] = kvc::PlanRun{h->g.P, fpp, kNumSpecial, 0, n_scale};
    a.runs[a.n_runs++] = kvc::PlanRun{h->g.P, fpp, kNumSpecial, evicted_hi, s};
    if (camera_stream(h->cfg))
      a.runs[a.n_runs++] = kvc::PlanRun{h->g.first_camera, h->cfg.page_size, 1, evicted_lo, evicted_hi};
  }
  int32_t n_pages = n_patch;
  for (int r = 0; r < a.n_runs; ++r) n_pages += kvc::run_pages(a.runs[r]);
  if (n_pages == 0) return KVC_ERR_EMPTY;
  if (n_pages > h->g.max_entries) return KVC_ERR_INVALID_ARG;
  const int kernel = h->device ? attn_kernel_for(h) : 1;
  if (kernel < 0) return KVC_ERR_INVALID_ARG;
  const int32_t tr = tile_rows_for(h, kernel);
  a.n_patch = n_patch;
  a.page_size = h->cfg.page_size;
  a.tile_rows = tr;
  a.max_pages = h->g.max_pages;
  for (int32_t i = 0; i < n_scale; ++i) a.patch_ids[i] = b.scale.at(i);
  for (int32_t i = 0; i < n_live; ++i) a.patch_ids[n_scale + i] = b.live.at(i);
  // Host copy of the visible entries (the device plan kernel writes the same).
  int32_t e = 0;
  for (; e < n_patch; ++e) {
    h->plan_ids[e] = a.patch_ids[e];
    h->plan_row0[e] = 0;
    h->plan_valid[e] = h->cfg.page_size;
  }
  for (int r = 0; r < a.n_runs; ++r) {
    const int32_t n = kvc::run_pages(a.runs[r]);
    for (int32_t i = 0; i < n; ++i, ++e)
      kvc::run_entry(a.runs[r], i, &h->plan_ids[e], &h->plan_row0[e], &h->plan_valid[e]);
  }
  // Tensor-core plans pack tiles in 8-row units when no tile can span more
  // than two entries; the count is ceil(units / 16), never more than one page
  // per tile gives.
  constexpr int32_t U = kvc::kPackUnitRows;
  bool pack = kernel == 2 && h->opt_pack && tr == kvc::kTcTileRows;
  int64_t units = 0, n_tiles = 0;
  for (int32_t i = 0; i < n_pages; ++i) {
    const int32_t u = (h->plan_valid[i] + U - 1) / U;
    if (i + 1 < n_pages && u < kvc::kPackMinUnits) pack = false;
    units += u;
    n_tiles += (h->plan_valid[i] + tr - 1) / tr;
  }
  if (pack) n_tiles = (units + tr / U - 1) / (tr / U);
  if (n_tiles > h->g.L.max_tiles) return KVC_ERR_INVALID_ARG;
  a.pack = pack ? 1 : 0;
  if (h->device) {
    cudaError_t err = kvc::launch_plan(a, h->ws, h->g.L, (cudaStream_t)stream, h->opt_pdl);
    if (err != cudaSuccess) return KVC_ERR_CUDA;
    ++h->launches;
  }
  for (int32_t i = 0; i < n_patch; ++i) h->plan_snapshot[i] = a.patch_ids[i];
  h->plan_n_scale = n_scale;
  h->plan_n_live = n_live;
  h->plan_special_frames = s;
  h->plan_n_pages = n_pages;
  // For the default policy this is compute_last_page_len: the last special
  // page's tokens ([KVC] "Physical Page Layout and Indexing").
  h->plan_lpl = h->plan_valid[n_pages - 1];
  h->plan_n_tiles = (int32_t)n_tiles;
  h->plan_packed = pack;
  h->plan_tile_rows = tr;
  h->plan_kernel = kernel;
  h->has_plan = true;
  return KVC_OK;
}

int kvc_run(kvc_handle* h, int32_t block, const void* Q, void* out, int32_t n_q, kvc_stream stream) {
  NvtxRange range("kvc_run");
  int rc = check_run(h, block, Q, out, n_q);
  if (rc || n_q == 0) return rc;
  const int kernel = h->plan_kernel;
  const Shape shape = choose_shape(h, kernel, n_q);
  const int splits = shape.splits;
  const kvc::AttnArgs a = attn_args(h, block, Q, out, n_q, splits);
  cudaStream_t st = (cudaStream_t)stream;
  const bool timed = timed_launch(h);
  if (timed) record_timing(h, 0, st);
  cudaError_t err;
  if (kernel == 2) {
    kvc::TcBatchArgs tb = tc_batch_header(h, Q, out, n_q);
    tb.q_tiles = shape.qt;
    tb.count = 1;
    h->last_qt = shape.qt;
    h->last_splits = splits;
    tb.req[0] = tc_request(h, block, 0, n_q, splits);
    err = kvc::launch_attn_tc(tb, st);
  } else {
    err = kvc::launch_attn_simt(a, h->cfg.dtype, st);
    h->last_qt = 0;
    h->last_splits = splits;
  }
  if (timed) record_timing(h, 1, st);
  if (err != cudaSuccess) return KVC_ERR_CUDA;
  ++h->launches;
  ++h->attn_launches;
  if (splits > 1) {
    err = kvc::launch_merge(a, h->cfg.dtype, st);
    if (err != cudaSuccess) return KVC_ERR_CUDA;
    ++h->launches;
  }
  return KVC_OK;
}

// Several independent streams in one launch: FlashInfer's batch plan takes a
// qo_indptr with one entry per request ([KVC] "Kernel-Level Execution Flow");
// the pages only ever use one.  Request r is handle hs[r]'s block blocks[r]
// with query rows [qo_indptr[r], qo_indptr[r+1]) of Q / out.
int kvc_run_batch(kvc_handle* const* hs, const int32_t* blocks, int32_t count, const void* Q, void* out,
                  const int32_t* qo_indptr, kvc_stream stream) {
  NvtxRange range("kvc_run_batch");
  if (!hs || !blocks || !qo_indptr || count < 1 || count > kvc::kTcMaxBatch) return KVC_ERR_INVALID_ARG;
  if (qo_indptr[0] != 0) return KVC_ERR_INVALID_ARG;
  for (int32_t r = 0; r < count; ++r) {
    kvc_handle* h = hs[r];
    if (!h) return KVC_ERR_INVALID_ARG;
    if (qo_indptr[r + 1] < qo_indptr[r]) return KVC_ERR_INVALID_ARG;
    for (int32_t o = 0; o < r; ++o)
      if (hs[o] == h) return KVC_ERR_INVALID_ARG;   // each handle's partials serve one request
    const kvc_config& c0 = hs[0]->cfg;
    if (h->cfg.num_heads != c0.num_heads || h->cfg.head_dim != c0.head_dim || h->cfg.dtype != c0.dtype ||
        h->cfg.sm_scale != c0.sm_scale)
      return KVC_ERR_INVALID_ARG;
  }
  const int64_t row_bytes = hs[0]->g.row_bytes;
  const int32_t rows = qo_indptr[count];
  // Every request checked before anything is launched.
  bool all_tc = true;
  for (int32_t r = 0; r < count; ++r) {
    const int32_t n_q = qo_indptr[r + 1] - qo_indptr[r];
    const char* q = n_q ? (const char*)Q + (int64_t)qo_indptr[r] * row_bytes : nullptr;
    char* o = n_q ? (char*)out + (int64_t)qo_indptr[r] * row_bytes : nullptr;
    int rc = check_run(hs[r], blocks[r], q, o, n_q);
    if (rc) return rc;
    all_tc = all_tc && hs[r]->plan_kernel == 2;
  }
  if (rows == 0) return KVC_OK;
  if (!all_tc) {
    // No batched CUDA-core kernel: the requests run one after the other.
    for (int32_t r = 0; r < count; ++r) {
      const int32_t n_q = qo_indptr[r + 1] - qo_indptr[r];
      if (n_q == 0) continue;
      int rc = kvc_run(hs[r], blocks[r], (const char*)Q + (int64_t)qo_indptr[r] * row_bytes,
                       (char*)out + (int64_t)qo_indptr[r] * row_bytes, n_q, stream);
      if (rc) return rc;
    }
    return KVC_OK;
  }
  // One shape for the whole launch: the cost model over all requests' CTAs,
  // the largest per-request tile count and all requests' merge traffic.
  kvc_handle* h0 = hs[0];
  int max_s = 1 << 30, max_tiles = 1;
  int64_t blocks2 = 0, blocks1 = 0;
  for (int32_t r = 0; r < count; ++r) {
    const kvc_handle* h = hs[r];
    const int32_t n_q = qo_indptr[r + 1] - qo_indptr[r];
    if (h->cfg.max_kv_splits < max_s) max_s = h->cfg.max_kv_splits;
    if (h->plan_n_tiles > max_tiles) max_tiles = h->plan_n_tiles;
    blocks2 += (n_q + 255) / 256;
    blocks1 += (n_q + 127) / 128;
  }
  if (max_s > max_tiles) max_s = max_tiles;
  if (max_s < 1) max_s = 1;
  const Shape shape = choose_tc_shape(h0, max_s, blocks2, blocks1, max_tiles, rows);
  const int splits = shape.splits;
  kvc::TcBatchArgs tb = tc_batch_header(h0, Q, out, rows);
  tb.q_tiles = shape.qt;
  tb.count = count;
  h0->last_qt = shape.qt;
  h0->last_splits = splits;
  for (int32_t r = 0; r < count; ++r) {
    const int32_t n_q = qo_indptr[r + 1] - qo_indptr[r];
    const int s_r = splits < hs[r]->plan_n_tiles ? splits : hs[r]->plan_n_tiles;
    tb.req[r] = tc_request(hs[r], blocks[r], qo_indptr[r], n_q, s_r > 0 ? s_r : 1);
  }
  cudaStream_t st = (cudaStream_t)stream;
  const bool timed = timed_launch(h0);
  if (timed) record_timing(h0, 0, st);
  cudaError_t err = kvc::launch_attn_tc(tb, st);
  if (timed) record_timing(h0, 1, st);
  if (err != cudaSuccess) return KVC_ERR_CUDA;
  ++h0->launches;
  ++h0->attn_launches;
  for (int32_t r = 0; r < count; ++r) {
    if (tb.req[r].n_splits <= 1 || tb.req[r].n_q == 0) continue;
    const int32_t n_q = tb.req[r].n_q;
    const kvc::AttnArgs a = attn_args(hs[r], blocks[r], (const char*)Q + (int64_t)qo_indptr[r] * row_bytes,
                                      (char*)out + (int64_t)qo_indptr[r] * row_bytes, n_q, tb.req[r].n_splits);
    err = kvc::launch_merge(a, hs[r]->cfg.dtype, st);
    if (err != cudaSuccess) return KVC_ERR_CUDA;
    ++h0->launches;
  }
  return KVC_OK;
}

// Phase 1 ([KVC] "FlashInferAttention Layer Implementation", batch mode;
// [SLOTS] "scale frames永不驱逐"): dense bidirectional attention of the first
// frames as one block, then append_frame per frame.  Appending the frames to
// an empty block first makes its visible set exactly their n_frames * T
// tokens, and non-causal attention over a set does not depend on the order
// of its keys, so the paged kernel computes the dense attention.
int kvc_prefill(kvc_handle* h, int32_t block, const void* Q, const void* K, const void* V, int32_t n_frames,
                void* out, kvc_stream stream) {
  int rc = check_block(h, block);
  if (rc) return rc;
  if (!h->device) return KVC_ERR_NO_DEVICE;
  const Block& b = h->blocks[block];
  if (n_frames < 1 || b.frame_count != 0 || b.special_frames != 0 || b.scale.size != 0 || b.live.size != 0)
    return KVC_ERR_INVALID_ARG;
  const int64_t n_q = (int64_t)n_frames * h->g.T;
  if (n_q > h->cfg.max_query_tokens) return KVC_ERR_INVALID_ARG;
  if (!Q || !K || !V || !out || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out))
    return KVC_ERR_INVALID_ARG;
  if (n_frames > b.free_list.size) return KVC_ERR_NO_FREE_PAGE;
  if (n_frames > h->cfg.max_total_frames) return KVC_ERR_SPECIAL_POOL_FULL;
  const int64_t frame_bytes = h->g.T * h->g.row_bytes;
  int32_t appended = 0;
  for (; appended < n_frames; ++appended) {
    rc = kvc_append_frame(h, block, (const char*)K + appended * frame_bytes,
                          (const char*)V + appended * frame_bytes, stream);
    if (rc) break;
  }
  bool planned = false;
  if (rc == KVC_OK && block == 0) planned = (rc = kvc_plan(h, stream)) == KVC_OK;
  if (rc == KVC_OK) rc = kvc_run(h, block, Q, out, (int32_t)n_q, stream);
  if (rc != KVC_OK) {
    // Leave the bookkeeping as it was (cache bytes are not part of it); a
    // plan made here described the frames just undone, so it is dropped.
    for (int32_t f = 0; f < appended; ++f) kvc_rollback_last_frame(h, block);
    if (planned) h->has_plan = false;
  }
  return rc;
}

int kvc_get_cache_stats(const kvc_handle* h, int32_t block, kvc_stats* out) {
  int rc = check_block(h, block);
  if (rc) return rc;
  if (!out) return KVC_ERR_INVALID_ARG;
  const Block& b = h->blocks[block];
  out->frame_count = b.frame_count;
  out->scale_pages = b.scale.size;
  out->live_pages = b.live.size;
  out->free_pages = b.free_list.size;
  out->special_tokens = (int64_t)kNumSpecial * b.special_frames;
  return KVC_OK;
}

int kvc_get_plan(const kvc_handle* h, int32_t* indptr2, int32_t* indices, int32_t cap,
                 int32_t* n_pages, int32_t* last_page_len) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->has_plan) return KVC_ERR_NO_PLAN;
  if (n_pages) *n_pages = h->plan_n_pages;
  if (last_page_len) *last_page_len = h->plan_lpl;
  if (indptr2) { indptr2[0] = 0; indptr2[1] = h->plan_n_pages; }
  if (indices) {
    if (cap < h->plan_n_pages) return KVC_ERR_INVALID_ARG;
    std::memcpy(indices, h->plan_ids, sizeof(int32_t) * h->plan_n_pages);
  }
  return KVC_OK;
}

int kvc_get_plan_ranges(const kvc_handle* h, int32_t* indices, int32_t* first_rows, int32_t* valid_lens,
                        int32_t cap, int32_t* n_pages) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->has_plan) return KVC_ERR_NO_PLAN;
  if (n_pages) *n_pages = h->plan_n_pages;
  if ((indices || first_rows || valid_lens) && cap < h->plan_n_pages) return KVC_ERR_INVALID_ARG;
  if (indices) std::memcpy(indices, h->plan_ids, sizeof(int32_t) * h->plan_n_pages);
  if (first_rows) std::memcpy(first_rows, h->plan_row0, sizeof(int32_t) * h->plan_n_pages);
  if (valid_lens) std::memcpy(valid_lens, h->plan_valid, sizeof(int32_t) * h->plan_n_pages);
  return KVC_OK;
}

int kvc_get_deques(const kvc_handle* h, int32_t block, int32_t* scale, int32_t* n_scale,
                   int32_t* live, int32_t* n_live, int32_t* free_list, int32_t* n_free) {
  int rc = check_block(h, block);
  if (rc) return rc;
  const Block& b = h->blocks[block];
  if (n_scale) *n_scale = b.scale.size;
  if (n_live) *n_live = b.live.size;
  if (n_free) *n_free = b.free_list.size;
  if (scale) for (int32_t i = 0; i < b.scale.size; ++i) scale[i] = b.scale.at(i);
  if (live) for (int32_t i = 0; i < b.live.size; ++i) live[i] = b.live.at(i);
  if (free_list) for (int32_t i = 0; i < b.free_list.size; ++i) free_list[i] = b.free_list.at(i);
  return KVC_OK;
}

int kvc_read_device_ranges(kvc_handle* h, int32_t* indices, int32_t* first_rows, int32_t* valid_lens,
                           int32_t cap, int32_t* n_pages, kvc_stream stream) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->device) return KVC_ERR_NO_DEVICE;
  int32_t n = 0;
  int rc = kvc_read_device_plan(h, indices, valid_lens, cap, &n, nullptr, stream);
  if (rc) return rc;
  if (n_pages) *n_pages = n;
  if (first_rows && n > 0) {
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(first_rows, h->ws + h->g.L.page_row0, 4 * (size_t)n, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  return KVC_OK;
}

int kvc_read_device_plan(kvc_handle* h, int32_t* indices, int32_t* valid_lens, int32_t cap,
                         int32_t* n_pages, int32_t* last_page_len, kvc_stream stream) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->device) return KVC_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  kvc::DevPlanHeader hd;
  if (cudaMemcpyAsync(&hd, h->ws + h->g.L.header, sizeof(hd), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (n_pages) *n_pages = hd.n_pages;
  if (last_page_len) *last_page_len = hd.last_page_len;
  if (hd.n_pages < 0 || hd.n_pages > h->g.max_entries) return KVC_ERR_INVALID_ARG;
  if ((indices || valid_lens) && cap < hd.n_pages) return KVC_ERR_INVALID_ARG;
  if (hd.n_pages > 0) {
    if (indices && cudaMemcpyAsync(indices, h->ws + h->g.L.page_ids, 4 * (size_t)hd.n_pages,
                                   cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return KVC_ERR_CUDA;
    if (valid_lens && cudaMemcpyAsync(valid_lens, h->ws + h->g.L.page_valid, 4 * (size_t)hd.n_pages,
                                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
  }
  return KVC_OK;
}

int kvc_device_status(kvc_handle* h, kvc_stream stream) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->device) return KVC_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t flag = 0;
  if (cudaMemcpyAsync(&flag, h->ws + h->g.L.status, sizeof(flag), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (flag == 0) return KVC_OK;
  if (cudaMemsetAsync(h->ws + h->g.L.status, 0, 256, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVC_ERR_CUDA;
  return flag == kvc::kStatusBounds ? KVC_ERR_DEVICE_BOUNDS : KVC_ERR_DEVICE_TIMEOUT;
}

int kvc_set_option(kvc_handle* h, int32_t option, int64_t value) {
  if (!h) return KVC_ERR_INVALID_ARG;
  switch (option) {
    case KVC_OPT_ATTN_KERNEL:
      if (value < 0 || value > 2) return KVC_ERR_INVALID_ARG;
      if (value == 2 && !h->maps) return KVC_ERR_INVALID_ARG;
      h->opt_kernel = (int)value;
      h->has_plan = false;      // tile sizes differ between kernels
      return KVC_OK;
    case KVC_OPT_NUM_SPLITS:
      if (value < 0 || value > h->cfg.max_kv_splits) return KVC_ERR_INVALID_ARG;
      h->opt_splits = (int)value;
      return KVC_OK;
    case KVC_OPT_QUERY_TILES:
      if (value < 0 || value > 2) return KVC_ERR_INVALID_ARG;
      h->opt_qtiles = (int)value;
      return KVC_OK;
    case KVC_OPT_PDL:
      if (value < 0 || value > 1) return KVC_ERR_INVALID_ARG;
      h->opt_pdl = value != 0;
      return KVC_OK;
    case KVC_OPT_PACK_TILES:
      if (value < 0 || value > 1) return KVC_ERR_INVALID_ARG;
      h->opt_pack = value != 0;
      h->has_plan = false;      // the tile list changes
      return KVC_OK;
    case KVC_OPT_WAIT_BUDGET:
      if (value < 0) return KVC_ERR_INVALID_ARG;
      h->wait_budget = value;
      return KVC_OK;
    case KVC_OPT_STALL_TEST:
      if (value < 0 || value > 1) return KVC_ERR_INVALID_ARG;
      h->stall_test = (int)value;
      return KVC_OK;
    case KVC_OPT_TIMING:
      if (value < 0 || value > 0x7fffffff) return KVC_ERR_INVALID_ARG;
      if (value && !h->ev) {
        if (!h->device) return KVC_ERR_NO_DEVICE;
        cudaEvent_t* ev = (cudaEvent_t*)std::calloc(2 * kEventPairs, sizeof(cudaEvent_t));
        bool* used = (bool*)std::calloc(kEventPairs, sizeof(bool));
        if (!ev || !used) { std::free(ev); std::free(used); return KVC_ERR_INVALID_ARG; }
        for (int i = 0; i < 2 * kEventPairs; ++i) {
          if (cudaEventCreate(&ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            std::free(ev);
            std::free(used);
            return KVC_ERR_CUDA;
          }
        }
        h->ev = ev;
        h->ev_used = used;
      }
      drain_timing(h);                          // earlier samples keep their own scale
      h->timing = value != 0;
      h->timing_every = value > 1 ? (int32_t)value : 1;
      h->timing_count = 0;
      return KVC_OK;
    default:
      return KVC_ERR_INVALID_ARG;
  }
}

int kvc_get_counters(kvc_handle* h, int64_t* kernel_launches, int64_t* attn_launches, double* attn_ms,
                     int32_t reset) {
  if (!h) return KVC_ERR_INVALID_ARG;
  drain_timing(h);
  if (kernel_launches) *kernel_launches = h->launches;
  if (attn_launches) *attn_launches = h->attn_launches;
  if (attn_ms) *attn_ms = h->attn_ms;
  if (reset) {
    h->launches = 0;
    h->attn_launches = 0;
    h->attn_ms = 0.0;
  }
  return KVC_OK;
}

int kvc_get_plan_tiles(const kvc_handle* h, int32_t* n_tiles, int32_t* packed) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (!h->has_plan) return KVC_ERR_NO_PLAN;
  if (n_tiles) *n_tiles = h->plan_n_tiles;
  if (packed) *packed = h->plan_packed ? 1 : 0;
  return KVC_OK;
}

int kvc_get_launch_shape(const kvc_handle* h, int32_t* q_tiles, int32_t* splits) {
  if (!h) return KVC_ERR_INVALID_ARG;
  if (q_tiles) *q_tiles = h->last_qt;
  if (splits) *splits = h->last_splits;
  return KVC_OK;
}

const char* kvc_strerror(int code) {
  switch (code) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_NO_FREE_PAGE: return "no free patch page";
    case KVC_ERR_SPECIAL_POOL_FULL: return "special token pool full (max_total_frames reached)";
    case KVC_ERR_NOTHING_TO_ROLLBACK: return "nothing to roll back";
    case KVC_ERR_ROLLBACK_AFTER_EVICT: return "rollback after eviction";
    case KVC_ERR_NO_PLAN: return "no plan";
    case KVC_ERR_STALE_PLAN: return "stale plan: block state differs from the planned state";
    case KVC_ERR_CUDA: return "CUDA error";
    case KVC_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case KVC_ERR_EMPTY: return "no visible token";
    case KVC_ERR_NO_DEVICE: return "bookkeeping-only handle";
    case KVC_ERR_TOO_LARGE: return "too many pages or KV tiles for the static scratch array";
    case KVC_ERR_DEVICE_BOUNDS: return "device bounds check failed (KVC_CHECKED build)";
    default: return "unknown error";
  }
}

}  // extern "C"
