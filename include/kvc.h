/*
 * kvc.h -- C ABI of the GB300 two-stream paged KV cache and its per-frame
 * paged attention (libkvc.so).
 *
 * Pages cited by tag, then section:
 *   [KVC]   "How LingBot-Map Implements the KV Cache Mechanism for Streaming
 *           Inference with FlashInfer Integration"
 *   [PERF]  "How to Improve Streaming Inference Performance with FlashInfer KV
 *           Cache Backend"
 *   [SLOTS] "LingBot-Map KV缓存机制深度揭秘：scale frames与keyframes如何占用slot"
 *
 * Model.  A model of `num_blocks` transformer blocks keeps one paged cache
 * per block, all in ONE caller-owned device buffer laid out as
 *     cache[num_blocks][max_num_pages][2][page_size][num_heads][head_dim]
 * (index 0 = K, 1 = V; [KVC] "Physical Page Layout and Indexing").  Pages
 * 0..P-1, P = scale_frames + sliding_window + headroom, hold one frame's
 * patch tokens each and are recycled; pages P..max_num_pages-1 form the
 * append-only special stream, floor(page_size/6) frames per page
 * ([SLOTS] "双流分页布局", "特殊 token 流").  A frame's K/V/Q are
 * [6 + page_size, num_heads, head_dim] row-major (NHD), rows 0..5 the
 * special tokens (camera, 4 registers, scale), rows 6.. the patch tokens
 * ([SLOTS] intro).
 *
 * Conventions.
 *   - Every call returns KVC_OK (0) or a negative KVC_ERR_* code; a call that
 *     fails leaves the host bookkeeping exactly as it was.
 *   - Host bookkeeping is synchronous.  Device work is enqueued on the
 *     `stream` argument (a cudaStream_t; NULL = the legacy default stream) and
 *     its buffers must stay valid until the stream has passed it.
 *   - The library allocates no device memory.  The caller allocates the cache
 *     and the workspace (sizes from kvc_required_bytes, 256-byte aligned) and
 *     keeps ownership; the library borrows them until kvc_destroy.
 *   - A handle is not thread-safe; calls on one handle must be serialised.
 *   - Element pointers (K, V, Q, out) are device pointers to contiguous
 *     arrays of the configured dtype, 16-byte aligned.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { KVC_BF16 = 0, KVC_F16 = 1, KVC_F32 = 2 } kvc_dtype;

enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = -1,         /* bad handle, block, size, pointer or option    */
  KVC_ERR_NO_FREE_PAGE = -2,        /* patch pool exhausted (uncommitted frames)     */
  KVC_ERR_SPECIAL_POOL_FULL = -3,   /* max_total_frames frames already appended      */
  KVC_ERR_NOTHING_TO_ROLLBACK = -4, /* no uncommitted append on this block           */
  KVC_ERR_ROLLBACK_AFTER_EVICT = -5,/* the append to undo is no longer the newest    */
  KVC_ERR_NO_PLAN = -6,             /* kvc_run before any kvc_plan (or after clean)  */
  KVC_ERR_STALE_PLAN = -7,          /* block state differs from the planned state    */
  KVC_ERR_CUDA = -8,                /* a CUDA runtime call failed                    */
  KVC_ERR_DEVICE_TIMEOUT = -9,      /* a kernel gave up waiting (kvc_device_status)  */
  KVC_ERR_EMPTY = -10,              /* plan of a cache with no visible token         */
  KVC_ERR_NO_DEVICE = -11,          /* device call on a bookkeeping-only handle      */
  KVC_ERR_TOO_LARGE = -12,          /* beyond kvc_paged_attention_static's scratch   */
  KVC_ERR_DEVICE_BOUNDS = -13       /* a bounds check failed (KVC_CHECKED builds)    */
};

typedef struct kvc_handle kvc_handle;
typedef void* kvc_stream; /* cudaStream_t */

/* Construction arguments ([PERF] "Minimal Streaming Inference Setup";
 * [KVC] "Lazy Initialization of the KV Cache").  Zero in sm_scale,
 * max_query_tokens, max_kv_splits or num_special_tokens selects the default
 * noted beside it; the other fields are used as given.  Limits: head_dim in
 * {32, 64, 128}; 6 <= page_size <= 65536; 1 <= P <= 1024;
 * num_heads * head_dim * element size a multiple of 16 bytes. */
typedef struct {
  int32_t num_blocks;         /* transformer blocks (layers), >= 1                 */
  int32_t num_heads;          /* H: query heads == KV heads                        */
  int32_t head_dim;           /* D                                                 */
  int32_t page_size;          /* patch tokens per frame == tokens per page (exact) */
  int32_t num_special_tokens; /* must be 6 (0 => 6)                                */
  int32_t scale_frames;       /* never-evicted anchor frames (pages: 8)            */
  int32_t sliding_window;     /* live window pages (pages: 64)                     */
  int32_t headroom;           /* spare patch pages (pages: 16)                     */
  int32_t max_total_frames;   /* special-stream capacity in frames (pages: 2048)   */
  int32_t dtype;              /* kvc_dtype of K, V, Q, out and the cache           */
  float sm_scale;             /* softmax scale; 0 => 1/sqrt(head_dim)              */
  int32_t max_query_tokens;   /* largest n_q of kvc_run; 0 => 6 + page_size        */
  int32_t max_kv_splits;      /* split-KV partial buffers; 0 => 32                 */
  int32_t special_policy;     /* KVC_SPECIAL_* flags; 0 => every frame's specials  */
} kvc_config;

/* What stays visible of an evicted frame's special tokens: the eviction
 * options cross_frame_special and camera_only that the block passes to
 * evict_frames ([KVC] "Streaming Forward Pass").  The pages do not say what
 * they do; this library reads them as follows.
 *   0 (cross_frame_special on, camera_only off): every frame's six specials
 *     stay visible after its patch page is evicted -- the pages' two-stream
 *     behaviour ([SLOTS] "特殊 token 流": the special stream is never evicted).
 *   KVC_SPECIAL_NO_CROSS_FRAME (cross_frame_special off): a frame's specials
 *     leave the visible set together with its patch page; the scale and live
 *     frames' specials stay.  camera_only then changes nothing.
 *   KVC_SPECIAL_CAMERA_ONLY (camera_only on): of an evicted frame's specials
 *     only the camera token (the first of the six) stays visible.  Every
 *     frame's camera token is then also written to a third append-only
 *     stream, the camera pages (page_size tokens per page, after the special
 *     pages; see kvc_get_geometry), so that the evicted frames' camera
 *     tokens form one contiguous run.
 * The special stream itself is the same in every policy. */
enum { KVC_SPECIAL_NO_CROSS_FRAME = 1, KVC_SPECIAL_CAMERA_ONLY = 2 };

/* get_cache_stats snapshot ([SLOTS] "动手验证"). */
typedef struct {
  int64_t frame_count;
  int64_t scale_pages;
  int64_t live_pages;
  int64_t free_pages;
  int64_t special_tokens;
} kvc_stats;

/* Byte sizes of the cache and of the workspace (plan tables, split-KV partial
 * outputs and the device status word) for `cfg`.  Validates cfg. */
int kvc_required_bytes(const kvc_config* cfg, size_t* cache_bytes, size_t* workspace_bytes);

/* Page geometry of the cache `cfg` describes ([PERF] "Two-Stream Page Pool
 * Architecture"; [SLOTS] "双流分页布局", "特殊 token 流"): P =
 * scale_frames + sliding_window + headroom patch pages, floor(page_size / 6)
 * frames per special page, ceil(max_total_frames / that) special pages; one
 * block's cache is [max_num_pages][2][page_size][H][D] (page_bytes per page,
 * block_bytes per block, blocks back to back).  Validates cfg. */
typedef struct {
  int32_t num_patch_pages;
  int32_t frames_per_special_page;
  int32_t num_special_pages;
  int32_t num_camera_pages;   /* KVC_SPECIAL_CAMERA_ONLY: ceil(max_total_frames / page_size), else 0 */
  int32_t max_num_pages;      /* patch + special + camera pages */
  int32_t tokens_per_frame;   /* 6 + page_size */
  int64_t page_bytes;
  int64_t block_bytes;
} kvc_geometry;
int kvc_get_geometry(const kvc_config* cfg, kvc_geometry* out);

/* Create a handle.  cache_dev / workspace_dev: caller-owned device buffers of
 * the sizes above, 256-byte aligned; the cache is zero-filled and the
 * workspace initialised on `stream` (the pages allocate with torch.empty: the
 * zero fill is this library's choice, so that cache bytes are defined).
 * Passing NULL for both gives a bookkeeping-only handle: every host call
 * works, device calls return KVC_ERR_NO_DEVICE.  All host memory the handle
 * will ever use is allocated here ([PERF] "Two-Stream Page Pool Architecture":
 * allocation happens once, at construction). */
int kvc_create(const kvc_config* cfg, void* cache_dev, void* workspace_dev, kvc_stream stream,
               kvc_handle** out);

/* Release the handle (not the caller's buffers).  Waits for nothing. */
int kvc_destroy(kvc_handle* h);

/* append_frame(block_idx, K, V) ([KVC] "Append and Evict API"; [SLOTS]
 * "scale frames永不驱逐"): take the left-most free patch page, route it to the
 * scale region while that holds fewer than scale_frames pages, else to the
 * live window; copy K/V rows 6.. into that page and rows 0..5 into slots
 * [6*(s%fpp), +6) of special page P + s/fpp, s = frames already in the
 * special stream.  K, V: device [6 + page_size, H, D]; on a
 * bookkeeping-only handle both must be NULL and only the bookkeeping runs.
 * Errors: NO_FREE_PAGE, SPECIAL_POOL_FULL, INVALID_ARG, CUDA (state
 * unchanged). */
int kvc_append_frame(kvc_handle* h, int32_t block, const void* K, const void* V, kvc_stream stream);

/* evict_frames(block_idx, scale_frames, sliding_window) ([SLOTS]
 * "keyframes滑动窗口"): while the live window holds more than sliding_window
 * pages, move its oldest page to the right end of the free list.  A no-op
 * while eviction is deferred.  An eviction that moves a page commits the
 * block's pending frames.  scale_frames must equal the configured value. */
int kvc_evict_frames(kvc_handle* h, int32_t block, int32_t scale_frames, int32_t sliding_window);

/* evict_frames with the block's two eviction options as the pages pass them
 * ([KVC] "Streaming Forward Pass": cross_frame_special, camera_only; nonzero =
 * on).  They must match the cache's special_policy (as scale_frames must
 * match the configured value), else INVALID_ARG; then as kvc_evict_frames. */
int kvc_evict_frames_ex(kvc_handle* h, int32_t block, int32_t scale_frames, int32_t sliding_window,
                        int32_t cross_frame_special, int32_t camera_only);

/* Manager-wide deferral switch, the `_defer_eviction` attribute ([PERF]
 * "Deferred Eviction Strategy"). */
int kvc_set_defer_eviction(kvc_handle* h, int32_t on);

/* execute_deferred_eviction ([SLOTS] "光流关键帧与回滚机制"): evict down to
 * sliding_window regardless of deferral and commit the pending frames. */
int kvc_execute_deferred_eviction(kvc_handle* h, int32_t block, int32_t scale_frames,
                                  int32_t sliding_window);

/* rollback_last_frame ([SLOTS] "光流关键帧与回滚机制"): undo the newest
 * uncommitted append exactly -- its page returns to the LEFT end of the free
 * list, the special and frame counts drop by one.  Cache bytes are not
 * touched.  Errors: NOTHING_TO_ROLLBACK, ROLLBACK_AFTER_EVICT. */
int kvc_rollback_last_frame(kvc_handle* h, int32_t block);

/* clean_kv_cache ([SLOTS] "窗口模式"): every block back to its construction
 * state (free list 0..P-1, nothing visible), deferral off, plan dropped. */
int kvc_clean(kvc_handle* h);

/* plan ([KVC] "Kernel-Level Execution Flow"; [PERF] "One-Time Planning
 * Pattern"): from block 0's state build the visible page table -- scale pages,
 * live window, then every special page -- and last_page_len, and write the
 * device page table / tile list for kvc_run on `stream`.  Call once per frame
 * after block 0's append/evict; every block then runs with it.  No host to
 * device copy: the page list travels as kernel arguments.  On a
 * bookkeeping-only handle only the host plan is built.  Errors: EMPTY. */
int kvc_plan(kvc_handle* h, kvc_stream stream);

/* run(block, Q, out) ([KVC] "Kernel-Level Execution Flow"): non-causal
 * softmax attention, scale sm_scale, of Q [n_q, H, D] over block `block`'s
 * visible tokens in plan order, written to out [n_q, H, D] (same dtype).
 * fp32 accumulation and softmax; split-KV partials merged by log-sum-exp.
 * 0 <= n_q <= max_query_tokens.  Errors: NO_PLAN, STALE_PLAN (this block's
 * pages differ from the plan's), INVALID_ARG, CUDA. */
int kvc_run(kvc_handle* h, int32_t block, const void* Q, void* out, int32_t n_q, kvc_stream stream);

/* Several independent streams in one launch.  FlashInfer's batch plan takes
 * a qo_indptr with one entry per request ([KVC] "Kernel-Level Execution
 * Flow"); the pages only ever pass one, so this call has no counterpart there
 * beyond that signature.  Request r (0 <= r < count <= 16) is handle hs[r]'s
 * block blocks[r] with query rows [qo_indptr[r], qo_indptr[r+1]) of Q and out
 * ([qo_indptr[count], H, D], the dtype of every handle).  The handles are
 * distinct, share num_heads, head_dim, dtype and sm_scale, and each has a
 * current plan for its block (as kvc_run requires).  With the tensor-core
 * kernel all requests go into one launch, with one KV split count chosen for
 * the whole batch (each handle's partial buffers hold its own request's
 * splits); otherwise the requests run one after another.  Launch counters and
 * KVC_OPT_TIMING are kept by hs[0].  qo_indptr is a host array.  Errors:
 * INVALID_ARG (count, pointers, qo_indptr not starting at 0 or decreasing,
 * repeated handles, different geometry), and for the first failing request
 * those of kvc_run -- nothing is launched then. */
int kvc_run_batch(kvc_handle* const* hs, const int32_t* blocks, int32_t count, const void* Q, void* out,
                  const int32_t* qo_indptr, kvc_stream stream);

/* Phase 1, batch mode ([KVC] "FlashInferAttention Layer Implementation";
 * [SLOTS] "scale frames永不驱逐"): the first n_frames frames attend to each
 * other densely and bidirectionally as one block, then are appended frame by
 * frame.  K and V are [n_frames * (6 + page_size), H, D], frame after frame,
 * each frame laid out as kvc_append_frame expects; Q and out are the same
 * shape.  The block must be empty (fresh, or after kvc_clean).  The frames
 * are appended (no eviction), then -- for block 0 -- the plan is rebuilt, and
 * the queries attend over the block's visible tokens, which are exactly the
 * n_frames frames' tokens; the result is the dense attention because the
 * order of keys does not change a softmax-weighted sum.  Blocks other than 0
 * use block 0's plan, as in streaming, so block 0 is prefilled first.
 * n_frames * (6 + page_size) <= max_query_tokens.  Errors: INVALID_ARG (block
 * not empty, sizes, pointers), NO_FREE_PAGE, SPECIAL_POOL_FULL, STALE_PLAN,
 * NO_DEVICE, CUDA; on an error the block's bookkeeping is left unchanged. */
int kvc_prefill(kvc_handle* h, int32_t block, const void* Q, const void* K, const void* V, int32_t n_frames,
                void* out, kvc_stream stream);

/* get_cache_stats(block_idx) ([SLOTS] "动手验证"). */
int kvc_get_cache_stats(const kvc_handle* h, int32_t block, kvc_stats* out);

/* Host copy of the current plan: indptr2 = {0, n_pages}, indices[0..n_pages)
 * (if cap allows), n_pages, last_page_len.  Errors: NO_PLAN, INVALID_ARG
 * (cap too small; n_pages is still written). */
int kvc_get_plan(const kvc_handle* h, int32_t* indptr2, int32_t* indices, int32_t cap,
                 int32_t* n_pages, int32_t* last_page_len);

/* Host copy of the current plan as row ranges: visible entry i is rows
 * [first_rows[i], first_rows[i] + valid_lens[i]) of page indices[i] (with the
 * default special policy every first row is 0 and this is kvc_get_plan's
 * table).  Arrays of cap entries, any may be NULL.  Errors: NO_PLAN,
 * INVALID_ARG (cap too small; n_pages is still written). */
int kvc_get_plan_ranges(const kvc_handle* h, int32_t* indices, int32_t* first_rows, int32_t* valid_lens,
                        int32_t cap, int32_t* n_pages);

/* Snapshot of a block's deques (left to right) for parity checks; each array
 * needs room for P entries.  Any pointer may be NULL. */
int kvc_get_deques(const kvc_handle* h, int32_t block, int32_t* scale, int32_t* n_scale,
                   int32_t* live, int32_t* n_live, int32_t* free_list, int32_t* n_free);

/* Synchronously copy back the DEVICE page table written by kvc_plan:
 * indices and per-page valid token counts (cap entries each), n_pages and
 * last_page_len.  For parity tests; synchronises `stream`. */
int kvc_read_device_plan(kvc_handle* h, int32_t* indices, int32_t* valid_lens, int32_t cap,
                         int32_t* n_pages, int32_t* last_page_len, kvc_stream stream);

/* The device page table as row ranges (indices, first rows, valid counts);
 * for parity tests; synchronises `stream`. */
int kvc_read_device_ranges(kvc_handle* h, int32_t* indices, int32_t* first_rows, int32_t* valid_lens,
                           int32_t cap, int32_t* n_pages, kvc_stream stream);

/* Read and clear the device status word (synchronises `stream`).  Returns
 * KVC_ERR_DEVICE_BOUNDS if a kernel of a KVC_CHECKED build found a page id,
 * slot, tile row or TMA coordinate outside the cache (it skipped the access);
 * else
 * KVC_OK, or KVC_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait
 * since the last call. */
int kvc_device_status(kvc_handle* h, kvc_stream stream);

/* Tuning / test options (kvc_set_option). */
enum {
  KVC_OPT_ATTN_KERNEL = 1, /* 0 auto, 1 CUDA-core kernel, 2 tensor-core (tcgen05) kernel */
  KVC_OPT_NUM_SPLITS = 2,  /* 0 auto, else the number of KV splits (<= max_kv_splits)     */
  KVC_OPT_WAIT_BUDGET = 3, /* bounded-wait budget in SM clock cycles; 0 => default (~2 s) */
  KVC_OPT_TIMING = 4,      /* N >= 1: time attention launches with CUDA events on their
                              stream -- every one (N = 1), or one in every N: the (N/2)-th
                              of each group of N launches counted from this call, whose
                              time then counts N times in kvc_get_counters (a bench whose
                              step makes N launches of one shape times one per step);
                              0: off                                                         */
  KVC_OPT_STALL_TEST = 5,  /* test only, 1: the tensor-core kernel first waits on a barrier
                              that nothing signals, so its bounded wait runs out and the run
                              reports KVC_ERR_DEVICE_TIMEOUT (no output is written)           */
  KVC_OPT_QUERY_TILES = 6, /* tensor-core kernel: 128-row query tiles per CTA; 0 auto (a
                              cost model picks tiles and splits per launch), 1 (both softmax
                              warp groups share one tile, taking alternate KV tiles), 2 (one
                              warp group per tile)                                           */
  KVC_OPT_PACK_TILES = 7,  /* tensor-core kernel: 1 (default) packs the KV tiles across page
                              boundaries in units of 8 rows -- a page's last tile is filled
                              with the next page's first rows -- when every visible page but
                              the last has at least 113 rows (otherwise the plan keeps one
                              page per tile); 0 never packs.  Takes effect at the next
                              kvc_plan.                                                      */
  KVC_OPT_PDL = 8          /* 1 (default): launch with programmatic dependent launch, so that
                              each kernel of the library is set up while the kernel before it
                              in the stream drains (it touches no memory before that kernel has
                              completed); 0: ordinary launches                              */
};
int kvc_set_option(kvc_handle* h, int32_t option, int64_t value);

/* Counters since creation (or the last reset with reset != 0): kernel
 * launches made by the library, attention launches, and -- with
 * KVC_OPT_TIMING -- the summed device time of the timed attention launches in
 * milliseconds, each counted N times when one launch in every N is timed
 * (synchronises the pending timing events). */
int kvc_get_counters(kvc_handle* h, int64_t* kernel_launches, int64_t* attn_launches,
                     double* attn_ms, int32_t reset);

/* Paged attention that allocates nothing.  The pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory -- for
 * example code embedded in a host framework that owns all GPU memory and lends
 * out only the KV cache and the Q / output buffers, so that it cannot provide
 * the workspace kvc_create needs.  It computes what kvc_run computes (CUDA-core
 * kernel, split-KV partials merged by log-sum-exp) for one block's cache, but
 * keeps all its scratch (KV tile list, partial outputs, status word) in a
 * 32 MiB array inside the library, which every GPU that runs it holds until
 * the process exits.  It calls no cudaMalloc / cudaFree.
 *   cache_block: device [pages][2][page_size][H][D] of `dtype` (one block).
 *   page_ids, valid_lens: HOST arrays of n_pages entries, in attention order;
 *     each id must address a page of cache_block, 1 <= valid_lens[i] <=
 *     page_size.  Q, out: device [n_q, H, D].  sm_scale 0 => 1/sqrt(D).
 * Limits: n_pages <= 1024 and at most 16384 KV tiles (64 rows each, 32 for
 * head_dim 128), else KVC_ERR_TOO_LARGE; the number of KV splits is cut to
 * what fits in the array.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept with the CUDA
 * context it belongs to: after cudaDeviceReset (or any other replacement of
 * the device's context) the next call looks it up again, so it too must come
 * before any capture.  Every call shares the one array, so
 * calls whose work overlaps on the GPU (other streams, other threads) race:
 * serialise them.  The status word is cleared on every call. */
int kvc_paged_attention_static(const void* cache_block, int32_t dtype, int32_t num_heads,
                               int32_t head_dim, int32_t page_size, const int32_t* page_ids,
                               const int32_t* valid_lens, int32_t n_pages, const void* Q, void* out,
                               int32_t n_q, float sm_scale, kvc_stream stream);

/* Shape of the handle's latest attention launch (kvc_run, or kvc_run_batch
 * with this handle first): 128-row query tiles per CTA of the tensor-core
 * kernel (0 for the CUDA-core kernel) and KV splits.  Diagnostics. */
int kvc_get_launch_shape(const kvc_handle* h, int32_t* q_tiles, int32_t* splits);

/* KV tiles of the current plan and whether they are packed (1: tiles of 128
 * rows cross page boundaries, see KVC_OPT_PACK_TILES; 0: one page per tile).
 * KVC_ERR_NO_PLAN before the first kvc_plan.  Diagnostics. */
int kvc_get_plan_tiles(const kvc_handle* h, int32_t* n_tiles, int32_t* packed);

/* Static message for a status code. */
const char* kvc_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H_ */
