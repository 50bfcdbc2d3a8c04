// kvc_paged_attention_static: paged attention that allocates nothing.
//
// Some callers cannot allocate device memory at all: code running inside a
// host framework that owns every byte of GPU memory and only lends out the KV
// cache and the Q / output buffers, plug-ins whose memory budget is fixed
// before they are loaded, or code that must not call cudaMalloc while other
// work is in flight on the device.  Such callers cannot give kvc_create a
// workspace.  This entry point runs the same paged attention (the CUDA-core
// kernel plus the split-KV merge) with its scratch -- the KV tile list, the
// split partial outputs and their log2-sum-exp, a status word -- in one
// file-scope device array of kScratchBytes.  The caller passes only the cache,
// the visible page list (host arrays) and Q / out.
//
// Host code must not hand the array's name to a kernel: in host code that
// name is a host-side stand-in, not a device address.  The device address is
// taken once per device with cudaGetSymbolAddress while that device is
// current (setup_device below) and passed to the kernels.  It is remembered
// together with the context it was taken in: if that context is destroyed and
// a new one made (cudaDeviceReset), the module is loaded again, possibly at
// another address, and the next call looks the address up again.
#include "kvc.h"
#include "kvc_internal.h"

#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

namespace kvc {
namespace {

// 32 MiB of scratch, held by every GPU on which this module is loaded until
// the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr size_t kStatusBytes = 256;
constexpr int kMaxStaticPages = 1024;
constexpr int kMaxStaticTiles = 16384;
constexpr size_t kTilesBytes = sizeof(KvTile) * kMaxStaticTiles;
constexpr size_t kPartialBase = kStatusBytes + kTilesBytes;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_dev[kMaxDevices];   // device address per device, once set up
CUcontext g_scratch_ctx[kMaxDevices];        // the context that address belongs to
int g_num_sms[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's current context, through the runtime's entry-point query (no
// link against the driver library).
bool current_context(CUcontext* ctx) {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  *ctx = nullptr;
  return fn && fn(ctx) == CUDA_SUCCESS && *ctx != nullptr;
}

// Once per device (and again if its context was replaced), with that device
// current: the array's device address and the SM count.
int setup_device(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  // Before the runtime's first call on this thread there may be no current
  // context yet; the symbol lookup below makes the device's context current.
  CUcontext ctx = nullptr;
  if (current_context(&ctx) && g_scratch_dev[dev] && g_scratch_ctx[dev] == ctx) return KVC_OK;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return KVC_ERR_CUDA;
  if (!current_context(&ctx)) return KVC_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVC_ERR_CUDA;
  g_num_sms[dev] = sms;
  g_scratch_dev[dev] = static_cast<unsigned char*>(p);
  g_scratch_ctx[dev] = ctx;
  return KVC_OK;
}

// The caller's page list, passed by value: page ids, valid rows and the index
// of each page's first tile.
struct StaticPages {
  int32_t n_pages;
  int32_t tile_rows;
  int32_t ids[kMaxStaticPages];
  int32_t valid[kMaxStaticPages];
  int32_t tile0[kMaxStaticPages];
};

__global__ void static_tiles_kernel(const __grid_constant__ StaticPages p, KvTile* __restrict__ tiles) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n_pages; i += gridDim.x * blockDim.x) {
    int32_t token0 = 0;   // token positions are informational only
    for (int32_t t = 0, r0 = 0; r0 < p.valid[i]; ++t, r0 += p.tile_rows) {
      KvTile k;
      k.page = p.ids[i];
      k.row0 = r0;
      k.rows = min(p.tile_rows, p.valid[i] - r0);
      k.token0 = token0 + r0;
      k.page2 = -1;
      k.row0_2 = 0;
      k.rows2 = 0;
      k.pad = 0;
      tiles[p.tile0[i] + t] = k;
    }
  }
}

StaticPages g_pages_arg;   // host staging of the kernel argument (guarded below)
std::mutex g_call_mutex;

}  // namespace
}  // namespace kvc

extern "C" int kvc_paged_attention_static(const void* cache_block, int32_t dtype, int32_t num_heads,
                                          int32_t head_dim, int32_t page_size, const int32_t* page_ids,
                                          const int32_t* valid_lens, int32_t n_pages, const void* Q,
                                          void* out, int32_t n_q, float sm_scale, kvc_stream stream) {
  using namespace kvc;
  // Host-side checks first: nothing below touches the device until they pass.
  if (dtype < KVC_BF16 || dtype > KVC_F32) return KVC_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return KVC_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > 4096 || page_size < 1 || n_q < 0) return KVC_ERR_INVALID_ARG;
  if (n_pages < 1 || !page_ids || !valid_lens) return KVC_ERR_INVALID_ARG;
  if (n_pages > kMaxStaticPages) return KVC_ERR_TOO_LARGE;
  if (!(sm_scale >= 0.0f) || !std::isfinite(sm_scale)) return KVC_ERR_INVALID_ARG;
  const int tr = simt_tile_rows(head_dim);
  int64_t n_tiles = 0;
  for (int32_t i = 0; i < n_pages; ++i) {
    if (page_ids[i] < 0 || valid_lens[i] < 1 || valid_lens[i] > page_size) return KVC_ERR_INVALID_ARG;
    n_tiles += (valid_lens[i] + tr - 1) / tr;
  }
  if (n_tiles > kMaxStaticTiles) return KVC_ERR_TOO_LARGE;
  if (n_q == 0) return KVC_OK;
  if (!cache_block || !Q || !out || ((uintptr_t)Q & 15u) || ((uintptr_t)out & 15u) ||
      ((uintptr_t)cache_block & 15u))
    return KVC_ERR_INVALID_ARG;
  const int64_t elem = dtype == KVC_F32 ? 4 : 2;
  if (((int64_t)num_heads * head_dim * elem) % 16 != 0) return KVC_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVC_ERR_INVALID_ARG;
  int rc = setup_device(dev);
  if (rc) return rc;
  unsigned char* scratch = g_scratch_dev[dev];
  cudaStream_t st = (cudaStream_t)stream;

  // Split-KV partials must fit in what is left of the array; one split needs none.
  const size_t per_split = (size_t)n_q * num_heads * (head_dim + 1) * sizeof(float);
  int64_t fit = (int64_t)((kScratchBytes - kPartialBase) / per_split);
  const int64_t base = (int64_t)((n_q + 127) / 128) * num_heads;
  const int64_t slots = (int64_t)g_num_sms[dev] * 2;
  int splits = 1;
  double best = 1e300;
  const int64_t max_s = std::min<int64_t>(std::min<int64_t>(fit, n_tiles), 256);
  for (int s = 1; s <= max_s; ++s) {
    const int64_t waves = (base * s + slots - 1) / slots;
    const int64_t per = (n_tiles + s - 1) / s;
    const double cost = (double)waves * per * (1.0 + (s > 1 ? 0.02 * s : 0.0));
    if (cost < best - 1e-9) { best = cost; splits = s; }
  }

  std::lock_guard<std::mutex> lock(g_call_mutex);
  StaticPages& p = g_pages_arg;
  p.n_pages = n_pages;
  p.tile_rows = tr;
  int32_t t0 = 0;
  for (int32_t i = 0; i < n_pages; ++i) {
    p.ids[i] = page_ids[i];
    p.valid[i] = valid_lens[i];
    p.tile0[i] = t0;
    t0 += (valid_lens[i] + tr - 1) / tr;
  }
  // The status word must start at zero; tiles and partials are fully written
  // before they are read.
  if (cudaMemsetAsync(scratch, 0, kStatusBytes, st) != cudaSuccess) return KVC_ERR_CUDA;
  KvTile* tiles = reinterpret_cast<KvTile*>(scratch + kStatusBytes);
  static_tiles_kernel<<<(n_pages + 127) / 128, 128, 0, st>>>(p, tiles);
  if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;

  AttnArgs a;
  a.pdl = 0;
  a.q = Q;
  a.out = out;
  a.cache = cache_block;
  a.tiles = tiles;
  a.part_o = reinterpret_cast<float*>(scratch + kPartialBase);
  a.part_lse = reinterpret_cast<float*>(scratch + kPartialBase +
                                        (size_t)splits * n_q * num_heads * head_dim * sizeof(float));
  a.status = reinterpret_cast<int32_t*>(scratch);
  a.n_q = n_q;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.page_size = page_size;
  a.n_tiles = (int32_t)n_tiles;
  a.n_splits = splits;
  a.max_pages = 0x7fffffff;   // the caller's cache extent is not known here
  const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / std::sqrt((float)head_dim);
  a.sm_scale_log2 = scale * 1.4426950408889634f;
  a.wait_budget = 4000000000LL;
  a.stall_test = 0;
  if (launch_attn_simt(a, dtype, st) != cudaSuccess) return KVC_ERR_CUDA;
  if (splits > 1 && launch_merge(a, dtype, st) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}
