// CUDA kernels of libkvc.so other than the tensor-core attention:
//   append_kernel    -- scatter of one frame's K/V into its patch page and the
//                       special stream (16-byte vector copies)
//   plan_kernel      -- device page table, per-page valid lengths, KV tile list
//   attn_simt_kernel -- paged attention on the CUDA cores (fp32 math), used for
//                       fp32 caches and for head sizes without a tensor-core path
//   merge_kernel     -- log-sum-exp merge of split-KV partial outputs
//
// Pages cited by tag, then section:
//   [KVC]   "How LingBot-Map Implements the KV Cache Mechanism for Streaming
//           Inference with FlashInfer Integration"
//   [SLOTS] "LingBot-Map KV缓存机制深度揭秘：scale frames与keyframes如何占用slot"

#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace kvc {
namespace {

// ----------------------------------------------------------------- append
// One frame's K/V [6 + ps, H, D]: rows 0..5 (camera, 4 registers, scale) go to
// slots [special_slot, +6) of the special page, rows 6.. fill the patch page
// ([SLOTS] "双流分页布局", "特殊 token 流"; [KVC] "Append and Evict API").
// With a camera stream (camera_page >= 0), row 0 is also copied to row
// camera_slot of the camera page.
// grid = (ceil(row16 / blockDim), 2 * (6 + ps + cam)); one thread moves 16 bytes.
__global__ void append_kernel(char* __restrict__ cache_block, const char* __restrict__ K,
                              const char* __restrict__ V, int32_t page, int32_t special_page,
                              int32_t special_slot, int32_t camera_page, int32_t camera_slot,
                              int32_t page_size, int64_t row_bytes, int32_t max_pages,
                              int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  const int32_t T = kNumSpecial + page_size;
  if (KVC_CHECKED && (page < 0 || page >= max_pages || special_page < 0 || special_page >= max_pages ||
                      special_slot < 0 || special_slot + kNumSpecial > page_size ||
                      (camera_page >= 0 && (camera_page >= max_pages || camera_slot < 0 ||
                                            camera_slot >= page_size)))) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) record_bounds(status, 101, page);
    return;
  }
  const int32_t rows = T + (camera_page >= 0 ? 1 : 0);
  const int32_t kv = blockIdx.y / rows;
  const int32_t r = blockIdx.y - kv * rows;
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c * 16 >= row_bytes) return;
  const char* src = (kv ? V : K) + (int64_t)(r < T ? r : 0) * row_bytes + c * 16;
  int64_t dst_row;
  if (r == T)
    dst_row = ((int64_t)camera_page * 2 + kv) * page_size + camera_slot;
  else if (r < kNumSpecial)
    dst_row = ((int64_t)special_page * 2 + kv) * page_size + special_slot + r;
  else
    dst_row = ((int64_t)page * 2 + kv) * page_size + (r - kNumSpecial);
  uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
  *reinterpret_cast<uint4*>(cache_block + dst_row * row_bytes + c * 16) = v;
}

// ------------------------------------------------------------------- plan
// Visible order: scale pages, live window, then the pages of the special
// (and camera) runs; every page contributes rows [row0, row0 + valid)
// ([KVC] "Patch Pages vs. Special Pages"; [SLOTS] "双流分页布局").  With the
// default special policy there is one run, every special page from row 0, a
// non-last page holding 6*fpp tokens and the last last_page_len.

__device__ __forceinline__ int32_t cdiv(int32_t x, int32_t u) { return (x + u - 1) / u; }

// Entry e of the visible list: page id, first row, valid rows, and where it
// starts in units of u rows (every entry rounded up to whole units) and in
// tokens.  Only a run's first and last page can be partial, so the offsets
// have a closed form.  e == the entry count gives the totals (id -1).
struct PlanEntry {
  int32_t id, row0, v, unit0, token0;
};

__device__ PlanEntry plan_entry(const PlanArgs& a, int32_t e, int32_t u) {
  PlanEntry x;
  if (e < a.n_patch) {
    x.id = a.patch_ids[e];
    x.row0 = 0;
    x.v = a.page_size;
    x.unit0 = e * cdiv(a.page_size, u);
    x.token0 = e * a.page_size;
    return x;
  }
  int32_t entry = a.n_patch, unit = a.n_patch * cdiv(a.page_size, u), token = a.n_patch * a.page_size;
  for (int32_t r = 0; r < a.n_runs; ++r) {
    const PlanRun& run = a.runs[r];
    const int32_t n = run_pages(run);
    if (n == 0) continue;
    int32_t id, row0, v0, vf, vl;
    run_entry(run, 0, &id, &row0, &v0);
    run_entry(run, n > 1 ? 1 : 0, &id, &row0, &vf);
    if (e < entry + n) {
      const int32_t k = e - entry;
      run_entry(run, k, &x.id, &x.row0, &x.v);
      x.unit0 = unit + (k == 0 ? 0 : cdiv(v0, u) + (k - 1) * cdiv(vf, u));
      x.token0 = token + (k == 0 ? 0 : v0 + (k - 1) * vf);
      return x;
    }
    run_entry(run, n - 1, &id, &row0, &vl);
    unit += n == 1 ? cdiv(v0, u) : cdiv(v0, u) + (n - 2) * cdiv(vf, u) + cdiv(vl, u);
    token += n == 1 ? v0 : v0 + (n - 2) * vf + vl;
    entry += n;
  }
  x.id = -1;
  x.row0 = x.v = 0;
  x.unit0 = unit;
  x.token0 = token;
  return x;
}

// Tiles: without packing, every entry is cut into tiles of tile_rows rows.
// Packed (tensor-core plans whose entries but the last have >= 15 units of 8
// rows): tile t covers units [16 t, 16 t + 16) of the concatenated entries;
// the entry holding unit 16 t writes it -- its own rows from there, and, if
// the tile has room left, the next entry's first rows.
__global__ void plan_kernel(const __grid_constant__ PlanArgs a, char* __restrict__ ws,
                            WorkspaceLayout L) {
  pdl_trigger();
  pdl_wait();
  const int32_t tr = a.tile_rows;
  const int32_t u = a.pack ? kPackUnitRows : tr;     // unit of the tile offsets
  const int32_t per_tile = tr / u;                   // units per tile
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.page_ids);
  int32_t* valid = reinterpret_cast<int32_t*>(ws + L.page_valid);
  int32_t* first = reinterpret_cast<int32_t*>(ws + L.page_row0);
  KvTile* tiles = reinterpret_cast<KvTile*>(ws + L.tiles);
  int32_t n_entries = a.n_patch;
  for (int32_t r = 0; r < a.n_runs; ++r) n_entries += run_pages(a.runs[r]);
  const PlanEntry end = plan_entry(a, n_entries, u);
  const int32_t n_tiles = cdiv(end.unit0, per_tile);
  for (int32_t e = threadIdx.x; e < n_entries; e += blockDim.x) {
    const PlanEntry x = plan_entry(a, e, u);
    const int32_t t_lo = cdiv(x.unit0, per_tile), t_hi = cdiv(x.unit0 + cdiv(x.v, u), per_tile);
    if (KVC_CHECKED && (e >= L.max_pages || x.id < 0 || x.id >= a.max_pages || x.row0 < 0 || x.v < 1 ||
                        x.row0 + x.v > a.page_size || t_hi > L.max_tiles)) {
      record_bounds(reinterpret_cast<int32_t*>(ws + L.status), 201, e);
      continue;
    }
    ids[e] = x.id;
    valid[e] = x.v;
    first[e] = x.row0;
    PlanEntry y;
    y.id = -1;
    if (a.pack && e + 1 < n_entries) y = plan_entry(a, e + 1, u);
    for (int32_t t = t_lo; t < t_hi; ++t) {
      const int32_t r0 = (t * per_tile - x.unit0) * u;   // first row of the tile within the entry
      KvTile k;
      k.page = x.id;
      k.row0 = x.row0 + r0;
      k.rows = min(tr, x.v - r0);
      k.token0 = x.token0 + r0;
      k.page2 = -1;
      k.row0_2 = 0;
      k.rows2 = 0;
      k.pad = 0;
      const int32_t room = tr - cdiv(k.rows, u) * u;    // packed: rows left after whole units
      if (a.pack && room > 0 && y.id >= 0) {
        k.page2 = y.id;
        k.row0_2 = y.row0;
        k.rows2 = min(room, y.v);
      }
      tiles[t] = k;
    }
  }
  if (threadIdx.x == 0) {
    DevPlanHeader h;
    h.n_pages = n_entries;
    h.last_page_len = n_entries > 0 ? plan_entry(a, n_entries - 1, u).v : 0;
    h.n_tiles = n_tiles;
    h.n_tokens = end.token0;
    *reinterpret_cast<DevPlanHeader*>(ws + L.header) = h;
  }
}

// -------------------------------------------------------- element helpers
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// ------------------------------------------------------ CUDA-core attention
// One thread per query row, one CTA per (128-row query tile, head, KV split).
// K/V tiles of BN rows are staged in shared memory as fp32; scores and the
// online softmax are fp32, in the log2 domain (scores pre-multiplied by
// sm_scale * log2 e).  Output: final O (one split) or the split's normalised
// partial O and its log2-sum-exp.
constexpr int kSimtThreads = 128;

template <typename T, int D, int BN>
__global__ void __launch_bounds__(kSimtThreads)
attn_simt_kernel(const AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sK[BN][D];
  __shared__ float sV[BN][D];
  const int h = blockIdx.y;
  const int split = blockIdx.z;
  const int row = blockIdx.x * kSimtThreads + threadIdx.x;
  const bool active = row < a.n_q;
  const int H = a.num_heads;
  const int64_t row_elems = (int64_t)H * D;
  const T* qp = reinterpret_cast<const T*>(a.q) + ((int64_t)(active ? row : 0) * H + h) * D;
  float q[D];
#pragma unroll
  for (int d = 0; d < D; ++d) q[d] = to_f(qp[d]) * a.sm_scale_log2;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int t0 = (int)(((int64_t)split * a.n_tiles) / a.n_splits);
  const int t1 = (int)(((int64_t)(split + 1) * a.n_tiles) / a.n_splits);
  const T* cache = reinterpret_cast<const T*>(a.cache);
  for (int t = t0; t < t1; ++t) {
    const KvTile tile = a.tiles[t];
    if (KVC_CHECKED && (tile.page < 0 || tile.page >= a.max_pages || tile.row0 < 0 || tile.rows < 1 ||
                        tile.rows > BN || tile.row0 + tile.rows > a.page_size)) {
      if (threadIdx.x == 0) record_bounds(a.status, 301, t);
      continue;                                        // uniform over the CTA: skip the tile
    }
    const int64_t kbase = (((int64_t)tile.page * 2 + 0) * a.page_size + tile.row0) * row_elems + (int64_t)h * D;
    const int64_t vbase = (((int64_t)tile.page * 2 + 1) * a.page_size + tile.row0) * row_elems + (int64_t)h * D;
    for (int idx = threadIdx.x; idx < tile.rows * D; idx += kSimtThreads) {
      const int r = idx / D, d = idx - r * D;
      sK[r][d] = to_f(cache[kbase + (int64_t)r * row_elems + d]);
      sV[r][d] = to_f(cache[vbase + (int64_t)r * row_elems + d]);
    }
    __syncthreads();
    if (active) {
      // Keys in chunks of 8: scores, chunk max, rescale, accumulate.
      for (int j0 = 0; j0 < tile.rows; j0 += 8) {
        float s[8];
        float cmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          float x = -INFINITY;
          if (j < tile.rows) {
            x = 0.f;
#pragma unroll
            for (int d = 0; d < D; ++d) x = fmaf(q[d], sK[j][d], x);
          }
          s[jj] = x;
          cmax = fmaxf(cmax, x);
        }
        const float m_new = fmaxf(m, cmax);
        const float alpha = exp2f(m - m_new);
        l *= alpha;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] *= alpha;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          if (j < tile.rows) {
            const float p = exp2f(s[jj] - m_new);
            l += p;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = fmaf(p, sV[j][d], acc[d]);
          }
        }
        m = m_new;
      }
    }
    __syncthreads();
  }
  if (!active) return;
  const float inv = 1.f / l;
  if (a.n_splits == 1) {
    T* op = reinterpret_cast<T*>(a.out) + ((int64_t)row * H + h) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) op[d] = from_f<T>(acc[d] * inv);
  } else {
    float* po = a.part_o + (((int64_t)split * a.n_q + row) * H + h) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) po[d] = acc[d] * inv;
    a.part_lse[((int64_t)split * a.n_q + row) * H + h] = m + log2f(l);
  }
}

// -------------------------------------------------------------- LSE merge
// out = sum_s 2^(lse_s - lse) O_s with lse = log2 sum_s 2^lse_s
// ([KVC] "Kernel-Level Execution Flow": the split-KV partials of one query row
// and head combined by their log-sum-exp).  D / 4 threads per (query row, head),
// one float4 of the head dimension each, so a (row, head) is one contiguous
// 4 D-byte read per split; the split loop is unrolled to keep several splits'
// loads in flight.
template <typename T, int D>
__global__ void merge_kernel(const AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int TPR = D / 4;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rh = gid / TPR;                      // row * H + head
  const int c = (int)(gid - rh * TPR);
  const int64_t n_rh = (int64_t)a.n_q * a.num_heads;
  if (rh >= n_rh) return;
  const float* lse = a.part_lse + rh;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + rh * D) + c;
  const int64_t po_stride = n_rh * (D / 4);
  // One pass with a running max: each split's weight and partial are loaded
  // together, so the unrolled loop keeps several splits' loads in flight.
  float mx = -INFINITY, wsum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < a.n_splits; ++s) {
    const float l_s = __ldg(lse + s * n_rh);
    const float4 p = __ldg(po + s * po_stride);
    const float m_new = fmaxf(mx, l_s);
    const float scale = exp2f(mx - m_new);         // 0 on the first split
    const float wt = exp2f(l_s - m_new);
    mx = m_new;
    wsum = fmaf(wsum, scale, wt);
    o.x = fmaf(wt, p.x, o.x * scale);
    o.y = fmaf(wt, p.y, o.y * scale);
    o.z = fmaf(wt, p.z, o.z * scale);
    o.w = fmaf(wt, p.w, o.w * scale);
  }
  const float inv = 1.f / wsum;
  T* op = reinterpret_cast<T*>(a.out) + rh * D + 4 * c;
  if constexpr (sizeof(T) == 2) {                    // one 8-byte store
    union { T t[4]; uint2 u; } w;
    w.t[0] = from_f<T>(o.x * inv);
    w.t[1] = from_f<T>(o.y * inv);
    w.t[2] = from_f<T>(o.z * inv);
    w.t[3] = from_f<T>(o.w * inv);
    *reinterpret_cast<uint2*>(op) = w.u;
  } else {
    *reinterpret_cast<float4*>(op) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  }
}

template <typename T, int D>
cudaError_t simt_dispatch(const AttnArgs& a, cudaStream_t st) {
  constexpr int BN = D >= 128 ? 32 : 64;
  dim3 grid((a.n_q + kSimtThreads - 1) / kSimtThreads, a.num_heads, a.n_splits);
  return launch_kernel(attn_simt_kernel<T, D, BN>, grid, dim3(kSimtThreads), 0, st, a.pdl != 0, a);
}

template <typename T>
cudaError_t simt_by_dim(const AttnArgs& a, cudaStream_t st) {
  switch (a.head_dim) {
    case 32: return simt_dispatch<T, 32>(a, st);
    case 64: return simt_dispatch<T, 64>(a, st);
    case 128: return simt_dispatch<T, 128>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t merge_by_dim(const AttnArgs& a, cudaStream_t st) {
  const int64_t n_rh = (int64_t)a.n_q * a.num_heads;
  const int threads = 256;
  // D / 4 threads per (row, head)
  const unsigned blocks = (unsigned)((n_rh * (a.head_dim / 4) + threads - 1) / threads);
  if (blocks == 0) return cudaSuccess;
  const bool pdl = a.pdl != 0;
  switch (a.head_dim) {
    case 32: return launch_kernel(merge_kernel<T, 32>, dim3(blocks), dim3(threads), 0, st, pdl, a);
    case 64: return launch_kernel(merge_kernel<T, 64>, dim3(blocks), dim3(threads), 0, st, pdl, a);
    case 128: return launch_kernel(merge_kernel<T, 128>, dim3(blocks), dim3(threads), 0, st, pdl, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int simt_tile_rows(int head_dim) { return head_dim >= 128 ? 32 : 64; }

cudaError_t launch_append(void* cache_block, const void* K, const void* V, int32_t page,
                          int32_t special_page, int32_t special_slot, int32_t camera_page,
                          int32_t camera_slot, int32_t page_size, int64_t row_bytes, int32_t max_pages,
                          int32_t* status, cudaStream_t stream, bool pdl) {
  const int64_t row16 = row_bytes / 16;
  const int threads = row16 >= 128 ? 128 : (int)((row16 + 31) / 32 * 32);
  const unsigned rows = (unsigned)(kNumSpecial + page_size + (camera_page >= 0 ? 1 : 0));
  dim3 grid((unsigned)((row16 + threads - 1) / threads), 2u * rows);
  return launch_kernel(append_kernel, grid, dim3(threads), 0, stream, pdl, static_cast<char*>(cache_block),
                       static_cast<const char*>(K), static_cast<const char*>(V), page, special_page,
                       special_slot, camera_page, camera_slot, page_size, row_bytes, max_pages, status);
}

cudaError_t launch_plan(const PlanArgs& a, void* workspace, const WorkspaceLayout& L,
                        cudaStream_t stream, bool pdl) {
  return launch_kernel(plan_kernel, dim3(1), dim3(256), 0, stream, pdl, a, static_cast<char*>(workspace), L);
}

cudaError_t launch_attn_simt(const AttnArgs& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return simt_by_dim<__nv_bfloat16>(a, stream);
    case 1: return simt_by_dim<__half>(a, stream);
    case 2: return simt_by_dim<float>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(const AttnArgs& a, int dtype, cudaStream_t stream) {
  switch (dtype) {
    case 0: return merge_by_dim<__nv_bfloat16>(a, stream);
    case 1: return merge_by_dim<__half>(a, stream);
    case 2: return merge_by_dim<float>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvc
