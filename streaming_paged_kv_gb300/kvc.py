"""ctypes binding of libkvc.so (include/kvc.h), same names as the C ABI.

Argument marshalling only: every step of the cache and of the attention runs
in the C++/CUDA library.  Importing this module loads ``libkvc.so`` and raises
ImportError if it has not been built (``streaming_paged_kv_gb300.build``);
there is no fallback.

``PagedKVCache`` is a convenience owner: it allocates the cache and the
workspace as torch device tensors (PyTorch supplies device memory and
streams), creates the handle and forwards torch tensors' pointers.
"""

import ctypes
import os
import sys

_PKG = os.path.dirname(os.path.abspath(__file__))
# KVC_CHECKED=1 selects the build with device-side bounds checks; KVC_LIB names
# another build of the same library (the sanitizer test's host build).
LIB_PATH = os.environ.get("KVC_LIB") or os.path.join(
    _PKG, "libkvc_checked.so" if os.environ.get("KVC_CHECKED") == "1" else "libkvc.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run streaming_paged_kv_gb300.build.build()")
lib = ctypes.CDLL(LIB_PATH)

KVC_BF16, KVC_F16, KVC_F32 = 0, 1, 2
DTYPE_CODE = {"bf16": KVC_BF16, "f16": KVC_F16, "f32": KVC_F32}

ERRORS = {
    0: "OK", -1: "INVALID_ARG", -2: "NO_FREE_PAGE", -3: "SPECIAL_POOL_FULL",
    -4: "NOTHING_TO_ROLLBACK", -5: "ROLLBACK_AFTER_EVICT", -6: "NO_PLAN", -7: "STALE_PLAN",
    -8: "CUDA", -9: "DEVICE_TIMEOUT", -10: "EMPTY", -11: "NO_DEVICE", -12: "TOO_LARGE",
    -13: "DEVICE_BOUNDS",
}
KVC_OPT_ATTN_KERNEL, KVC_OPT_NUM_SPLITS, KVC_OPT_WAIT_BUDGET, KVC_OPT_TIMING, KVC_OPT_STALL_TEST = 1, 2, 3, 4, 5
KVC_OPT_QUERY_TILES = 6
KVC_OPT_PACK_TILES = 7
KVC_OPT_PDL = 8

try:
    _DEBUG_EVERY = max(0, int(os.environ.get("KVC_DEBUG", "0") or 0))   # see PagedKVCache.plan
except ValueError:
    _DEBUG_EVERY = 0
KVC_SPECIAL_NO_CROSS_FRAME, KVC_SPECIAL_CAMERA_ONLY = 1, 2


class kvc_config(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_special_tokens", ctypes.c_int32), ("scale_frames", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32), ("headroom", ctypes.c_int32),
        ("max_total_frames", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("max_query_tokens", ctypes.c_int32),
        ("max_kv_splits", ctypes.c_int32), ("special_policy", ctypes.c_int32),
    ]


class kvc_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("frame_count", "scale_pages", "live_pages", "free_pages", "special_tokens")]


class KvcError(RuntimeError):
    def __init__(self, rc, call=""):
        self.rc = rc
        self.code = ERRORS.get(rc, str(rc))
        msg = lib.kvc_strerror(rc).decode()
        super().__init__(f"{call}: {self.code} ({msg})" if call else f"{self.code} ({msg})")


class Geometry(ctypes.Structure):
    _fields_ = [("num_patch_pages", ctypes.c_int32), ("frames_per_special_page", ctypes.c_int32),
                ("num_special_pages", ctypes.c_int32), ("num_camera_pages", ctypes.c_int32),
                ("max_num_pages", ctypes.c_int32),
                ("tokens_per_frame", ctypes.c_int32), ("page_bytes", ctypes.c_int64),
                ("block_bytes", ctypes.c_int64)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_PI32 = ctypes.POINTER(ctypes.c_int32)
_SIGS = {
    "kvc_required_bytes": [ctypes.POINTER(kvc_config), ctypes.POINTER(ctypes.c_size_t),
                           ctypes.POINTER(ctypes.c_size_t)],
    "kvc_get_geometry": [ctypes.POINTER(kvc_config), ctypes.POINTER(Geometry)],
    "kvc_create": [ctypes.POINTER(kvc_config), _P, _P, _P, ctypes.POINTER(_P)],
    "kvc_destroy": [_P],
    "kvc_append_frame": [_P, _I32, _P, _P, _P],
    "kvc_evict_frames": [_P, _I32, _I32, _I32],
    "kvc_evict_frames_ex": [_P, _I32, _I32, _I32, _I32, _I32],
    "kvc_set_defer_eviction": [_P, _I32],
    "kvc_execute_deferred_eviction": [_P, _I32, _I32, _I32],
    "kvc_rollback_last_frame": [_P, _I32],
    "kvc_clean": [_P],
    "kvc_plan": [_P, _P],
    "kvc_run": [_P, _I32, _P, _P, _I32, _P],
    "kvc_prefill": [_P, _I32, _P, _P, _P, _I32, _P, _P],
    "kvc_run_batch": [ctypes.POINTER(_P), _PI32, _I32, _P, _P, _PI32, _P],
    "kvc_get_cache_stats": [_P, _I32, ctypes.POINTER(kvc_stats)],
    "kvc_get_plan": [_P, _PI32, _PI32, _I32, _PI32, _PI32],
    "kvc_get_plan_ranges": [_P, _PI32, _PI32, _PI32, _I32, _PI32],
    "kvc_read_device_ranges": [_P, _PI32, _PI32, _PI32, _I32, _PI32, _P],
    "kvc_get_deques": [_P, _I32, _PI32, _PI32, _PI32, _PI32, _PI32, _PI32],
    "kvc_read_device_plan": [_P, _PI32, _PI32, _I32, _PI32, _PI32, _P],
    "kvc_device_status": [_P, _P],
    "kvc_set_option": [_P, _I32, _I64],
    "kvc_get_counters": [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                         ctypes.POINTER(ctypes.c_double), _I32],
    "kvc_get_launch_shape": [_P, _PI32, _PI32],
    "kvc_get_plan_tiles": [_P, _PI32, _PI32],
    "kvc_paged_attention_static": [_P, _I32, _I32, _I32, _I32, _PI32, _PI32, _I32, _P, _P, _I32,
                                   ctypes.c_float, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.kvc_strerror.argtypes = [ctypes.c_int]
lib.kvc_strerror.restype = ctypes.c_char_p


def _check(rc, call):
    if rc != 0:
        raise KvcError(rc, call)
    return rc


def special_policy(cross_frame_special=True, camera_only=False):
    """kvc_config.special_policy for the two eviction options."""
    return (0 if cross_frame_special else KVC_SPECIAL_NO_CROSS_FRAME) | \
        (KVC_SPECIAL_CAMERA_ONLY if camera_only else 0)


def make_config(num_blocks, num_heads, head_dim, page_size, dtype="bf16", scale_frames=8,
                sliding_window=64, headroom=16, max_total_frames=2048, sm_scale=0.0,
                max_query_tokens=0, max_kv_splits=0, cross_frame_special=True, camera_only=False):
    """kvc_config with the pages' defaults (8 / 64 / 16 / 2048)."""
    return kvc_config(num_blocks, num_heads, head_dim, page_size, 6, scale_frames,
                      sliding_window, headroom, max_total_frames, DTYPE_CODE[dtype],
                      float(sm_scale), max_query_tokens, max_kv_splits,
                      special_policy(cross_frame_special, camera_only))


# ----------------------------------------------------- same-name wrappers
def kvc_required_bytes(cfg):
    c, w = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib.kvc_required_bytes(ctypes.byref(cfg), ctypes.byref(c), ctypes.byref(w)),
           "kvc_required_bytes")
    return c.value, w.value


def kvc_get_geometry(cfg):
    g = Geometry()
    _check(lib.kvc_get_geometry(ctypes.byref(cfg), ctypes.byref(g)), "kvc_get_geometry")
    return g


def kvc_create(cfg, cache_ptr=None, workspace_ptr=None, stream=None):
    h = _P()
    _check(lib.kvc_create(ctypes.byref(cfg), cache_ptr, workspace_ptr, stream, ctypes.byref(h)),
           "kvc_create")
    return h


def kvc_destroy(h):
    return _check(lib.kvc_destroy(h), "kvc_destroy")


def kvc_append_frame(h, block, k_ptr, v_ptr, stream=None):
    return _check(lib.kvc_append_frame(h, block, k_ptr, v_ptr, stream), "kvc_append_frame")


def kvc_evict_frames(h, block, scale_frames, sliding_window):
    return _check(lib.kvc_evict_frames(h, block, scale_frames, sliding_window), "kvc_evict_frames")


def kvc_evict_frames_ex(h, block, scale_frames, sliding_window, cross_frame_special, camera_only):
    return _check(lib.kvc_evict_frames_ex(h, block, scale_frames, sliding_window, int(bool(cross_frame_special)),
                                          int(bool(camera_only))), "kvc_evict_frames_ex")


def kvc_set_defer_eviction(h, on):
    return _check(lib.kvc_set_defer_eviction(h, int(bool(on))), "kvc_set_defer_eviction")


def kvc_execute_deferred_eviction(h, block, scale_frames, sliding_window):
    return _check(lib.kvc_execute_deferred_eviction(h, block, scale_frames, sliding_window),
                  "kvc_execute_deferred_eviction")


def kvc_rollback_last_frame(h, block):
    return _check(lib.kvc_rollback_last_frame(h, block), "kvc_rollback_last_frame")


def kvc_clean(h):
    return _check(lib.kvc_clean(h), "kvc_clean")


def kvc_plan(h, stream=None):
    return _check(lib.kvc_plan(h, stream), "kvc_plan")


def kvc_run(h, block, q_ptr, out_ptr, n_q, stream=None):
    return _check(lib.kvc_run(h, block, q_ptr, out_ptr, n_q, stream), "kvc_run")


def kvc_prefill(h, block, q_ptr, k_ptr, v_ptr, n_frames, out_ptr, stream=None):
    return _check(lib.kvc_prefill(h, block, q_ptr, k_ptr, v_ptr, n_frames, out_ptr, stream), "kvc_prefill")


def kvc_run_batch(handles, blocks, q_ptr, out_ptr, qo_indptr, stream=None):
    n = len(handles)
    hs = (_P * n)(*handles)
    bl = (ctypes.c_int32 * n)(*blocks)
    qi = (ctypes.c_int32 * (n + 1))(*qo_indptr)
    return _check(lib.kvc_run_batch(hs, bl, n, q_ptr, out_ptr, qi, stream), "kvc_run_batch")


def run_batch(caches, blocks, q, out, rows):
    """Attention of several streams in one launch: request r is caches[r]
    (a PagedKVCache) block blocks[r] with the next rows[r] rows of the ragged
    q / out ([sum(rows), H, D]).  Returns out."""
    qo = [0]
    for n in rows:
        qo.append(qo[-1] + int(n))
    if len(rows) != len(caches) or qo[-1] != q.shape[0] or out.shape != q.shape:
        raise ValueError("rows must give one count per cache and add up to q's length")
    kvc_run_batch([c.h for c in caches], blocks, caches[0]._ptr(q), caches[0]._ptr(out), qo,
                  caches[0]._stream())
    return out


def kvc_get_cache_stats(h, block):
    s = kvc_stats()
    _check(lib.kvc_get_cache_stats(h, block, ctypes.byref(s)), "kvc_get_cache_stats")
    return {n: getattr(s, n) for n, _ in kvc_stats._fields_}


def kvc_get_plan(h, cap=4096):
    indptr = (ctypes.c_int32 * 2)()
    idx = (ctypes.c_int32 * cap)()
    n, lpl = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.kvc_get_plan(h, indptr, idx, cap, ctypes.byref(n), ctypes.byref(lpl)), "kvc_get_plan")
    return list(idx[:n.value]), [indptr[0], indptr[1]], lpl.value


def kvc_get_plan_ranges(h, cap=8192):
    bufs = [(ctypes.c_int32 * cap)() for _ in range(3)]
    n = ctypes.c_int32()
    _check(lib.kvc_get_plan_ranges(h, bufs[0], bufs[1], bufs[2], cap, ctypes.byref(n)), "kvc_get_plan_ranges")
    return tuple(list(b[:n.value]) for b in bufs)


def kvc_read_device_ranges(h, stream=None, cap=8192):
    bufs = [(ctypes.c_int32 * cap)() for _ in range(3)]
    n = ctypes.c_int32()
    _check(lib.kvc_read_device_ranges(h, bufs[0], bufs[1], bufs[2], cap, ctypes.byref(n), stream),
           "kvc_read_device_ranges")
    return tuple(list(b[:n.value]) for b in bufs)


def kvc_get_deques(h, block, cap=1024):
    bufs = [(ctypes.c_int32 * cap)() for _ in range(3)]
    ns = [ctypes.c_int32() for _ in range(3)]
    _check(lib.kvc_get_deques(h, block, bufs[0], ctypes.byref(ns[0]), bufs[1], ctypes.byref(ns[1]),
                              bufs[2], ctypes.byref(ns[2])), "kvc_get_deques")
    return tuple(list(b[:n.value]) for b, n in zip(bufs, ns))


def kvc_read_device_plan(h, stream=None, cap=4096):
    idx = (ctypes.c_int32 * cap)()
    valid = (ctypes.c_int32 * cap)()
    n, lpl = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.kvc_read_device_plan(h, idx, valid, cap, ctypes.byref(n), ctypes.byref(lpl), stream),
           "kvc_read_device_plan")
    return list(idx[:n.value]), list(valid[:n.value]), lpl.value


def kvc_device_status(h, stream=None):
    """Returns the status code (0 or -9) rather than raising."""
    return lib.kvc_device_status(h, stream)


def kvc_set_option(h, option, value):
    return _check(lib.kvc_set_option(h, option, int(value)), "kvc_set_option")


def kvc_get_counters(h, reset=False):
    a, b, ms = _I64(), _I64(), ctypes.c_double()
    _check(lib.kvc_get_counters(h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(ms), int(reset)),
           "kvc_get_counters")
    return a.value, b.value, ms.value


def kvc_paged_attention_static(cache_ptr, dtype, num_heads, head_dim, page_size, page_ids,
                               valid_lens, q_ptr, out_ptr, n_q, sm_scale=0.0, stream=None):
    """Paged attention with no allocation (scratch inside the library): for
    callers that cannot allocate device memory.  page_ids / valid_lens are
    host sequences; see include/kvc.h for the limits and the sharing rules."""
    n = len(page_ids)
    ids = (ctypes.c_int32 * max(n, 1))(*page_ids)
    valid = (ctypes.c_int32 * max(n, 1))(*valid_lens)
    return _check(lib.kvc_paged_attention_static(cache_ptr, DTYPE_CODE.get(dtype, dtype), num_heads,
                                                 head_dim, page_size, ids, valid, n, q_ptr, out_ptr,
                                                 n_q, float(sm_scale), stream),
                  "kvc_paged_attention_static")


def kvc_get_launch_shape(h):
    """(query tiles per CTA, KV splits) of the handle's latest attention launch."""
    qt, sp = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.kvc_get_launch_shape(h, ctypes.byref(qt), ctypes.byref(sp)), "kvc_get_launch_shape")
    return qt.value, sp.value


def kvc_get_plan_tiles(h):
    """(KV tiles, packed) of the handle's current plan."""
    n, packed = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.kvc_get_plan_tiles(h, ctypes.byref(n), ctypes.byref(packed)), "kvc_get_plan_tiles")
    return n.value, bool(packed.value)


def kvc_strerror(rc):
    return lib.kvc_strerror(rc).decode()


# ------------------------------------------------------- torch convenience
class PagedKVCache:
    """Owns the device cache + workspace (torch tensors) and a kvc handle.

    ``device=None`` makes a bookkeeping-only handle (no GPU needed).
    Methods take torch tensors and the current torch CUDA stream.
    """

    def __init__(self, num_blocks, num_heads, head_dim, page_size, dtype="bf16", scale_frames=8,
                 sliding_window=64, headroom=16, max_total_frames=2048, sm_scale=0.0,
                 max_query_tokens=0, max_kv_splits=0, device="cuda", cross_frame_special=True,
                 camera_only=False):
        self.cfg = make_config(num_blocks, num_heads, head_dim, page_size, dtype, scale_frames,
                               sliding_window, headroom, max_total_frames, sm_scale,
                               max_query_tokens, max_kv_splits, cross_frame_special, camera_only)
        self.cross_frame_special, self.camera_only = bool(cross_frame_special), bool(camera_only)
        self.dtype = dtype
        self.num_blocks, self.num_heads, self.head_dim = num_blocks, num_heads, head_dim
        self.page_size = page_size
        self.scale_frames, self.sliding_window = scale_frames, sliding_window
        geo = kvc_get_geometry(self.cfg)          # the library's page geometry
        self.num_patch_pages = geo.num_patch_pages
        self.frames_per_special_page = geo.frames_per_special_page
        self.num_special_pages = geo.num_special_pages
        self.num_camera_pages = geo.num_camera_pages
        self.max_num_pages = geo.max_num_pages
        self.cache_bytes, self.workspace_bytes = kvc_required_bytes(self.cfg)
        self.device = device
        self.cache = self.workspace = None
        if device is None:
            self.h = kvc_create(self.cfg)
        else:
            import torch
            self.cache = torch.empty(self.cache_bytes, dtype=torch.uint8, device=device)
            self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)
            self.h = kvc_create(self.cfg, self.cache.data_ptr(), self.workspace.data_ptr(),
                                self._stream())

    def _stream(self):
        if self.device is None:
            return None
        import torch
        return torch.cuda.current_stream().cuda_stream

    def _ptr(self, t):
        if t is None:
            return None
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()

    def cache_view(self, block):
        """The cache of one block as a torch tensor [pages, 2, ps, H, D] (raw view)."""
        import torch
        from .inputs import TORCH_DTYPE
        per = self.cache_bytes // self.num_blocks
        raw = self.cache[block * per:(block + 1) * per]
        return raw.view(TORCH_DTYPE[self.dtype]).view(
            self.max_num_pages, 2, self.page_size, self.num_heads, self.head_dim)

    def append_frame(self, block, k=None, v=None):
        kvc_append_frame(self.h, block, self._ptr(k), self._ptr(v), self._stream())

    def evict_frames(self, block, scale_frames=None, sliding_window=None, cross_frame_special=None,
                     camera_only=None):
        sf = self.scale_frames if scale_frames is None else scale_frames
        sw = self.sliding_window if sliding_window is None else sliding_window
        if cross_frame_special is None and camera_only is None:
            kvc_evict_frames(self.h, block, sf, sw)
        else:
            kvc_evict_frames_ex(self.h, block, sf, sw,
                                self.cross_frame_special if cross_frame_special is None else cross_frame_special,
                                self.camera_only if camera_only is None else camera_only)

    def set_defer_eviction(self, on):
        kvc_set_defer_eviction(self.h, on)

    def execute_deferred_eviction(self, block, scale_frames=None, sliding_window=None):
        kvc_execute_deferred_eviction(
            self.h, block, self.scale_frames if scale_frames is None else scale_frames,
            self.sliding_window if sliding_window is None else sliding_window)

    def rollback_last_frame(self, block):
        kvc_rollback_last_frame(self.h, block)

    def clean(self):
        kvc_clean(self.h)

    def plan(self):
        kvc_plan(self.h, self._stream())
        if _DEBUG_EVERY:
            # KVC_DEBUG=N: every N plans (one per streamed frame) print each
            # block's slot usage, like the pages' LINGBOT_DEBUG_KV ([SLOTS]
            # "动手验证"): scale_pg / live_pg / free_pg / special.
            self._plans = getattr(self, "_plans", 0) + 1
            if self._plans % _DEBUG_EVERY == 0:
                for b in range(self.num_blocks):
                    st = self.stats(b)
                    print(f"[kvc] frame {st['frame_count']} block {b}: scale_pg={st['scale_pages']} "
                          f"live_pg={st['live_pages']} free_pg={st['free_pages']} "
                          f"special={st['special_tokens']}", file=sys.stderr)

    def run(self, block, q, out):
        kvc_run(self.h, block, self._ptr(q), self._ptr(out), q.shape[0], self._stream())
        return out

    def prefill(self, block, q, k, v, out):
        """Phase 1: n_frames = q.shape[0] // (6 + page_size) frames attend to each
        other densely, then are appended to the (empty) block."""
        T = 6 + self.page_size
        if q.shape[0] % T or k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
            raise ValueError("prefill wants Q, K, V, out of shape [n_frames * (6 + page_size), H, D]")
        kvc_prefill(self.h, block, self._ptr(q), self._ptr(k), self._ptr(v), q.shape[0] // T,
                    self._ptr(out), self._stream())
        return out

    def stats(self, block):
        return kvc_get_cache_stats(self.h, block)

    def plan_table(self):
        return kvc_get_plan(self.h)

    def plan_ranges(self):
        """(indices, first_rows, valid_lens) of the current plan (host copy)."""
        return kvc_get_plan_ranges(self.h)

    def deques(self, block):
        return kvc_get_deques(self.h, block)

    def set_option(self, option, value):
        kvc_set_option(self.h, option, value)

    def close(self):
        if getattr(self, "h", None):
            kvc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
