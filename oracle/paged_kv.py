"""Page bookkeeping of the two-stream paged KV cache, simulated with deques.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Every block of the model owns an identical cache.  Its patch pages
``0 .. P-1`` (``P = scale_frames + sliding_window + headroom``) move between
three deques -- ``scale``, ``live`` and ``free`` -- and its special pages
``P .. P+S-1`` form an append-only stream holding the 6 special tokens of
every frame ([SLOTS] "双流分页布局"; [KVC] "Physical Page Layout and
Indexing"; [PERF] "Two-Stream Page Pool Architecture").

The cache mirror stores raw element bits (uint16 for bf16/f16, uint32 for
fp32) so that the device cache can be compared with it byte for byte.
"""

from collections import deque

import numpy as np

# Number of special tokens per frame: camera, 4 registers, scale
# ([SLOTS] "特殊 token 流"; [SLOTS] intro, token layout [camera, register x4, scale, patch...]).
NUM_SPECIAL = 6

_BITS_DTYPE = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32}


class OracleError(Exception):
    """A call the bookkeeping rejects; ``code`` names the reason."""

    def __init__(self, code, msg=""):
        super().__init__(f"{code}: {msg}" if msg else code)
        self.code = code


class _BlockState:
    """Deques and counters of one block (one transformer layer)."""

    def __init__(self, num_patch_pages):
        self.reset(num_patch_pages)

    def reset(self, num_patch_pages):
        # Construction state: every patch page is free, in ID order (reading 2).
        self.free = deque(range(num_patch_pages))
        self.scale = deque()
        self.live = deque()
        self.special_frames = 0      # frames written to the special stream
        self.frame_count = 0
        self.undo = []               # (page, region) of uncommitted appends


class OraclePagedKV:
    """Bookkeeping + byte mirror of a ``num_blocks``-layer paged KV cache.

    Constructor keywords follow the manager's arguments in [PERF] "Minimal
    Streaming Inference Setup": the patch pool is ``scale_frames +
    sliding_window + headroom`` pages ([KVC] FAQ "How is memory bounded in
    streaming mode?"), one page per frame's patch tokens so
    ``page_size == tokens_per_frame - 6`` ([SLOTS] intro: one patch page holds
    exactly one frame's patch tokens; [PERF] "Page-Size Handling for FA2 vs
    FA3": exact page sizes, no padding).
    """

    def __init__(self, num_blocks, page_size, num_heads, head_dim, dtype="bf16",
                 scale_frames=8, sliding_window=64, headroom=16,
                 max_total_frames=2048, mirror_blocks=None,
                 cross_frame_special=True, camera_only=False):
        if dtype not in _BITS_DTYPE:
            raise ValueError(dtype)
        if page_size < NUM_SPECIAL:
            raise ValueError("page_size must hold at least one frame's special tokens")
        self.num_blocks = num_blocks
        self.page_size = page_size
        self.num_heads = num_heads
        self.head_dim = head_dim
        self.dtype = dtype
        self.scale_frames = scale_frames
        self.sliding_window = sliding_window
        self.headroom = headroom
        self.max_total_frames = max_total_frames
        # Patch pool size: 8 + 64 + 16 = 88 by default ([SLOTS] "双流分页布局").
        self.num_patch_pages = scale_frames + sliding_window + headroom
        # floor(page_size / 6) frames' specials per special page
        # ([SLOTS] "特殊 token 流": 42 frames per page at page_size 256).
        self.frames_per_special_page = page_size // NUM_SPECIAL
        # The special pool is sized from max_total_frames ([SLOTS] "特殊 token 流").
        self.num_special_pages = -(-max_total_frames // self.frames_per_special_page)
        # The two eviction options of [KVC] "Streaming Forward Pass" (the block
        # passes both to evict_frames; the pages never say what they do).
        # Reading taken: cross_frame_special -- a frame's special tokens stay
        # visible after its patch page is evicted (the pages' default
        # behaviour: the special stream is never evicted, [SLOTS] "特殊 token
        # 流"); with it off they leave the visible set together with the patch
        # page.  camera_only -- of an evicted frame's specials only the camera
        # token (the first of the six) stays visible.  The special stream
        # itself is unchanged (append-only); for camera_only every frame's
        # camera token is also written to a third append-only stream, the
        # camera pages, page_size tokens per page, so that the evicted frames'
        # camera tokens form one contiguous run.
        self.cross_frame_special = bool(cross_frame_special)
        self.camera_only = bool(camera_only)
        self.camera_stream = self.cross_frame_special and self.camera_only
        self.num_camera_pages = -(-max_total_frames // page_size) if self.camera_stream else 0
        self.first_camera_page = self.num_patch_pages + self.num_special_pages
        self.max_num_pages = self.num_patch_pages + self.num_special_pages + self.num_camera_pages
        self.tokens_per_frame = NUM_SPECIAL + page_size
        self.defer_eviction = False
        self.blocks = [_BlockState(self.num_patch_pages) for _ in range(num_blocks)]
        if mirror_blocks is None:
            mirror_blocks = range(num_blocks)
        bits = _BITS_DTYPE[dtype]
        # kv_caches[block]: [max_num_pages, 2, page_size, H, D], 0 = K, 1 = V
        # ([KVC] "Physical Page Layout and Indexing").  Zero at construction.
        self.mirror = {
            b: np.zeros((self.max_num_pages, 2, page_size, num_heads, head_dim), dtype=bits)
            for b in mirror_blocks
        }

    # ------------------------------------------------------------------ append
    def append_frame(self, block, k_bits, v_bits):
        """Write one frame's K/V ``[6 + page_size, H, D]`` into block ``block``.

        Rows 0..5 (the special tokens) go to the special stream, rows 6.. (the
        patch tokens) to a fresh patch page.  The page is routed to the scale
        region while it holds fewer than ``scale_frames`` pages, else to the
        live sliding window ([SLOTS] "scale frames永不驱逐": the routing rule of
        ``_write_patch_page``; [KVC] "Append and Evict API").
        """
        st = self._block(block)
        T = self.tokens_per_frame
        want = (T, self.num_heads, self.head_dim)
        if k_bits.shape != want or v_bits.shape != want:
            raise OracleError("INVALID_ARG", f"K/V must be {want}")
        if st.special_frames >= self.max_total_frames:
            raise OracleError("SPECIAL_POOL_FULL")
        if not st.free:
            raise OracleError("NO_FREE_PAGE")
        page = st.free.popleft()
        if len(st.scale) < self.scale_frames:
            st.scale.append(page)
            region = "scale"
        else:
            st.live.append(page)
            region = "live"
        s = st.special_frames
        if block in self.mirror:
            m = self.mirror[block]
            # Patch tokens fill the whole page: one page = one frame's patches.
            m[page, 0, :, :, :] = k_bits[NUM_SPECIAL:]
            m[page, 1, :, :, :] = v_bits[NUM_SPECIAL:]
            # Special tokens: frame-aligned packing (reading 1).
            sp_page = self.num_patch_pages + s // self.frames_per_special_page
            slot = NUM_SPECIAL * (s % self.frames_per_special_page)
            m[sp_page, 0, slot:slot + NUM_SPECIAL] = k_bits[:NUM_SPECIAL]
            m[sp_page, 1, slot:slot + NUM_SPECIAL] = v_bits[:NUM_SPECIAL]
            if self.camera_stream:
                # The camera token (row 0) also goes to camera position s.
                cam_page = self.first_camera_page + s // self.page_size
                m[cam_page, 0, s % self.page_size] = k_bits[0]
                m[cam_page, 1, s % self.page_size] = v_bits[0]
        st.special_frames = s + 1
        st.frame_count += 1
        st.undo.append((page, region))
        return page

    # ---------------------------------------------------------------- eviction
    def evict_frames(self, block, scale_frames, sliding_window, cross_frame_special=None,
                     camera_only=None):
        """FIFO eviction of the live window down to ``sliding_window`` pages.

        The oldest live page goes back to the free list; scale pages are never
        evicted, and what stays visible of an evicted frame's special tokens
        is set by the construction's cross_frame_special / camera_only
        ([SLOTS] "keyframes滑动窗口"; [KVC] "Append and Evict API",
        "Streaming Forward Pass").  Passing either option with a value other
        than the construction's is rejected, like a different scale_frames.
        A no-op while eviction is deferred ([PERF] "Deferred Eviction
        Strategy").
        """
        st = self._block(block)
        self._check_scale_arg(scale_frames, sliding_window)
        self._check_special_args(cross_frame_special, camera_only)
        if self.defer_eviction:
            return 0
        return self._evict(st, sliding_window, commit_always=False)

    def set_defer_eviction(self, on):
        """Manager-wide deferral switch ([PERF] "Deferred Eviction for Keyframe Decisions")."""
        self.defer_eviction = bool(on)

    def execute_deferred_eviction(self, block, scale_frames, sliding_window):
        """Do the backlog eviction and commit the pending frames
        ([SLOTS] "光流关键帧与回滚机制": keyframe -> execute_deferred_eviction)."""
        st = self._block(block)
        self._check_scale_arg(scale_frames, sliding_window)
        return self._evict(st, sliding_window, commit_always=True)

    def _evict(self, st, window, commit_always):
        moved = 0
        while len(st.live) > window:
            st.free.append(st.live.popleft())
            moved += 1
        if moved or commit_always:
            st.undo.clear()
        return moved

    # ---------------------------------------------------------------- rollback
    def rollback_last_frame(self, block):
        """Undo the last uncommitted append exactly: its patch page returns to
        the free list, the special count and the frame count drop by one
        ([SLOTS] "光流关键帧与回滚机制").  Cache bytes are left as they are."""
        st = self._block(block)
        if not st.undo:
            raise OracleError("NOTHING_TO_ROLLBACK")
        page, region = st.undo.pop()
        dq = st.scale if region == "scale" else st.live
        if not dq or dq[-1] != page:        # cannot happen: evictions commit
            raise OracleError("ROLLBACK_AFTER_EVICT")
        dq.pop()
        st.free.appendleft(page)
        st.special_frames -= 1
        st.frame_count -= 1

    def clean(self):
        """Reset every block to its construction state (``clean_kv_cache`` at
        each window start, [SLOTS] "窗口模式").  Cache bytes stay as they are."""
        for st in self.blocks:
            st.reset(self.num_patch_pages)
        self.defer_eviction = False

    # ------------------------------------------------------------------- plan
    def visible_page_table(self, block=0):
        """Visible pages in attention order: scale pages, then the live window,
        then every special page; specials last so that only the last page can
        be partial ([KVC] "Patch Pages vs. Special Pages"; [SLOTS] "双流分页布局").

        Returns ``(indices, indptr, last_page_len, valid_lens)``: FlashInfer's
        plan arguments for one request ([KVC] "Kernel-Level Execution Flow")
        plus the number of valid tokens of every visible page.  With a
        special-token policy other than the default, see
        ``visible_ranges`` (the pages' tokens then need not start at row 0)."""
        indices, first_rows, valid = self.visible_ranges(block)
        if not indices:
            return [], [0, 0], 0, []
        return indices, [0, len(indices)], valid[-1], valid

    def visible_ranges(self, block=0):
        """``(indices, first_rows, valid_lens)``: page i of the visible
        sequence contributes its rows ``[first_rows[i], first_rows[i] +
        valid_lens[i])``.  Order: scale pages, live window, special pages,
        camera pages.

        Default policy: every special page from row 0, the last one holding
        ``last_page_len`` tokens ([KVC] "Physical Page Layout and Indexing":
        compute_last_page_len).  The special stream position of a frame is its
        append order, so the scale frames are positions ``[0, n_scale)`` and
        the live frames ``[s - n_live, s)`` (appends go to the right end of the
        live window, eviction takes its left end, rollback its right end).
        Without cross-frame specials only those two runs are visible; with
        camera_only the evicted frames' camera tokens, camera positions
        ``[n_scale, s - n_live)``, are visible as well."""
        st = self._block(block)
        fpp = self.frames_per_special_page
        s = st.special_frames
        n_scale, n_live = len(st.scale), len(st.live)
        indices = list(st.scale) + list(st.live)
        first = [0] * len(indices)
        valid = [self.page_size] * len(indices)
        if self.cross_frame_special and not self.camera_only:
            runs = [(0, s)]
        elif n_scale >= s - n_live:
            runs = [(0, s)]                      # nothing evicted yet
        else:
            runs = [(0, n_scale), (s - n_live, s)]
        for a, b in runs:
            # frames [a, b): page P + f // fpp, rows 6 (f % fpp) .. +6
            for p in range(a // fpp, -(-b // fpp)) if b > a else ():
                lo = max(a, p * fpp) - p * fpp
                hi = min(b, (p + 1) * fpp) - p * fpp
                indices.append(self.num_patch_pages + p)
                first.append(NUM_SPECIAL * lo)
                valid.append(NUM_SPECIAL * (hi - lo))
        if self.camera_stream and n_scale < s - n_live:
            a, b, ps = n_scale, s - n_live, self.page_size
            for c in range(a // ps, -(-b // ps)):
                lo = max(a, c * ps) - c * ps
                hi = min(b, (c + 1) * ps) - c * ps
                indices.append(self.first_camera_page + c)
                first.append(lo)
                valid.append(hi - lo)
        return indices, first, valid

    def stats(self, block):
        """``get_cache_stats``: the five-field snapshot of [SLOTS] "动手验证"."""
        st = self._block(block)
        return {
            "frame_count": st.frame_count,
            "scale_pages": len(st.scale),
            "live_pages": len(st.live),
            "free_pages": len(st.free),
            "special_tokens": NUM_SPECIAL * st.special_frames,
        }

    def deques(self, block):
        st = self._block(block)
        return list(st.scale), list(st.live), list(st.free)

    # ---------------------------------------------------------------- gather
    def gather_visible(self, block, plan_block=0):
        """Dense K/V bits ``[n_visible, H, D]`` of block ``block`` in page order,
        using the visible table of ``plan_block`` (plan once, run for every
        block: [PERF] "One-Time Planning Pattern")."""
        if block not in self.mirror:
            raise ValueError(f"block {block} is not mirrored")
        indices, first, valid = self.visible_ranges(plan_block)
        m = self.mirror[block]
        ks = [m[p, 0, r:r + n] for p, r, n in zip(indices, first, valid)]
        vs = [m[p, 1, r:r + n] for p, r, n in zip(indices, first, valid)]
        if not ks:
            shape = (0, self.num_heads, self.head_dim)
            return np.zeros(shape, m.dtype), np.zeros(shape, m.dtype)
        return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)

    # ---------------------------------------------------------------- helpers
    def _block(self, block):
        if not 0 <= block < self.num_blocks:
            raise OracleError("INVALID_ARG", f"block {block}")
        return self.blocks[block]

    def _check_special_args(self, cross_frame_special, camera_only):
        # The options are the construction's; another value is rejected.
        if cross_frame_special is not None and bool(cross_frame_special) != self.cross_frame_special:
            raise OracleError("INVALID_ARG", "cross_frame_special")
        if camera_only is not None and bool(camera_only) != self.camera_only:
            raise OracleError("INVALID_ARG", "camera_only")

    def _check_scale_arg(self, scale_frames, sliding_window):
        # Routing uses the constructor's scale_frames; a different value is rejected.
        if scale_frames != self.scale_frames or sliding_window < 0:
            raise OracleError("INVALID_ARG", "scale_frames/sliding_window")
