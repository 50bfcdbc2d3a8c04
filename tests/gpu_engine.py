"""GPU engine (libkvc.so through the C ABI) and oracle engine driven side by
side on the same seeded inputs, for the parity tests."""

import numpy as np
import torch

from oracle import OraclePagedKV, paged_attention
from oracle.attention import bits_to_f64
from streaming_paged_kv_gb300.inputs import frame_qkv, k_head_scale, to_bits

TOL = {"bf16": (2e-2, 5e-3), "f16": (2e-2, 5e-3), "f32": (1e-4, 1e-4)}


def compare(got, want, dtype):
    """(max-abs error, relative RMS error) of a device output against the oracle."""
    g = got.detach().to("cpu", torch.float64).numpy()
    err = np.abs(g - want)
    rel = float(np.sqrt(((g - want) ** 2).sum() / max((want ** 2).sum(), 1e-300)))
    return float(err.max()), rel


class ParityEngine:
    """Drives the library and the oracle with identical calls; checks attention
    outputs at the frames in ``check_frames`` and cache bytes / device plans on
    request."""

    def __init__(self, kvc, w, seed=0, check_frames=(), kernel=0, splits=0, rows=None,
                 check_bytes=False, check_device_plan=False, mirror_blocks=None, qtiles=0,
                 cross_frame_special=True, camera_only=False):
        self.kvc, self.w, self.seed = kvc, w, seed
        self.policy = dict(cross_frame_special=cross_frame_special, camera_only=camera_only)
        self.c = kvc.PagedKVCache(w.num_layers, w.num_heads, w.head_dim, w.page_size, w.dtype,
                                  w.scale_frames, w.sliding_window, w.headroom, w.max_total_frames,
                                  **self.policy)
        if kernel:
            self.c.set_option(kvc.KVC_OPT_ATTN_KERNEL, kernel)
        if splits:
            self.c.set_option(kvc.KVC_OPT_NUM_SPLITS, splits)
        if qtiles:
            self.c.set_option(kvc.KVC_OPT_QUERY_TILES, qtiles)
        self.orc = OraclePagedKV(w.num_layers, w.page_size, w.num_heads, w.head_dim, w.dtype,
                                 w.scale_frames, w.sliding_window, w.headroom, w.max_total_frames,
                                 mirror_blocks=mirror_blocks, **self.policy)
        self.head_scale = k_head_scale(seed, w.wid, w.num_heads) if w.k_head_scale else None
        self.check_frames = set(check_frames)
        self.rows = rows
        self.check_bytes = check_bytes
        self.check_device_plan = check_device_plan
        self.results = []        # (frame, block, max_abs, rel_rms)
        self.plans = []          # (frame, (n_tiles, packed), oracle visible ranges) at checked frames
        self._plan = None
        self._q = {}

    def _inputs(self, b, f):
        w = self.w
        return frame_qkv(self.seed, w.wid, f, b, w.page_size, w.num_heads, w.head_dim, w.dtype,
                         self.head_scale)

    def append(self, b, f):
        q, k, v = self._inputs(b, f)
        self._q[b] = q
        self.c.append_frame(b, k.cuda(), v.cuda())
        if b in self.orc.mirror:
            self.orc.append_frame(b, to_bits(k), to_bits(v))
        else:
            self.orc.append_frame(b, np.empty(k.shape, np.uint16 if self.w.dtype != "f32" else np.uint32),
                                  np.empty(k.shape, np.uint16 if self.w.dtype != "f32" else np.uint32))

    def evict(self, b):
        if self.policy["cross_frame_special"] and not self.policy["camera_only"]:
            self.c.evict_frames(b)
        else:
            self.c.evict_frames(b, **self.policy)         # kvc_evict_frames_ex
        self.orc.evict_frames(b, self.w.scale_frames, self.w.sliding_window, **self.policy)

    def set_defer(self, on):
        self.c.set_defer_eviction(on)
        self.orc.set_defer_eviction(on)

    def execute(self, b):
        self.c.execute_deferred_eviction(b)
        self.orc.execute_deferred_eviction(b, self.w.scale_frames, self.w.sliding_window)

    def rollback(self, b):
        self.c.rollback_last_frame(b)
        self.orc.rollback_last_frame(b)

    def clean(self):
        self.c.clean()
        self.orc.clean()

    def plan(self):
        self.c.plan()
        self._plan = (self.kvc.kvc_get_plan_tiles(self.c.h), tuple(self.orc.visible_ranges(0)))
        if self.check_device_plan:
            idx, valid, lpl = self.kvc.kvc_read_device_plan(self.c.h, self.c._stream())
            o_idx, _, o_lpl, o_valid = self.orc.visible_page_table(0)
            assert (idx, valid, lpl) == (o_idx, o_valid, o_lpl)
            want = tuple(self.orc.visible_ranges(0))
            assert tuple(self.kvc.kvc_read_device_ranges(self.c.h, self.c._stream())) == want
            assert tuple(self.c.plan_ranges()) == want

    def attend(self, b, f):
        q = self._q[b]
        qd = q.cuda()
        out = torch.empty_like(qd)
        self.c.run(b, qd, out)
        if f in self.check_frames and b in self.orc.mirror:
            if not self.plans or self.plans[-1][0] != f:
                self.plans.append((f,) + self._plan)
            want = paged_attention(self.orc, b, to_bits(q), rows=self.rows)
            got = out if self.rows is None else out[torch.as_tensor(self.rows, device=out.device)]
            torch.cuda.synchronize()
            mx, rel = compare(got, want, self.w.dtype)
            self.results.append((f, b, mx, rel))

    def after_frame(self, f, kind):
        if self.check_bytes:
            torch.cuda.synchronize()
            for b in self.orc.mirror:
                dev = to_bits(self.c.cache_view(b).cpu())
                assert np.array_equal(dev, self.orc.mirror[b]), (f, kind, b)

    def worst(self):
        if not self.results:
            return 0.0, 0.0
        return max(r[2] for r in self.results), max(r[3] for r in self.results)

    def close(self):
        self.c.close()


def _frame_job(args):
    from streaming_paged_kv_gb300.inputs import frame_qkv
    return frame_qkv(*args)


def make_pool(workers=None):
    """Process pool for input generation (spawn context: safe next to an
    initialised CUDA context)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    n = workers or max(1, min(16, (os.cpu_count() or 2) - 1))
    return cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))


class FrameSource:
    """Seeded frames of one workload, generated by a process pool with a
    bounded look-ahead (at most `ahead` frames in flight or buffered)."""

    def __init__(self, w, pool, seed=0, ahead=48):
        self.w, self.pool, self.seed, self.ahead = w, pool, seed, ahead
        self.head_scale = k_head_scale(seed, w.wid, w.num_heads) if w.k_head_scale else None

    def frames(self, frame_ids, layer):
        from collections import deque
        w = self.w
        ids = iter(frame_ids)
        pending = deque()

        def submit():
            for f in ids:
                pending.append(self.pool.submit(_frame_job, (self.seed, w.wid, f, layer, w.page_size,
                                                             w.num_heads, w.head_dim, w.dtype,
                                                             self.head_scale)))
                return True
            return False

        for _ in range(self.ahead):
            if not submit():
                break
        while pending:
            out = pending.popleft().result()
            submit()
            yield out
