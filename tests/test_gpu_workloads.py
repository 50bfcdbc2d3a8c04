"""Parity on the workloads at their own sizes, through the C ABI.

The 518x378 stream runs all 2048 frames in the launch configuration the
benchmark times (same heads, head size, page size, query rows and split
choice; one layer instead of 24 -- a layer's launch does not depend on the
others), with the oracle checking sampled query rows of sampled frames.  The
windowed stream runs one full 1568-frame window plus the reset into the next;
the deferred stream runs its 400 frames; the 224x224 stream its 200 frames.
"""

import numpy as np
import pytest
import torch

from oracle import OraclePagedKV, paged_attention
from streaming_paged_kv_gb300.inputs import keyframe_decisions, to_bits
from streaming_paged_kv_gb300.workloads import WORKLOADS, schedule
from gpu_engine import FrameSource, compare, make_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    ex = make_pool()
    yield ex
    ex.shutdown()


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _run(kvc, pool, w, check, rows=None, seed=0):
    """Stream workload w (one layer) through the library and the oracle;
    compare attention at the frames in `check` on `rows`."""
    w1 = w.with_(num_layers=1)
    c = kvc.PagedKVCache(1, w.num_heads, w.head_dim, w.page_size, w.dtype, w.scale_frames,
                         w.sliding_window, w.headroom, w.max_total_frames)
    orc = OraclePagedKV(1, w.page_size, w.num_heads, w.head_dim, w.dtype, w.scale_frames,
                        w.sliding_window, w.headroom, w.max_total_frames)
    src = FrameSource(w1, pool, seed)
    decisions = keyframe_decisions(seed, w.wid, w.n_frames) if w.mode == "defer" else None
    events = list(schedule(w1, decisions))
    frame_ids = [f for f, kind in events if kind != "clean"]
    results = []
    try:
        it = src.frames(frame_ids, 0)
        for f, kind in events:
            if kind == "clean":
                c.clean()
                orc.clean()
                continue
            q, k, v = next(it)
            provisional = kind in ("accept", "reject")
            c.set_defer_eviction(provisional)
            orc.set_defer_eviction(provisional)
            c.append_frame(0, k.cuda(), v.cuda())
            orc.append_frame(0, to_bits(k), to_bits(v))
            c.evict_frames(0)
            orc.evict_frames(0, w.scale_frames, w.sliding_window)
            c.plan()
            idx, _, lpl = c.plan_table()
            o_idx, _, o_lpl, _ = orc.visible_page_table(0)
            assert (idx, lpl) == (o_idx, o_lpl), f
            if f in check:
                qd = q.cuda()
                out = torch.empty_like(qd)
                c.run(0, qd, out)
                want = paged_attention(orc, 0, to_bits(q), rows=rows)
                got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
                torch.cuda.synchronize()
                results.append((f, kind) + compare(got, want, w.dtype))
            if kind == "accept":
                c.execute_deferred_eviction(0)
                orc.execute_deferred_eviction(0, w.scale_frames, w.sliding_window)
            elif kind == "reject":
                c.rollback_last_frame(0)
                orc.rollback_last_frame(0)
            c.set_defer_eviction(False)
            orc.set_defer_eviction(False)
        assert kvc.kvc_device_status(c.h, c._stream()) == 0
        torch.cuda.synchronize()
        dev = to_bits(c.cache_view(0).cpu())
        assert np.array_equal(dev, orc.mirror[0])                 # every cache byte
        shape = kvc.kvc_get_launch_shape(c.h)
    finally:
        c.close()
    assert len(results) == len(check), results
    worst = max(r[2] for r in results), max(r[3] for r in results)
    assert worst[0] <= 2e-2 and worst[1] <= 5e-3, results
    return results, shape


def test_s518_full_stream_sampled_rows(kvc, pool):
    w = WORKLOADS["s518"]
    rng = np.random.default_rng(4)
    check = {0, 1, 7, 8, 9, 71, 72, 73, 165, 166, 167, 1000, 2047} | set(rng.integers(0, 2048, 4).tolist())
    rows = sorted(set(range(0, 1005, 16)) | {1004, 6, 5})
    _, shape = _run(kvc, pool, w, check, rows)
    # The launch-shape model keeps two query tiles per CTA at full context
    # (1005 rows: 4 query blocks x 16 heads, many KV splits).
    assert shape[0] == 2 and shape[1] > 1, shape


def test_windowed_one_window_and_reset(kvc, pool):
    w = WORKLOADS["win518"].with_(n_frames=1568 + 30)
    # keyframes and non-keyframes late in the window, the reset, frames of the next window
    check = {0, 8, 9, 21, 1550, 1555, 1567, 1568, 1569, 1576, 1580}
    rows = sorted(set(range(0, 1005, 32)) | {1004})
    _run(kvc, pool, w, check, rows)


def test_deferred_stream_full(kvc, pool):
    w = WORKLOADS["defer"]
    check = {0, 7, 8, 9, 50, 150, 300, 399}
    _run(kvc, pool, w, check)


def test_s224_full_stream(kvc, pool):
    w = WORKLOADS["s224"]
    check = {0, 41, 42, 72, 73, 150, 199}
    _, shape = _run(kvc, pool, w, check)
    # Under one wave of two-tile CTAs (262 rows: 2 blocks x 16 heads) the model
    # takes one query tile per CTA.
    assert shape[0] == 1, shape


def test_bounded_wait_reports_timeout_and_recovers(kvc):
    """The tensor-core kernel's MMA warp waits on a barrier nothing signals
    (KVC_OPT_STALL_TEST) with a short budget: the wait runs out, the kernel
    records the timeout, every role drains, TMEM is freed and the kernel
    returns; the host sees KVC_ERR_DEVICE_TIMEOUT, and the next run with the
    normal settings is correct (the context is still usable)."""
    from streaming_paged_kv_gb300.inputs import frame_qkv
    c = kvc.PagedKVCache(1, 4, 64, 256, "bf16", 2, 4, 2, 64)
    try:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, 2)
    except kvc.KvcError:
        c.close()
        pytest.skip("no tensor-core kernel")
    orc = OraclePagedKV(1, 256, 4, 64, "bf16", 2, 4, 2, 64)
    for f in range(8):
        q, k, v = frame_qkv(1, 2, f, 0, 256, 4, 64)
        c.append_frame(0, k.cuda(), v.cuda())
        orc.append_frame(0, to_bits(k), to_bits(v))
        c.evict_frames(0)
        orc.evict_frames(0, 2, 4)
    c.plan()
    qd = q.cuda()
    out = torch.empty_like(qd)
    c.set_option(kvc.KVC_OPT_WAIT_BUDGET, 2_000_000)    # about a millisecond
    c.set_option(kvc.KVC_OPT_STALL_TEST, 1)
    c.run(0, qd, out)
    assert kvc.kvc_device_status(c.h, c._stream()) == -9
    assert kvc.kvc_device_status(c.h, c._stream()) == 0    # reading clears the status
    c.set_option(kvc.KVC_OPT_STALL_TEST, 0)
    c.set_option(kvc.KVC_OPT_WAIT_BUDGET, 0)
    c.run(0, qd, out)
    assert kvc.kvc_device_status(c.h, c._stream()) == 0
    want = paged_attention(orc, 0, to_bits(q))
    mx, rel = compare(out, want, "bf16")
    assert mx <= 2e-2 and rel <= 5e-3
    c.close()
