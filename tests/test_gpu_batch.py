"""Several independent streams in one launch (kvc_run_batch) against the oracle.

Each stream has its own handle, cache, plan and frame count (so its own
visible set: before the first eviction, after it, with a partial special
page); the batched launch must give every stream what the oracle gives for
that stream alone.  Also: ragged and empty query ranges, every split count,
16 streams (the maximum), the CUDA-core path (run one after another), and
errors that must launch nothing.
"""

import numpy as np
import pytest
import torch

from gpu_engine import TOL, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


class _Stream:
    """One stream: a library cache and the oracle, fed the same frames."""

    def __init__(self, kvc, wid, n_frames, ps=256, H=16, D=64, dtype="bf16", scale=8, window=64,
                 headroom=16, max_total_frames=256, max_query_tokens=0):
        from oracle import OraclePagedKV
        from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
        self.ps, self.H, self.D, self.dtype = ps, H, D, dtype
        self.c = kvc.PagedKVCache(1, H, D, ps, dtype, scale, window, headroom, max_total_frames,
                                  max_query_tokens=max_query_tokens)
        self.orc = OraclePagedKV(1, ps, H, D, dtype, scale, window, headroom, max_total_frames)
        for f in range(n_frames):
            q, k, v = frame_qkv(11, wid, f, 0, ps, H, D, dtype)
            self.c.append_frame(0, k.cuda(), v.cuda())
            self.c.evict_frames(0)
            self.orc.append_frame(0, to_bits(k), to_bits(v))
            self.orc.evict_frames(0, scale, window)
        self.c.plan()
        self.q = q                       # the last frame's queries

    def want(self, q):
        from oracle import paged_attention
        from streaming_paged_kv_gb300.inputs import to_bits
        return paged_attention(self.orc, 0, to_bits(q))


def _run_and_check(kvc, streams, qs):
    rows = [q.shape[0] for q in qs]
    q = torch.cat(qs).cuda()
    out = torch.full_like(q, float("nan"))
    kvc.run_batch([s.c for s in streams], [0] * len(streams), q, out, rows)
    torch.cuda.synchronize()
    res = []
    r0 = 0
    for s, qi, n in zip(streams, qs, rows):
        if n:
            res.append(compare(out[r0:r0 + n], s.want(qi), s.dtype))
        r0 += n
    return res


def test_four_streams_one_launch(kvc):
    streams = [_Stream(kvc, 60 + i, n) for i, n in enumerate([3, 10, 75, 40])]
    res = _run_and_check(kvc, streams, [s.q for s in streams])
    for mx, rel in res:
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], res
    launches = kvc.kvc_get_counters(streams[0].c.h)[1]
    assert launches == 1                 # one attention launch for all four


@pytest.mark.parametrize("splits", [1, 2, 7, 32])
def test_split_counts(kvc, splits):
    streams = [_Stream(kvc, 70 + i, n) for i, n in enumerate([12, 80])]
    streams[0].c.set_option(kvc.KVC_OPT_NUM_SPLITS, splits)
    res = _run_and_check(kvc, streams, [s.q for s in streams])
    for mx, rel in res:
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], (splits, res)


def test_ragged_and_empty_query_ranges(kvc):
    streams = [_Stream(kvc, 80 + i, n, max_query_tokens=600) for i, n in enumerate([5, 9, 20, 33])]
    g = np.random.default_rng(5)
    qs = [torch.from_numpy(g.standard_normal((n, 16, 64)).astype(np.float32)).to(torch.bfloat16)
          for n in (1, 0, 600, 129)]
    res = _run_and_check(kvc, streams, qs)
    assert len(res) == 3
    for mx, rel in res:
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], res


def test_sixteen_streams(kvc):
    streams = [_Stream(kvc, 100 + i, 2 + 5 * i, max_total_frames=128) for i in range(16)]
    res = _run_and_check(kvc, streams, [s.q for s in streams])
    assert len(res) == 16
    for mx, rel in res:
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], res


def test_cuda_core_path_runs_in_turn(kvc):
    streams = [_Stream(kvc, 120 + i, n, ps=16, H=2, D=32, dtype="f32", scale=2, window=4, headroom=2,
                       max_total_frames=16) for i, n in enumerate([4, 9])]
    res = _run_and_check(kvc, streams, [s.q for s in streams])
    for mx, rel in res:
        assert mx <= TOL["f32"][0], res


def test_errors_launch_nothing(kvc):
    a, b = _Stream(kvc, 130, 6), _Stream(kvc, 131, 7)
    q = torch.cat([a.q, b.q]).cuda()
    out = torch.full_like(q, float("nan"))
    n = a.q.shape[0]
    with pytest.raises(kvc.KvcError) as e:               # the same handle twice
        kvc.run_batch([a.c, a.c], [0, 0], q, out, [n, n])
    assert e.value.code == "INVALID_ARG"
    other = _Stream(kvc, 132, 4, H=8, max_query_tokens=262)
    with pytest.raises(kvc.KvcError) as e:               # different geometry
        kvc.kvc_run_batch([a.c.h, other.c.h], [0, 0], a.c._ptr(q), a.c._ptr(out), [0, n, 2 * n])
    assert e.value.code == "INVALID_ARG"
    from streaming_paged_kv_gb300.inputs import frame_qkv
    _, k, v = frame_qkv(11, 131, 7, 0, 256, 16, 64)
    b.c.append_frame(0, k.cuda(), v.cuda())             # b's plan is now stale
    with pytest.raises(kvc.KvcError) as e:
        kvc.run_batch([a.c, b.c], [0, 0], q, out, [n, n])
    assert e.value.code == "STALE_PLAN"
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()                 # nothing was written
