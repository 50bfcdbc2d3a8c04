"""kvc_paged_attention_static -- the entry point for callers that cannot
allocate device memory (for example code inside a host framework that owns
all GPU memory and lends out only the KV cache and the Q / output buffers, so
it has no workspace to give kvc_create).  It keeps its scratch in an array
inside the library; this test checks, through the C ABI, that two calls in a
row give what kvc_run gives for the same cache and queries.

This file is named to be collected last, so that a run that stops at the first
failure has run every other test before it.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ABS, REL_RMS = 2e-2, 5e-3          # the bf16 tolerance of the parity tests


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _diff(a, b):
    a = a.to(torch.float64)
    b = b.to(torch.float64)
    return float((a - b).abs().max()), float((a - b).norm() / b.norm())


def test_static_scratch_matches_kvc_run_two_calls_in_a_row(kvc):
    from streaming_paged_kv_gb300.inputs import frame_qkv
    H, D, ps = 16, 64, 999
    c = kvc.PagedKVCache(1, H, D, ps, "bf16", scale_frames=2, sliding_window=3, headroom=2,
                         max_total_frames=64)
    stream = c._stream()
    results = []
    for f in range(7):
        q, k, v = frame_qkv(3, 77, f, 0, ps, H, D)
        c.append_frame(0, k.cuda(), v.cuda())
        c.evict_frames(0)
        c.plan()
        if f < 5:
            continue
        qd = q.cuda()
        ref = torch.empty_like(qd)
        c.run(0, qd, ref)
        ids, _, _ = kvc.kvc_get_plan(c.h)
        _, valid, _ = kvc.kvc_read_device_plan(c.h, stream)
        out = torch.full_like(qd, float("nan"))
        kvc.kvc_paged_attention_static(c.cache.data_ptr(), "bf16", H, D, ps, ids, valid,
                                       qd.data_ptr(), out.data_ptr(), qd.shape[0], 0.0, stream)
        torch.cuda.synchronize()
        results.append(_diff(out, ref))
    assert len(results) == 2
    for mx, rel in results:
        assert mx <= MAX_ABS and rel <= REL_RMS, results
    c.close()


def test_static_scratch_rejects_sizes_beyond_its_limit(kvc):
    ids = list(range(1025))
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_paged_attention_static(None, "bf16", 16, 64, 999, ids, [999] * 1025, None, None, 1)
    assert e.value.code == "TOO_LARGE"
    # 600 pages of 2048 rows are 600 x 32 = 19200 tiles of 64 rows: more than the 16384 the array holds.
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_paged_attention_static(None, "bf16", 16, 64, 2048, list(range(600)), [2048] * 600,
                                       None, None, 1)
    assert e.value.code == "TOO_LARGE"
