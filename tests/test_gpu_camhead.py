"""The camera head's isomorphic cache beside the trunk's ([SLOTS] "特殊 token
流", last sentence: an independent KV cache of the same form with the same
scale / window parameters), both driven in one stream: per frame every trunk
block appends, evicts, plans (block 0) and attends, then every camera-head
block does the same on its own cache.  Each cache is checked against its own
oracle through the C ABI: page tables every frame, cache bytes, attention.
"""

import numpy as np
import pytest
import torch

from streaming_paged_kv_gb300.workloads import PAIRED, WORKLOADS
from gpu_engine import ParityEngine, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _stream_pair(engines, n_frames):
    for f in range(n_frames):
        for e in engines:                      # trunk first, then the camera head
            for b in range(e.w.num_layers):
                e.append(b, f)
                e.evict(b)
                if b == 0:
                    e.plan()
                e.attend(b, f)
            e.after_frame(f, "key")


@pytest.mark.parametrize("window", [4, 64])
def test_trunk_and_camera_head_caches_in_one_stream(kvc, window):
    trunk_name, head_name = PAIRED["camcache"]
    small = dict(sliding_window=window, headroom=2 if window == 4 else 16, max_total_frames=400)
    n = 14 if window == 4 else 80
    tw = WORKLOADS[trunk_name].with_(num_layers=2, n_frames=n, **small)
    hw = WORKLOADS[head_name].with_(num_layers=2, n_frames=n, **small)
    assert (hw.scale_frames, hw.sliding_window, hw.headroom) == (tw.scale_frames, tw.sliding_window, tw.headroom)
    rows = list(range(0, 1005, 11)) + [1004]
    check = {0, 7, 8, 9, n - 1}
    trunk = ParityEngine(kvc, tw, check_frames=check, rows=rows, check_device_plan=True)
    head = ParityEngine(kvc, hw, check_frames=check, rows=rows, check_device_plan=True)
    _stream_pair([trunk, head], n)
    torch.cuda.synchronize()
    from streaming_paged_kv_gb300.inputs import to_bits
    for e in (trunk, head):
        for b in range(e.w.num_layers):
            assert np.array_equal(to_bits(e.c.cache_view(b).cpu()), e.orc.mirror[b])
        mx, rel = e.worst()
        assert len(e.results) == 2 * len(check), e.results
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
        assert kvc.kvc_device_status(e.c.h, e.c._stream()) == 0
    # Independent caches: the same frame schedule gives the same page tables,
    # different contents.
    assert trunk.c.plan_table() == head.c.plan_table()
    assert not torch.equal(trunk.c.cache_view(0), head.c.cache_view(0))
    trunk.close()
    head.close()
