"""GPU parity of the special-token policies -- the reading of the eviction
options cross_frame_special and camera_only ([KVC] "Streaming Forward Pass")
-- through the C ABI against the CPU oracle: device and host plan row ranges
bit-exact at every plan, cache bytes bit-exact (camera stream included), and
attention within the tolerance, on both attention kernels, through eviction,
deferral and rollback.
"""

import pytest
import torch

from streaming_paged_kv_gb300.workloads import WORKLOADS
from stream_driver import drive
from gpu_engine import ParityEngine, TOL

pytestmark = pytest.mark.gpu

POLICIES = [(False, False), (True, True)]      # (cross_frame_special, camera_only)


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


@pytest.mark.parametrize("cross,cam", POLICIES)
def test_policy_tiny_f32_every_frame(kvc, cross, cam):
    w = WORKLOADS["tiny"]
    e = ParityEngine(kvc, w, check_frames=range(12), check_bytes=True, check_device_plan=True,
                     cross_frame_special=cross, camera_only=cam)
    drive(w, e)
    mx, _ = e.worst()
    assert len(e.results) == 12 and mx <= TOL["f32"][0], e.results
    e.close()


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("cross,cam", POLICIES)
def test_policy_deferred_bf16(kvc, cross, cam, kernel):
    # 224x224 geometry, 2 layers, provisional frames accepted / rolled back,
    # through the first evictions (window 64) and a special page boundary (42 frames).
    w = WORKLOADS["defer"].with_(num_layers=2, n_frames=100)
    e = ParityEngine(kvc, w, check_frames={0, 8, 41, 42, 43, 75, 76, 99}, kernel=kernel,
                     check_device_plan=True, cross_frame_special=cross, camera_only=cam)
    drive(w, e)
    torch.cuda.synchronize()
    from streaming_paged_kv_gb300.inputs import to_bits
    import numpy as np
    for b in range(2):
        assert np.array_equal(to_bits(e.c.cache_view(b).cpu()), e.orc.mirror[b])
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    e.close()


@pytest.mark.parametrize("cross,cam", POLICIES)
def test_policy_s518_ragged(kvc, cross, cam):
    """999-row pages (ragged KV tiles) with a small window, so that frames are
    evicted within 14 frames and special runs start inside a page."""
    w = WORKLOADS["s518"].with_(num_layers=1, n_frames=14, sliding_window=4, headroom=2,
                                max_total_frames=400)
    rows = list(range(0, 1005, 9)) + [1004]
    e = ParityEngine(kvc, w, check_frames={0, 6, 7, 13}, rows=rows, check_device_plan=True,
                     check_bytes=True, cross_frame_special=cross, camera_only=cam)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    e.close()
