"""The attention-launch timing option (KVC_OPT_TIMING): every launch, or one
launch in every N (the (N/2)-th of each group of N) counted N times."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def test_sampled_timing_matches_every_launch(kvc):
    from streaming_paged_kv_gb300.inputs import frame_qkv
    c = kvc.PagedKVCache(1, 16, 64, 256, "bf16", max_total_frames=64)
    for f in range(40):
        _, k, v = frame_qkv(3, 2, f, 0, 256, 16, 64)
        c.append_frame(0, k.cuda(), v.cuda())
        c.evict_frames(0)
    c.plan()
    q = frame_qkv(3, 2, 40, 0, 256, 16, 64)[0].cuda()
    out = torch.empty_like(q)
    for _ in range(8):
        c.run(0, q, out)
    torch.cuda.synchronize()

    def timed(every, n):
        kvc.kvc_get_counters(c.h, reset=True)
        c.set_option(kvc.KVC_OPT_TIMING, every)
        for _ in range(n):
            c.run(0, q, out)
        torch.cuda.synchronize()
        _, launches, ms = kvc.kvc_get_counters(c.h, reset=True)
        c.set_option(kvc.KVC_OPT_TIMING, 0)
        return launches, ms

    n1, ms1 = timed(1, 48)
    n8, ms8 = timed(8, 48)                       # launches 4, 12, ..., 44 timed, each counted 8 times
    assert n1 == n8 == 48
    assert ms1 > 0 and ms8 > 0
    assert 0.7 < ms8 / ms1 < 1.4, (ms1, ms8)
    with pytest.raises(kvc.KvcError):
        c.set_option(kvc.KVC_OPT_TIMING, -1)
    assert kvc.kvc_device_status(c.h, c._stream()) == 0
    c.close()


def test_pdl_off_gives_identical_outputs(kvc):
    """KVC_OPT_PDL only changes how the kernels are launched: outputs with and
    without programmatic dependent launch are bit-identical (several layers,
    so that append, plan, attention and merge follow each other)."""
    from streaming_paged_kv_gb300.inputs import frame_qkv
    outs = []
    for pdl in (1, 0):
        c = kvc.PagedKVCache(3, 16, 64, 256, "bf16", max_total_frames=64)
        c.set_option(kvc.KVC_OPT_PDL, pdl)
        res = []
        for f in range(12):
            for b in range(3):
                q, k, v = frame_qkv(9, 2, f, b, 256, 16, 64)
                c.append_frame(b, k.cuda(), v.cuda())
                c.evict_frames(b)
                if b == 0:
                    c.plan()
                out = torch.empty_like(q.cuda())
                c.run(b, q.cuda(), out)
                res.append(out)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(c.h, c._stream()) == 0
        outs.append(torch.stack(res).cpu())
        c.close()
    assert torch.equal(outs[0], outs[1])
    with pytest.raises(kvc.KvcError):
        kvc.PagedKVCache(1, 16, 64, 256, "bf16", max_total_frames=64).set_option(kvc.KVC_OPT_PDL, 2)
