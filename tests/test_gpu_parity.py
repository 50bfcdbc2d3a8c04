"""GPU parity: libkvc.so through the C ABI against the CPU oracle.

Bit-exact: cache bytes after append / evict / rollback / reset, device page
tables.  Toleranced: attention outputs (bf16: max-abs 2e-2 and relative RMS
5e-3; fp32: 1e-4), on streams that span several KV tiles per page, ragged
page tails (999 = 7*128 + 103), partial special pages and every KV split
count.
"""

import numpy as np
import pytest
import torch

from streaming_paged_kv_gb300.workloads import WORKLOADS
from stream_driver import drive
from gpu_engine import ParityEngine, TOL, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _tc_available(kvc, w):
    c = kvc.PagedKVCache(1, w.num_heads, w.head_dim, w.page_size, w.dtype, w.scale_frames,
                         w.sliding_window, w.headroom, 64)
    try:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, 2)
        return True
    except kvc.KvcError:
        return False
    finally:
        c.close()


KERNELS = [1, 2]


def _kernel_or_skip(kvc, w, kernel):
    if kernel == 2 and not _tc_available(kvc, w):
        pytest.skip("no tensor-core kernel for this shape")


# ------------------------------------------------------------ bit-exact
def test_tiny_cache_bytes_and_device_plan_every_frame(kvc):
    w = WORKLOADS["tiny"]
    e = ParityEngine(kvc, w, check_frames=range(12), check_bytes=True, check_device_plan=True)
    drive(w, e)
    mx, rel = e.worst()
    assert len(e.results) == 12 and mx <= TOL["f32"][0], e.results
    e.close()


def test_defer_rollback_cache_bytes(kvc):
    # 224x224 geometry, 2 layers, provisional frames accepted / rolled back.
    w = WORKLOADS["defer"].with_(num_layers=2, n_frames=90)
    e = ParityEngine(kvc, w, check_frames={0, 8, 30, 75, 89}, check_device_plan=True)
    drive(w, e)
    torch.cuda.synchronize()
    for b in range(2):
        dev = e.c.cache_view(b).cpu()
        from streaming_paged_kv_gb300.inputs import to_bits
        assert np.array_equal(to_bits(dev), e.orc.mirror[b])
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


def test_clean_resets_plan_and_keeps_bytes(kvc):
    w = WORKLOADS["tiny"].with_(n_frames=5)
    e = ParityEngine(kvc, w, check_bytes=True)
    drive(w, e)
    e.clean()
    with pytest.raises(kvc.KvcError) as ex:
        q = torch.zeros(22, 2, 32, device="cuda")
        e.c.run(0, q, torch.empty_like(q))
    assert ex.value.code == "NO_PLAN"
    e.after_frame(-1, "clean")
    e.close()


# ----------------------------------------------------------- attention
@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_f32_all_frames(kvc, kernel):
    w = WORKLOADS["tiny"]
    _kernel_or_skip(kvc, w, kernel)
    e = ParityEngine(kvc, w, check_frames=range(12), kernel=kernel)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 1e-4, e.results
    e.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_s224_stream_bf16(kvc, kernel):
    # Through the first eviction and past it: frames 0..79 of the 224x224 stream.
    w = WORKLOADS["s224"].with_(num_layers=2, n_frames=80)
    _kernel_or_skip(kvc, w, kernel)
    e = ParityEngine(kvc, w, check_frames={0, 1, 7, 8, 9, 41, 42, 43, 71, 72, 73, 79}, kernel=kernel)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_split_counts(kvc, kernel, splits):
    w = WORKLOADS["s224"].with_(num_layers=1, n_frames=75)
    _kernel_or_skip(kvc, w, kernel)
    e = ParityEngine(kvc, w, check_frames={74}, kernel=kernel, splits=splits)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


@pytest.mark.parametrize("qtiles", [1, 2])
@pytest.mark.parametrize("splits", [1, 3, 7])
def test_query_tiles_per_cta(kvc, qtiles, splits):
    """Tensor-core kernel with one 128-row query tile per CTA (both softmax
    warp groups on alternate KV tiles of it) and with two: a 224x224 frame
    (262 rows: two full tiles and a 6-row tail) through the first eviction,
    with partial special pages."""
    w = WORKLOADS["s224"].with_(num_layers=1, n_frames=75)
    _kernel_or_skip(kvc, w, 2)
    e = ParityEngine(kvc, w, check_frames={0, 1, 9, 43, 74}, kernel=2, splits=splits, qtiles=qtiles)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


@pytest.mark.parametrize("qtiles", [1, 2])
def test_one_tile_splits(kvc, qtiles):
    """One KV split per tile (7 tiles: 3 pages x 2 + the 18-row special tile),
    with one and two query tiles per CTA: CTAs whose split is a single short
    tile, and splits of 1 and 3."""
    from oracle import OraclePagedKV, paged_attention
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    c = kvc.PagedKVCache(1, 16, 64, 256, "bf16", max_total_frames=64, max_kv_splits=16)
    try:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, 2)
    except kvc.KvcError:
        c.close()
        pytest.skip("no tensor-core kernel")
    orc = OraclePagedKV(1, 256, 16, 64, "bf16", 8, 64, 16, 64)
    for f in range(3):
        q, k, v = frame_qkv(21, 2, f, 0, 256, 16, 64)
        c.append_frame(0, k.cuda(), v.cuda())
        orc.append_frame(0, to_bits(k), to_bits(v))
    c.plan()
    c.set_option(kvc.KVC_OPT_QUERY_TILES, qtiles)
    want = paged_attention(orc, 0, to_bits(q))
    for splits in (7, 1, 3):                     # 3 pages x 2 tiles + 1 special tile = 7 tiles
        c.set_option(kvc.KVC_OPT_NUM_SPLITS, splits)
        qd = q.cuda()
        out = torch.empty_like(qd)
        c.run(0, qd, out)
        torch.cuda.synchronize()
        mx, rel = compare(out, want, "bf16")
        assert mx <= 2e-2 and rel <= 5e-3, (splits, mx, rel)
    assert kvc.kvc_device_status(c.h, c._stream()) == 0
    c.close()


@pytest.mark.parametrize("qtiles", [1, 2])
def test_s518_ragged_query_tiles(kvc, qtiles):
    """The 518x378 page geometry (999-row pages: ragged 103-row KV tiles; 1005
    query rows: a 109-row last query tile) with one and two query tiles per CTA."""
    w = WORKLOADS["s518"].with_(num_layers=1, n_frames=12, sliding_window=4, headroom=2,
                                max_total_frames=400)
    _kernel_or_skip(kvc, w, 2)
    rows = list(range(0, 1005, 5)) + [1004]
    e = ParityEngine(kvc, w, check_frames={0, 6, 11}, kernel=2, rows=rows, qtiles=qtiles)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_s518_exact_pages_ragged(kvc, kernel):
    # page_size 999: 7 full 128-row tiles + a 103-row tail per patch page;
    # special pages hold 996 valid rows; per-head K scaling sharpens the softmax.
    w = WORKLOADS["s518"].with_(num_layers=1, n_frames=12, sliding_window=4, headroom=2,
                                max_total_frames=400)
    _kernel_or_skip(kvc, w, kernel)
    rows = list(range(0, 1005, 7)) + [1004]
    e = ParityEngine(kvc, w, check_frames={0, 5, 11}, kernel=kernel, rows=rows)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= 2e-2 and rel <= 5e-3, e.results
    e.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_query_counts(kvc, kernel):
    """n_q = 0 is a no-op; ragged n_q (1, 127, 129, T) and Q rows beyond T up to
    max_query_tokens all attend over the same visible set."""
    from oracle import paged_attention
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    w = WORKLOADS["s224"].with_(num_layers=1)
    _kernel_or_skip(kvc, w, kernel)
    c = kvc.PagedKVCache(1, 16, 64, 256, "bf16", max_total_frames=64, max_query_tokens=600)
    if kernel:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, kernel)
    from oracle import OraclePagedKV
    orc = OraclePagedKV(1, 256, 16, 64, "bf16", 8, 64, 16, 64)
    for f in range(10):
        q, k, v = frame_qkv(5, 2, f, 0, 256, 16, 64)
        c.append_frame(0, k.cuda(), v.cuda())
        orc.append_frame(0, to_bits(k), to_bits(v))
    c.plan()
    qbig = torch.from_numpy(np.random.default_rng(0).standard_normal((600, 16, 64)).astype(np.float32)).to(torch.bfloat16)
    kvc.kvc_run(c.h, 0, None, None, 0, c._stream())
    for n in (1, 127, 129, 262, 600):
        qd = qbig[:n].cuda()
        out = torch.empty_like(qd)
        c.run(0, qd, out)
        want = paged_attention(orc, 0, to_bits(qbig[:n]))
        torch.cuda.synchronize()
        mx, rel = compare(out, want, "bf16")
        assert mx <= 2e-2 and rel <= 5e-3, (n, mx, rel)
    with pytest.raises(kvc.KvcError):
        qd = qbig.cuda()
        kvc.kvc_run(c.h, 0, qd.data_ptr(), qd.data_ptr(), 601, c._stream())
    c.close()


def test_stale_plan_detected(kvc):
    w = WORKLOADS["tiny"]
    c = kvc.PagedKVCache(2, 2, 32, 16, "f32", 2, 4, 2, 16)
    from streaming_paged_kv_gb300.inputs import frame_qkv
    q, k, v = frame_qkv(0, 1, 0, 0, 16, 2, 32, "f32")
    c.append_frame(0, k.cuda(), v.cuda())
    c.plan()
    qd = q.cuda()
    with pytest.raises(kvc.KvcError) as ex:
        c.run(1, qd, torch.empty_like(qd))           # block 1 has not appended yet
    assert ex.value.code == "STALE_PLAN"
    c.append_frame(1, k.cuda(), v.cuda())
    c.run(1, qd, torch.empty_like(qd))
    assert kvc.kvc_device_status(c.h, c._stream()) == 0
    c.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_max_jumps_inside_and_across_tiles(kvc, kernel):
    """Scores that jump far above the running max late in a tile (earlier P
    chunks of that tile must be rescaled) and in a late tile (O must be
    rescaled): a few keys are scaled up by 30 -- one patch row deep inside the
    first page, and the special rows of the newest frame, which come last."""
    from oracle import OraclePagedKV, paged_attention
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    w = WORKLOADS["s224"]
    _kernel_or_skip(kvc, w, kernel)
    c = kvc.PagedKVCache(1, 16, 64, 256, "bf16", max_total_frames=64)
    c.set_option(kvc.KVC_OPT_ATTN_KERNEL, kernel)
    orc = OraclePagedKV(1, 256, 16, 64, "bf16", 8, 64, 16, 64)
    for f in range(6):
        q, k, v = frame_qkv(11, 2, f, 0, 256, 16, 64)
        k = k.float()
        if f == 0:
            k[6 + 100] *= 30.0          # patch row 100 of the first page: chunk 3 of tile 0
        if f == 5:
            k[:6] *= 30.0               # newest specials: the last tile
        k = k.to(torch.bfloat16)
        c.append_frame(0, k.cuda(), v.cuda())
        orc.append_frame(0, to_bits(k), to_bits(v))
    c.plan()
    qd = q.cuda()
    out = torch.empty_like(qd)
    c.run(0, qd, out)
    want = paged_attention(orc, 0, to_bits(q))
    torch.cuda.synchronize()
    mx, rel = compare(out, want, "bf16")
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


# ------------------------------------------------------- dtypes / head sizes
@pytest.mark.parametrize("kernel", KERNELS)
def test_f16_stream(kvc, kernel):
    """fp16 caches: the tensor-core kernel's fp16 instantiation (P packed as
    fp16) and the CUDA-core kernel, through the first eviction, with splits."""
    w = WORKLOADS["s224"].with_(num_layers=1, n_frames=80, dtype="f16")
    _kernel_or_skip(kvc, w, kernel)
    e = ParityEngine(kvc, w, check_frames={0, 9, 40, 72, 79}, kernel=kernel, check_bytes=False)
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= TOL["f16"][0] and rel <= TOL["f16"][1], e.results
    e.close()


@pytest.mark.parametrize("head_dim", [32, 128])
def test_other_head_sizes_cuda_core(kvc, head_dim):
    """Head sizes without a tensor-core kernel run on the CUDA cores (bf16)."""
    w = WORKLOADS["s224"].with_(num_layers=1, n_frames=12, head_dim=head_dim, num_heads=8,
                                sliding_window=4, headroom=2, max_total_frames=64)
    e = ParityEngine(kvc, w, check_frames={0, 5, 11})
    drive(w, e)
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    c = e.c
    # auto kernel selection picked the CUDA-core kernel for this head size
    with pytest.raises(kvc.KvcError):
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, 2)
    e.close()
