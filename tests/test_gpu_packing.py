"""GPU parity of packed KV tiles: the tensor-core plan fills a page's last
128-row tile with the next visible page's first rows, in units of 8 rows,
when every visible page but the last has at least 15 such units.

The tile count and the packing decision are checked against a count made here
from the oracle's visible row ranges; attention against the oracle with
packing on and off, with split counts whose boundaries fall on packed tiles,
and with second segments that start inside a page (the live frames' special
run of the policy without cross-frame specials) or that are a short last page.
"""

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


def expected_tiles(ranges, tile=128, unit=8, min_units=15):
    """(tiles, packed) for visible row counts `ranges[2]`: packed tiles cover
    16 units of 8 rows of the concatenated pages, allowed when every page but
    the last has >= 15 units; otherwise ceil(rows / 128) per page."""
    valid = list(ranges[2])
    units = [-(-v // unit) for v in valid]
    if all(u >= min_units for u in units[:-1]):
        return -(-sum(units) // (tile // unit)), True
    return sum(-(-v // tile) for v in valid), False


def _check_plans(e, want_packed=None):
    assert e.plans
    for f, got, ranges in e.plans:
        want = expected_tiles(ranges)
        assert got == want, (f, got, want)
        if want_packed is not None:
            assert got[1] == want_packed, (f, got)


def _s518(**kw):
    return WORKLOADS["s518"].with_(num_layers=1, **kw)


def test_packed_counts_and_parity_s518(kvc):
    """999-row pages: 125 units each, so 12 patch pages and a 72-row special
    page take 95 packed tiles instead of 97; every tile boundary but the
    first page's is inside a page."""
    w = _s518(n_frames=12, sliding_window=4, headroom=2, max_total_frames=400)
    rows = list(range(0, 1005, 6)) + [1004]
    e = ParityEngine(kvc, w, check_frames={0, 1, 5, 11}, kernel=2, rows=rows)
    drive(w, e)
    _check_plans(e, want_packed=True)
    assert e.plans[-1][1] == (95, True)
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    e.close()


@pytest.mark.parametrize("qtiles", [1, 2])
def test_packed_vs_unpacked_splits(kvc, qtiles):
    """The same frame attended with packing on and off, each against the
    oracle, for split counts that put split boundaries on packed tiles (95
    tiles: 1, 5, 19, 95 splits) and with one and two query tiles per CTA."""
    from oracle import OraclePagedKV, paged_attention
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    c = kvc.PagedKVCache(1, 16, 64, 999, "bf16", 8, 4, 2, 400, max_kv_splits=128)
    c.set_option(kvc.KVC_OPT_ATTN_KERNEL, 2)
    c.set_option(kvc.KVC_OPT_QUERY_TILES, qtiles)
    orc = OraclePagedKV(1, 999, 16, 64, "bf16", 8, 4, 2, 400)
    for f in range(12):
        q, k, v = frame_qkv(33, 5, f, 0, 999, 16, 64)
        c.append_frame(0, k.cuda(), v.cuda())
        c.evict_frames(0)
        orc.append_frame(0, to_bits(k), to_bits(v))
        orc.evict_frames(0, 8, 4)
    rows = list(range(0, 1005, 4)) + [1004]
    want = paged_attention(orc, 0, to_bits(q), rows=rows)
    sel = torch.as_tensor(rows, device="cuda")
    for pack, n_tiles in ((1, 95), (0, 97)):
        c.set_option(kvc.KVC_OPT_PACK_TILES, pack)
        c.plan()
        assert kvc.kvc_get_plan_tiles(c.h) == (n_tiles, bool(pack))
        for splits in (1, 5, 19, n_tiles):
            c.set_option(kvc.KVC_OPT_NUM_SPLITS, splits)
            qd = q.cuda()
            out = torch.empty_like(qd)
            c.run(0, qd, out)
            torch.cuda.synchronize()
            mx, rel = compare(out[sel], want, "bf16")
            assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], (pack, splits, mx, rel)
    assert kvc.kvc_device_status(c.h, c._stream()) == 0
    c.close()


@pytest.mark.parametrize("cross,cam,frames", [(False, False, {59, 169}), (True, True, {59})])
def test_packed_second_segment_inside_a_page(kvc, cross, cam, frames):
    """Without cross-frame specials (20 scale frames: a 120-row run; window
    30: a 180-row run from row 180 of the same special page at frame 59), the
    tile that ends the scale frames' specials continues at row 180; at frame
    169 the live run is rows 840..995 of special page 0 and a 24-row last
    entry on page 1.  With camera_only the last entry is the evicted frames'
    10 camera rows."""
    w = _s518(n_frames=max(frames) + 1, scale_frames=20, sliding_window=30, headroom=2,
              max_total_frames=400)
    rows = list(range(0, 1005, 8)) + [1004]
    e = ParityEngine(kvc, w, check_frames=frames, kernel=2, rows=rows, check_device_plan=True,
                     cross_frame_special=cross, camera_only=cam)
    drive(w, e)
    _check_plans(e, want_packed=True)
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    assert kvc.kvc_device_status(e.c.h, e.c._stream()) == 0
    e.close()


def test_packing_declined_for_short_middle_entries(kvc):
    """A 48-row run of scale-frame specials in the middle of the visible list
    (8 scale frames, no cross-frame specials) keeps one page per tile."""
    w = _s518(n_frames=14, sliding_window=4, headroom=2, max_total_frames=400)
    rows = list(range(0, 1005, 10)) + [1004]
    e = ParityEngine(kvc, w, check_frames={13}, kernel=2, rows=rows, cross_frame_special=False)
    drive(w, e)
    _check_plans(e, want_packed=False)
    mx, rel = e.worst()
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], e.results
    e.close()
