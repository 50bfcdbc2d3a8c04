"""The C-ABI library loads on a machine without a GPU and exports every
function include/kvc.h declares; configuration validation needs no GPU."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvc():
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvc.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(kvc):
    names = declared_functions()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(kvc.lib, n)]
    assert not missing, missing


def test_required_bytes_and_validation(kvc):
    cfg = kvc.make_config(24, 16, 64, 999)
    cache, ws = kvc.kvc_required_bytes(cfg)
    # 88 patch + ceil(2048/166) = 13 special pages, K and V, 999 rows of 16*64 bf16 per block.
    assert cache == 24 * 101 * 2 * 999 * 16 * 64 * 2
    assert ws > 0
    for bad in (dict(head_dim=48), dict(page_size=5), dict(num_heads=0),
                dict(scale_frames=2000), dict(max_kv_splits=1000)):
        args = dict(num_blocks=1, num_heads=16, head_dim=64, page_size=256)
        args.update(bad)
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_required_bytes(kvc.make_config(**args))
        assert e.value.code == "INVALID_ARG"


def test_bookkeeping_handle_refuses_device_calls(kvc):
    c = kvc.PagedKVCache(1, 2, 32, 16, "f32", 2, 4, 2, 16, device=None)
    c.append_frame(0)
    c.plan()
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_run(c.h, 0, None, None, 0)
    assert e.value.code == "NO_DEVICE"
    assert kvc.kvc_device_status(c.h) == -11
    assert kvc.kvc_strerror(-7).startswith("stale plan")


def test_debug_print_every_n_frames():
    """KVC_DEBUG=N prints every block's slot usage every N plans (one per
    streamed frame), like the pages' LINGBOT_DEBUG_KV ([SLOTS] "动手验证")."""
    import subprocess
    import sys
    code = ("from streaming_paged_kv_gb300 import kvc\n"
            "c = kvc.PagedKVCache(2, 2, 32, 16, 'f32', 2, 4, 2, 16, device=None)\n"
            "for f in range(8):\n"
            "    for b in range(2):\n"
            "        c.append_frame(b); c.evict_frames(b)\n"
            "    c.plan()\n")
    env = dict(os.environ, KVC_DEBUG="4", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[kvc]")]
    assert lines == [
        "[kvc] frame 4 block 0: scale_pg=2 live_pg=2 free_pg=4 special=24",
        "[kvc] frame 4 block 1: scale_pg=2 live_pg=2 free_pg=4 special=24",
        "[kvc] frame 8 block 0: scale_pg=2 live_pg=4 free_pg=2 special=48",
        "[kvc] frame 8 block 1: scale_pg=2 live_pg=4 free_pg=2 special=48",
    ], r.stderr


def test_geometry_and_launch_shape_accessors(kvc):
    g = kvc.kvc_get_geometry(kvc.make_config(24, 16, 64, 999))
    assert (g.num_patch_pages, g.frames_per_special_page, g.num_special_pages, g.max_num_pages,
            g.tokens_per_frame) == (88, 166, 13, 101, 1005)
    assert g.block_bytes == 101 * g.page_bytes == 101 * 2 * 999 * 16 * 64 * 2
    c = kvc.PagedKVCache(1, 2, 32, 16, "f32", 2, 4, 2, 16, device=None)
    assert kvc.kvc_get_launch_shape(c.h) == (0, 0)      # no attention launched
    with pytest.raises(kvc.KvcError):
        kvc.kvc_get_plan_tiles(c.h)                      # no plan yet
    for _ in range(3):
        c.append_frame(0)
        c.evict_frames(0)
    c.plan()
    # A bookkeeping-only handle plans for the CUDA-core kernel (64-row tiles,
    # one page per tile): 3 patch pages of 16 rows, and the 3 frames' special
    # rows on two special pages of 2 frames each (12 and 6 rows).
    assert c.plan_ranges()[2] == [16, 16, 16, 12, 6]
    assert kvc.kvc_get_plan_tiles(c.h) == (5, False)
    c.clean()
    with pytest.raises(kvc.KvcError):
        kvc.kvc_get_plan_tiles(c.h)                      # clean drops the plan
    c.close()
