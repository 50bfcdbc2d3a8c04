"""Host page bookkeeping of libkvc.so (bookkeeping-only handles, no GPU)
against the oracle: deques, stats and plan tables bit-exact at every frame of
all five workloads at full length, plus error behaviour on random op mixes."""

import numpy as np
import pytest

from oracle import OraclePagedKV, OracleError
from streaming_paged_kv_gb300.workloads import WORKLOADS
from stream_driver import drive


@pytest.fixture(scope="module")
def kvc():
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


class BothBook:
    """Library (all blocks) + oracle (block 0 only), compared as they go."""

    def __init__(self, kvc, w, cross_frame_special=True, camera_only=False):
        self.kvc, self.w = kvc, w
        self.policy = dict(cross_frame_special=cross_frame_special, camera_only=camera_only)
        self.lib = kvc.PagedKVCache(w.num_layers, w.num_heads, w.head_dim, w.page_size, w.dtype,
                                    w.scale_frames, w.sliding_window, w.headroom,
                                    w.max_total_frames, device=None, **self.policy)
        self.orc = OraclePagedKV(1, w.page_size, w.num_heads, w.head_dim, w.dtype, w.scale_frames,
                                 w.sliding_window, w.headroom, w.max_total_frames, mirror_blocks=(),
                                 **self.policy)
        bits = np.uint32 if w.dtype == "f32" else np.uint16
        self.dummy = np.zeros((w.tokens_per_frame, w.num_heads, w.head_dim), bits)
        self.plans = 0

    def append(self, b, f):
        self.lib.append_frame(b)
        if b == 0:
            self.orc.append_frame(0, self.dummy, self.dummy)

    def evict(self, b):
        if self.policy["cross_frame_special"] and not self.policy["camera_only"]:
            self.lib.evict_frames(b)
        else:
            self.lib.evict_frames(b, **self.policy)       # kvc_evict_frames_ex
        if b == 0:
            self.orc.evict_frames(0, self.w.scale_frames, self.w.sliding_window, **self.policy)

    def set_defer(self, on):
        self.lib.set_defer_eviction(on)
        self.orc.set_defer_eviction(on)

    def execute(self, b):
        self.lib.execute_deferred_eviction(b)
        if b == 0:
            self.orc.execute_deferred_eviction(0, self.w.scale_frames, self.w.sliding_window)

    def rollback(self, b):
        self.lib.rollback_last_frame(b)
        if b == 0:
            self.orc.rollback_last_frame(0)

    def clean(self):
        self.lib.clean()
        self.orc.clean()

    def plan(self):
        self.lib.plan()
        idx, indptr, lpl = self.lib.plan_table()
        o_idx, o_indptr, o_lpl, _ = self.orc.visible_page_table(0)
        assert (idx, indptr, lpl) == (o_idx, o_indptr, o_lpl)
        assert tuple(self.lib.plan_ranges()) == tuple(self.orc.visible_ranges(0))
        self.plans += 1

    def attend(self, b, f):
        pass

    def after_frame(self, f, kind):
        want = self.orc.deques(0)
        for b in {0, self.w.num_layers - 1}:
            assert self.lib.deques(b) == tuple(want), (f, kind, b)
            assert self.lib.stats(b) == self.orc.stats(0), (f, kind, b)


@pytest.mark.parametrize("name", ["tiny", "s224", "defer", "s518", "win518"])
def test_bookkeeping_matches_oracle_full_length(kvc, name):
    w = WORKLOADS[name]
    eng = BothBook(kvc, w)
    drive(w, eng, attend=False)
    assert eng.plans == w.n_frames
    if name == "s518":
        assert eng.lib.stats(0) == {"frame_count": 2048, "scale_pages": 8, "live_pages": 64,
                                    "free_pages": 16, "special_tokens": 12288}
        idx, _, lpl = eng.lib.plan_table()
        assert len(idx) == 85 and lpl == 336


def test_errors_match_oracle_on_random_ops(kvc):
    rng = np.random.default_rng(2024)
    lib = kvc.PagedKVCache(2, 2, 32, 16, "f32", 2, 4, 2, 24, device=None)
    orc = OraclePagedKV(2, 16, 2, 32, "f32", 2, 4, 2, 24, mirror_blocks=())
    z = np.zeros((22, 2, 32), np.uint32)
    for step in range(3000):
        op = int(rng.integers(0, 8))
        b = int(rng.integers(0, 2))
        lib_err = orc_err = None
        calls = {
            0: (lambda: lib.append_frame(b), lambda: orc.append_frame(b, z, z)),
            1: (lambda: lib.append_frame(b), lambda: orc.append_frame(b, z, z)),
            2: (lambda: lib.evict_frames(b), lambda: orc.evict_frames(b, 2, 4)),
            3: (lambda: lib.rollback_last_frame(b), lambda: orc.rollback_last_frame(b)),
            4: (lambda: lib.execute_deferred_eviction(b), lambda: orc.execute_deferred_eviction(b, 2, 4)),
            5: (lambda: lib.set_defer_eviction(rng.random() < 0.5), None),
            6: (lambda: lib.rollback_last_frame(b), lambda: orc.rollback_last_frame(b)),
            7: (lambda: lib.clean(), lambda: orc.clean()),
        }
        if op == 7 and rng.random() < 0.9:
            continue
        lf, of = calls[op]
        if op == 5:
            on = bool(rng.random() < 0.5)
            lib.set_defer_eviction(on)
            orc.set_defer_eviction(on)
            continue
        try:
            lf()
        except kvc.KvcError as e:
            lib_err = e.code
        try:
            of()
        except OracleError as e:
            orc_err = e.code
        assert lib_err == orc_err, (step, op, lib_err, orc_err)
        for bb in range(2):
            assert lib.deques(bb) == tuple(orc.deques(bb))
            assert lib.stats(bb) == orc.stats(bb)


def test_plan_and_run_preconditions(kvc):
    lib = kvc.PagedKVCache(2, 2, 32, 16, "f32", 2, 4, 2, 16, device=None)
    with pytest.raises(kvc.KvcError) as e:
        lib.plan()
    assert e.value.code == "EMPTY"
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_get_plan(lib.h)
    assert e.value.code == "NO_PLAN"
    with pytest.raises(kvc.KvcError) as e:
        lib.evict_frames(0, scale_frames=3)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(kvc.KvcError) as e:
        lib.append_frame(2)
    assert e.value.code == "INVALID_ARG"
    for _ in range(16):
        lib.append_frame(0)
        lib.evict_frames(0)
    with pytest.raises(kvc.KvcError) as e:
        lib.append_frame(0)
    assert e.value.code == "SPECIAL_POOL_FULL"


@pytest.mark.parametrize("cross,cam", [(False, False), (True, True), (False, True)])
@pytest.mark.parametrize("name", ["tiny", "defer", "s518", "win518"])
def test_special_policy_plans_match_oracle_every_frame(kvc, name, cross, cam):
    """The special-token policies (cross_frame_special off; camera_only):
    visible row ranges, deques and stats equal the oracle's at every frame,
    through deferral, rollback and window resets."""
    w = WORKLOADS[name]
    if name == "win518":
        w = w.with_(n_frames=w.window_frames + 40)
    e = BothBook(kvc, w.with_(num_layers=min(w.num_layers, 2)), cross_frame_special=cross, camera_only=cam)
    drive(w.with_(num_layers=min(w.num_layers, 2)), e)
    assert e.plans > 0
    e.lib.close()


def test_special_policy_evict_arguments_must_match(kvc):
    c = kvc.PagedKVCache(1, 2, 32, 16, "f32", 2, 4, 2, 16, device=None, cross_frame_special=False)
    c.append_frame(0)
    c.evict_frames(0, cross_frame_special=False, camera_only=False)
    for kw in ({"cross_frame_special": True}, {"camera_only": True}):
        with pytest.raises(kvc.KvcError) as e:
            c.evict_frames(0, **kw)
        assert e.value.code == "INVALID_ARG"
    with pytest.raises(kvc.KvcError):
        kvc.kvc_required_bytes(kvc.make_config(1, 2, 32, 16, "f32").__class__(
            *[getattr(kvc.make_config(1, 2, 32, 16, "f32"), f) for f, _ in kvc.kvc_config._fields_[:-1]], 7))
    g = kvc.kvc_get_geometry(kvc.make_config(1, 16, 64, 999, camera_only=True))
    assert (g.num_camera_pages, g.max_num_pages) == (3, 88 + 13 + 3)
    assert kvc.kvc_get_geometry(kvc.make_config(1, 16, 64, 999)).num_camera_pages == 0
    c.close()


def test_free_pool_exhausted_by_deferred_frames(kvc):
    """More provisional frames than the pool holds: with eviction deferred
    the window keeps growing until no patch page is free; the next append
    returns NO_FREE_PAGE and changes nothing; rolling the provisional frames
    back restores the pool exactly (the same failure on the oracle)."""
    lib = kvc.PagedKVCache(1, 2, 32, 16, "f32", 2, 4, 2, 64, device=None)
    orc = OraclePagedKV(1, 16, 2, 32, "f32", 2, 4, 2, 64, mirror_blocks=())
    z = np.zeros((22, 2, 32), np.uint32)
    for _ in range(6):                           # scale 2 + window 4, committed
        lib.append_frame(0); lib.evict_frames(0)
        orc.append_frame(0, z, z); orc.evict_frames(0, 2, 4)
    before = lib.deques(0)
    lib.set_defer_eviction(True); orc.set_defer_eviction(True)
    for _ in range(2):                           # headroom 2: the pool is now empty
        lib.append_frame(0); lib.evict_frames(0)
        orc.append_frame(0, z, z); orc.evict_frames(0, 2, 4)
    full = (lib.deques(0), lib.stats(0))
    assert full[1]["free_pages"] == 0
    with pytest.raises(kvc.KvcError) as e:
        lib.append_frame(0)
    assert e.value.code == "NO_FREE_PAGE"
    with pytest.raises(OracleError) as oe:
        orc.append_frame(0, z, z)
    assert oe.value.code == "NO_FREE_PAGE"
    assert (lib.deques(0), lib.stats(0)) == full          # the failed call changed nothing
    for _ in range(2):
        lib.rollback_last_frame(0); orc.rollback_last_frame(0)
    assert lib.deques(0) == before == tuple(orc.deques(0))
    # No eviction has moved a page, so the first six frames are still
    # uncommitted (an eviction commits only when it moves a page): rollback
    # goes on undoing them, on both sides, until nothing is left.
    for _ in range(6):
        lib.rollback_last_frame(0); orc.rollback_last_frame(0)
        assert lib.deques(0) == tuple(orc.deques(0)) and lib.stats(0) == orc.stats(0)
    with pytest.raises(kvc.KvcError) as e:
        lib.rollback_last_frame(0)
    assert e.value.code == "NOTHING_TO_ROLLBACK"
    lib.close()
