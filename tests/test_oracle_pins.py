"""Pins of the CPU oracle to facts it does not produce itself.

* numbers the pages print (``tests/golden/page_facts.json``, each cited),
* page tables worked out by hand from the pages' rules for the tiny stream,
* invariants the pages state (healthy stats, rollback restores the slot
  exactly, reset = construction state, memory constant),
* paging transparency: attention over the paged cache equals attention over
  the frame-level visible token set built straight from the inputs,
* closed forms of softmax attention, a textbook triple loop and the library
  routine (torch SDPA in float64),
* planted mistakes in copies of the oracle that these pins must catch.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import OraclePagedKV, OracleError, dense_attention, paged_attention, prefill_attention
from oracle.attention import bits_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")
FACTS = json.load(open(GOLDEN, encoding="utf-8"))


def _tiny(**kw):
    args = dict(num_blocks=1, page_size=16, num_heads=2, head_dim=32, dtype="f32",
                scale_frames=2, sliding_window=4, headroom=2, max_total_frames=16)
    args.update(kw)
    return OraclePagedKV(**args)


def _f32_frame(rng, T, H, D):
    x = rng.standard_normal((T, H, D)).astype(np.float32)
    return x, x.view(np.uint32)


def _stream(cache, block, n, rng=None, window=None):
    window = cache.sliding_window if window is None else window
    T, H, D = cache.tokens_per_frame, cache.num_heads, cache.head_dim
    for _ in range(n):
        if rng is None:
            kb = np.zeros((T, H, D), np.uint16 if cache.dtype != "f32" else np.uint32)
            vb = kb
        else:
            _, kb = _f32_frame(rng, T, H, D)
            _, vb = _f32_frame(rng, T, H, D)
        cache.append_frame(block, kb, vb)
        cache.evict_frames(block, cache.scale_frames, window)


# ------------------------------------------------------------ page facts
def test_pool_sizes_printed_by_the_pages():
    f = FACTS["patch_pool"]
    c = OraclePagedKV(1, 256, 1, 8, "bf16", f["scale_frames"], f["sliding_window"],
                      f["headroom"], mirror_blocks=())
    assert c.num_patch_pages == f["total_pages"] == 88
    sp = FACTS["special_packing"]
    assert c.frames_per_special_page == sp["frames_per_page"] == 42
    assert c.max_total_frames == sp["default_max_total_frames"]
    ft = FACTS["frame_tokens_224"]
    assert c.tokens_per_frame == ft["tokens_per_frame"] == ft["patch_tokens"] + ft["special_tokens"]


def test_example_stream_healthy_stats():
    """[PERF] 'Minimal Streaming Inference Setup' run on block 0, checked against
    the healthy values of [SLOTS] '动手验证' at every frame."""
    ex, hs = FACTS["example_stream"], FACTS["healthy_stats"]
    c = OraclePagedKV(1, ex["tokens_per_frame"] - 6, ex["num_heads"], ex["head_dim"], "bf16",
                      ex["scale_frames"], ex["sliding_window"],
                      ex["max_num_frames"] - ex["scale_frames"] - ex["sliding_window"],
                      ex["max_total_frames"], mirror_blocks=())
    for f in range(ex["frames"]):
        _stream(c, 0, 1)
        s = c.stats(0)
        assert set(s) == set(hs["fields"])
        assert s["scale_pages"] == min(f + 1, hs["scale_pages"])
        assert s["live_pages"] <= hs["live_pages_max"]
        assert s["special_tokens"] == hs["special_tokens_per_frame"] * (f + 1)
        assert s["scale_pages"] + s["live_pages"] + s["free_pages"] == ex["max_num_frames"]
    assert c.stats(0) == {"frame_count": 100, "scale_pages": 8, "live_pages": 64,
                          "free_pages": 16, "special_tokens": 600}


def test_window_mode_span():
    from streaming_paged_kv_gb300.workloads import WORKLOADS, schedule
    wm = FACTS["window_mode"]
    w = WORKLOADS["win518"]
    assert w.window_slots == wm["window_size_slots"]
    assert w.scale_frames == wm["scale_slots"]
    assert w.window_frames == wm["frames_per_window"] == 1568
    ev = [k for f, k in schedule(w.with_(n_frames=wm["frames_per_window"]))]
    assert ev[0] == "clean" and ev.count("clean") == 1
    assert ev.count("key") == wm["window_size_slots"]


# ------------------------------------------------- hand-derived page tables
# Tiny stream (scale 2, window 4, headroom 2 => P = 8 patch pages 0..7; page
# size 16 => 2 frames per special page, special pages 8..15).  Worked by hand
# from the rules: allocation takes the left of the free list, the first 2 pages
# go to scale, later ones to the live window, eviction moves the oldest live
# page to the right of the free list once the window holds more than 4.
#   frames 0,1 -> pages 0,1 (scale)        frames 2..5 -> pages 2..5 (live)
#   frame 6 -> page 6, evict 2 (free 7,2)  frame 7 -> page 7, evict 3 (free 2,3)
#   frame 8 -> page 2, evict 4 (free 3,4)  frame 9 -> page 3, evict 5 (free 4,5)
#   frame 10 -> page 4, evict 6 (free 5,6) frame 11 -> page 5, evict 7 (free 6,7)
# Specials of s frames take ceil(s/2) pages; the last holds 6*(s - 2*(ceil(s/2)-1)).
HAND_TABLES = {
    7: ([0, 1, 3, 4, 5, 6, 8, 9, 10, 11], 6, [7, 2]),
    9: ([0, 1, 5, 6, 7, 2, 8, 9, 10, 11, 12], 6, [3, 4]),
    12: ([0, 1, 2, 3, 4, 5, 8, 9, 10, 11, 12, 13], 12, [6, 7]),
}


def _check_hand_tables(cache_cls):
    c = cache_cls(num_blocks=1, page_size=16, num_heads=2, head_dim=32, dtype="f32",
                  scale_frames=2, sliding_window=4, headroom=2, max_total_frames=16,
                  mirror_blocks=())
    bad = []
    for n in range(1, 13):
        _stream(c, 0, 1)
        if n in HAND_TABLES:
            idx, _, lpl, _ = c.visible_page_table(0)
            want_idx, want_lpl, want_free = HAND_TABLES[n]
            if idx != want_idx or lpl != want_lpl or c.deques(0)[2] != want_free:
                bad.append((n, idx, lpl, c.deques(0)[2]))
    return bad


def test_tiny_page_tables_match_hand_derivation():
    assert _check_hand_tables(OraclePagedKV) == []


# Special-token policies (the reading of the eviction options cross_frame_special
# and camera_only, [KVC] "Streaming Forward Pass"), same tiny stream.  The
# frames of the scale pages are 0 and 1, the live window holds the newest
# four; the special stream position of a frame is its append order, 2 frames
# per special page (frame f: page 8 + f // 2, rows 6 (f % 2) .. +6).  With
# camera_only one camera page follows the 8 special pages: page 16, camera
# position f = row f.  Worked by hand:
#   after 5 frames: nothing evicted yet (frames 0-1 scale, 2-4 live): every
#     special of frames 0-4 -- pages 8, 9 (rows 0-11) and 10 (rows 0-5).
#   after 7 frames: frame 2 evicted.  Scale specials: page 8 rows 0-11; live
#     frames 3-6: frame 3 = page 9 rows 6-11, frames 4-5 = page 10 rows 0-11,
#     frame 6 = page 11 rows 0-5.  camera_only adds camera page 16 row 2.
#   after 12 frames: frames 2-7 evicted.  Scale: page 8 rows 0-11; live frames
#     8-11: pages 12 and 13 rows 0-11.  camera_only adds page 16 rows 2-7.
POLICY_TABLES = {
    5: ([(8, 0, 12), (9, 0, 12), (10, 0, 6)], []),
    7: ([(8, 0, 12), (9, 6, 6), (10, 0, 12), (11, 0, 6)], [(16, 2, 1)]),
    12: ([(8, 0, 12), (12, 0, 12), (13, 0, 12)], [(16, 2, 6)]),
}


def _check_policy_tables(cache_cls):
    bad = []
    for cross, cam in ((False, False), (True, True), (False, True)):
        c = cache_cls(num_blocks=1, page_size=16, num_heads=2, head_dim=32, dtype="f32",
                      scale_frames=2, sliding_window=4, headroom=2, max_total_frames=16,
                      mirror_blocks=(), cross_frame_special=cross, camera_only=cam)
        for n in range(1, 13):
            _stream(c, 0, 1)
            if n not in POLICY_TABLES:
                continue
            idx, first, valid = c.visible_ranges(0)
            scale, live, _ = c.deques(0)
            special, camera = POLICY_TABLES[n]
            want = [(p, 0, 16) for p in scale + live] + special + (camera if (cross and cam) else [])
            if list(zip(idx, first, valid)) != want:
                bad.append((cross, cam, n, list(zip(idx, first, valid))))
    return bad


def test_special_policy_tables_match_hand_derivation():
    assert _check_policy_tables(OraclePagedKV) == []
    # The default policy is the pages' two-stream table: every special page from row 0.
    c = _tiny(mirror_blocks=())
    _stream(c, 0, 12)
    idx, first, valid = c.visible_ranges(0)
    assert first == [0] * len(idx) and idx == HAND_TABLES[12][0]


def test_special_policy_arguments_must_match_the_construction():
    c = _tiny(mirror_blocks=(), cross_frame_special=False)
    _stream(c, 0, 1)
    c.evict_frames(0, 2, 4, cross_frame_special=False, camera_only=False)
    for kw in ({"cross_frame_special": True}, {"camera_only": True}):
        with pytest.raises(OracleError) as e:
            c.evict_frames(0, 2, 4, **kw)
        assert e.value.code == "INVALID_ARG"
    # camera pages exist only with cross-frame specials kept camera-only
    assert _tiny(camera_only=True).max_num_pages == 8 + 8 + 1
    assert _tiny(camera_only=True, cross_frame_special=False).max_num_pages == 16
    assert _tiny().max_num_pages == 16


def test_full_size_end_states():
    # 518x378: 2048 frames, 166 frames per special page -> 13 special pages 88..100,
    # last page holds 2048 - 12*166 = 56 frames = 336 tokens.
    c = OraclePagedKV(1, 999, 16, 64, "bf16", 8, 64, 16, 2048, mirror_blocks=())
    _stream(c, 0, 2048)
    idx, indptr, lpl, valid = c.visible_page_table(0)
    assert len(idx) == 85 and idx[72:] == list(range(88, 101)) and indptr == [0, 85]
    assert lpl == 336 and valid[72:84] == [996] * 12 and valid[:72] == [999] * 72
    assert c.stats(0) == {"frame_count": 2048, "scale_pages": 8, "live_pages": 64,
                          "free_pages": 16, "special_tokens": 12288}
    assert sum(valid) == 72 * 999 + 6 * 2048
    with pytest.raises(OracleError) as e:
        _stream(c, 0, 1)
    assert e.value.code == "SPECIAL_POOL_FULL"
    # 224x224 after 200 frames: 42 frames per special page -> 5 pages, last holds 32 frames.
    c = OraclePagedKV(1, 256, 16, 64, "bf16", 8, 64, 16, 2048, mirror_blocks=())
    _stream(c, 0, 200)
    idx, _, lpl, valid = c.visible_page_table(0)
    assert len(idx) == 77 and lpl == 192 and c.stats(0)["special_tokens"] == 1200
    assert sum(valid) == 72 * 256 + 1200


# -------------------------------------------------------------- invariants
def _snapshot(c, block):
    idx, indptr, lpl, valid = c.visible_page_table(block)
    k, v = c.gather_visible(block) if block in c.mirror else (None, None)
    return (c.deques(block), c.stats(block), idx, indptr, lpl, valid,
            None if k is None else k.copy(), None if v is None else v.copy())


def _same(a, b):
    for x, y in zip(a, b):
        if isinstance(x, np.ndarray):
            if not np.array_equal(x, y):
                return False
        elif x != y:
            return False
    return True


def test_deferred_example_from_the_pages():
    """[PERF] 'Deferred Eviction for Keyframe Decisions': five appends with
    eviction deferred, then execute (commits) or rollback (undoes the last)."""
    c = OraclePagedKV(1, 256, 2, 8, "bf16", 8, 64, 16, 200, mirror_blocks=())
    _stream(c, 0, 72)                       # scale full, window full
    c.set_defer_eviction(True)
    _stream(c, 0, 5)
    assert c.stats(0)["live_pages"] == 69 and c.stats(0)["free_pages"] == 11
    before_last = None
    c2 = OraclePagedKV(1, 256, 2, 8, "bf16", 8, 64, 16, 200, mirror_blocks=())
    _stream(c2, 0, 72)
    c2.set_defer_eviction(True)
    _stream(c2, 0, 4)
    before_last = _snapshot(c2, 0)
    _stream(c2, 0, 1)
    c2.rollback_last_frame(0)
    assert _same(_snapshot(c2, 0), before_last)
    c.execute_deferred_eviction(0, 8, 64)
    assert c.stats(0)["live_pages"] == 64 and c.stats(0)["free_pages"] == 16
    with pytest.raises(OracleError) as e:
        c.rollback_last_frame(0)
    assert e.value.code == "NOTHING_TO_ROLLBACK"


def test_rollback_restores_exactly_random_ops():
    """Append + rollback is the identity on deques, counters, visible table and
    visible bytes ([SLOTS] '光流关键帧与回滚机制': the slot is fully restored)."""
    rng = np.random.default_rng(7)
    c = _tiny(max_total_frames=64)
    P = c.num_patch_pages
    for step in range(400):
        op = rng.integers(0, 6)
        try:
            if op <= 2:
                snap = _snapshot(c, 0)
                _, kb = _f32_frame(rng, 22, 2, 32)
                _, vb = _f32_frame(rng, 22, 2, 32)
                c.append_frame(0, kb, vb)
                if rng.random() < 0.5:
                    c.rollback_last_frame(0)
                    assert _same(_snapshot(c, 0), snap)
            elif op == 3:
                c.evict_frames(0, 2, 4)
            elif op == 4:
                c.set_defer_eviction(rng.random() < 0.5)
            else:
                c.execute_deferred_eviction(0, 2, 4)
        except OracleError as e:
            assert e.code in ("NO_FREE_PAGE", "SPECIAL_POOL_FULL", "NOTHING_TO_ROLLBACK")
            if e.code == "SPECIAL_POOL_FULL":
                c.clean()
        s, l, f = c.deques(0)
        assert len(s) + len(l) + len(f) == P
        assert sorted(s + l + f) == list(range(P))
        assert len(s) <= c.scale_frames
        idx = c.visible_page_table(0)[0]
        assert len(idx) == len(set(idx))


def test_failed_calls_leave_state_unchanged():
    c = _tiny()
    _stream(c, 0, 6)                          # scale 2 + live 4: window full
    c.set_defer_eviction(True)
    _stream(c, 0, 2)                          # uses the 2 headroom pages
    snap = _snapshot(c, 0)
    z = np.zeros((22, 2, 32), np.uint32)
    with pytest.raises(OracleError) as e:
        c.append_frame(0, z, z)
    assert e.value.code == "NO_FREE_PAGE" and _same(_snapshot(c, 0), snap)
    with pytest.raises(OracleError):
        c.append_frame(0, z[:5], z[:5])
    assert _same(_snapshot(c, 0), snap)
    with pytest.raises(OracleError):
        c.evict_frames(0, 3, 4)               # scale_frames differs from the constructor's
    with pytest.raises(OracleError):
        c.append_frame(1, z, z)               # no such block


def test_clean_is_construction_state():
    c = _tiny(num_blocks=2)
    fresh = [_snapshot(_tiny(num_blocks=2), b)[:6] for b in range(2)]
    for b in range(2):
        _stream(c, b, 9, np.random.default_rng(b))
    c.set_defer_eviction(True)
    c.clean()
    assert not c.defer_eviction
    for b in range(2):
        assert _same(_snapshot(c, b)[:6], fresh[b])


# ---------------------------------------------------- paging transparency
def _sdpa64(q, k, v):
    """Library routine: torch scaled_dot_product_attention in float64, [N,H,D] layout."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    return o[0].permute(1, 0, 2).numpy()


def _check_transparency(cache_cls, mode="stream", seed=3, n=12, cross=True, cam=False):
    """Attention over the paged cache vs attention over the frame-level
    visible set: patch tokens of the scale frames, of the live frames, then the
    special tokens of every kept frame in order ([SLOTS] '双流分页布局': visible
    range = scale pages + window pages + all special pages).  With the
    special-token policies: without cross-frame specials only the scale and
    live frames' specials; with camera_only those plus the camera token (row
    0) of every other kept frame."""
    rng = np.random.default_rng(seed)
    c = cache_cls(num_blocks=1, page_size=16, num_heads=2, head_dim=32, dtype="f32",
                  scale_frames=2, sliding_window=4, headroom=3, max_total_frames=16,
                  cross_frame_special=cross, camera_only=cam)
    kept = []                                   # (k, v) of committed or pending frames
    worst = 0.0
    for f in range(n):
        kf, kb = _f32_frame(rng, 22, 2, 32)
        vf, vb = _f32_frame(rng, 22, 2, 32)
        qf, qb = _f32_frame(rng, 22, 2, 32)
        provisional = mode == "defer" and f >= 2
        c.set_defer_eviction(provisional)
        c.append_frame(0, kb, vb)
        c.evict_frames(0, 2, 4)
        kept.append((kf, vf))
        scale_fr = kept[:2]
        # The window held at most 4 committed frames before this append; a
        # provisional frame sits on top of them until the decision.
        if provisional:
            n_live = min(4, len(kept) - 3) + 1
        else:
            n_live = min(4, max(0, len(kept) - 2))
        live_fr = kept[len(kept) - n_live:] if n_live > 0 else []
        evicted = kept[2:len(kept) - n_live]
        if cross and not cam:
            spec = [x[:6] for x, _ in kept], [y[:6] for _, y in kept]
        else:
            window = scale_fr + live_fr
            spec = [x[:6] for x, _ in window], [y[:6] for _, y in window]
            if cross and cam:
                spec = spec[0] + [x[:1] for x, _ in evicted], spec[1] + [y[:1] for _, y in evicted]
        K = np.concatenate([x[6:] for x, _ in scale_fr + live_fr] + spec[0])
        V = np.concatenate([y[6:] for _, y in scale_fr + live_fr] + spec[1])
        want = _sdpa64(qf.astype(np.float64), K.astype(np.float64), V.astype(np.float64))
        got = paged_attention(c, 0, qb)
        worst = max(worst, float(np.abs(got - want).max()))
        if provisional:
            if rng.random() < 0.5:
                c.rollback_last_frame(0)
                kept.pop()
            else:
                c.execute_deferred_eviction(0, 2, 4)
    return worst


def test_paging_is_transparent_stream():
    assert _check_transparency(OraclePagedKV, "stream") < 1e-12


def test_paging_is_transparent_defer():
    assert _check_transparency(OraclePagedKV, "defer", seed=5, n=16) < 1e-12


@pytest.mark.parametrize("cross,cam", [(False, False), (True, True), (False, True)])
@pytest.mark.parametrize("mode", ["stream", "defer"])
def test_paging_is_transparent_special_policies(cross, cam, mode):
    assert _check_transparency(OraclePagedKV, mode, seed=7, n=16, cross=cross, cam=cam) < 1e-12


def test_cache_bytes_are_the_frame_rows():
    rng = np.random.default_rng(11)
    c = _tiny()
    for s in range(5):
        _, kb = _f32_frame(rng, 22, 2, 32)
        _, vb = _f32_frame(rng, 22, 2, 32)
        page = c.append_frame(0, kb, vb)
        m = c.mirror[0]
        assert np.array_equal(m[page, 0], kb[6:]) and np.array_equal(m[page, 1], vb[6:])
        sp, slot = 8 + s // 2, 6 * (s % 2)
        assert np.array_equal(m[sp, 0, slot:slot + 6], kb[:6])
        assert np.array_equal(m[sp, 1, slot:slot + 6], vb[:6])


# ------------------------------------------------------ attention pins
def _brute(q, k, v, scale):
    """Textbook triple loop with the max-subtracted softmax, pure Python."""
    nq, h, d = q.shape
    out = np.zeros((nq, h, v.shape[2]))
    for t in range(nq):
        for hh in range(h):
            logits = [sum(q[t, hh, i] * k[j, hh, i] for i in range(d)) * scale
                      for j in range(k.shape[0])]
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            for i in range(v.shape[2]):
                out[t, hh, i] = sum(w[j] * v[j, hh, i] for j in range(k.shape[0])) / z
    return out


def _check_attention(fn):
    """Residuals of an attention implementation against the pins (inf when
    the implementation cannot even evaluate a case)."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((5, 2, 8))
    k = rng.standard_normal((9, 2, 8))
    v = rng.standard_normal((9, 2, 8))
    kk = np.repeat(k[:1], 9, axis=0)
    perm = rng.permutation(9)
    kd = k.copy()
    kd[4] = q[0] * 1e3          # one logit dominates by far: no overflow, output = that value
    cases = {
        "brute": lambda: fn(q, k, v) - _brute(q, k, v, 1 / math.sqrt(8)),
        "sdpa": lambda: fn(q, k, v) - _sdpa64(q, k, v),
        "q0_mean_v": lambda: fn(np.zeros_like(q), k, v) - v.mean(axis=0)[None],
        "equal_keys_mean_v": lambda: fn(q, kk, v) - v.mean(axis=0)[None],
        "one_token": lambda: fn(q, k[:1], v[:1]) - v[:1],
        "const_v": lambda: fn(q, k, np.full_like(v, 2.5)) - 2.5,
        "perm": lambda: fn(q, k[perm], v[perm]) - fn(q, k, v),
        "dominant": lambda: fn(q[:1], kd, v) - v[4][None],
        # V = identity exposes the probabilities themselves: rows sum to 1.
        "rows_sum_1": lambda: fn(q, k, np.eye(9)[:, None, :].repeat(2, axis=1)).sum(axis=2) - 1,
    }
    r = {}
    for name, case in cases.items():
        try:
            r[name] = float(np.abs(case()).max())
        except ValueError:
            r[name] = float("inf")
    return r


def test_dense_attention_pins():
    r = _check_attention(dense_attention)
    assert max(r.values()) < 1e-12, r


def test_prefill_is_paged_attention_of_an_empty_cache_after_the_appends():
    """Phase 1 ([KVC] "FlashInferAttention Layer Implementation"): dense
    attention over the frames' own tokens.  Appending them to an empty cache
    makes the visible set exactly those tokens (in page order: patches of each
    frame, then the specials), so the oracle's paged path -- gathered pages,
    written independently of the concatenation -- must give the same result;
    so must any reordering of the frames' keys.  Bidirectional: frame 0's
    queries depend on the last frame's values."""
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    F, ps, H, D = 3, 16, 2, 32
    frames = [frame_qkv(7, 1, f, 0, ps, H, D, "f32") for f in range(F)]
    qb = [to_bits(q) for q, _, _ in frames]
    kb = [to_bits(k) for _, k, _ in frames]
    vb = [to_bits(v) for _, _, v in frames]
    want = prefill_attention(qb, kb, vb, "f32")
    orc = OraclePagedKV(1, ps, H, D, "f32", 2, 4, 2, 16)
    for f in range(F):
        orc.append_frame(0, kb[f], vb[f])
    paged = paged_attention(orc, 0, np.concatenate(qb))
    assert np.abs(paged - want).max() < 1e-12
    perm = [2, 0, 1]
    shuffled = dense_attention(bits_to_f64(np.concatenate(qb), "f32"),
                               bits_to_f64(np.concatenate([kb[i] for i in perm]), "f32"),
                               bits_to_f64(np.concatenate([vb[i] for i in perm]), "f32"))
    assert np.abs(shuffled - want).max() < 1e-12
    vb2 = list(vb)
    vb2[F - 1] = to_bits(frames[F - 1][2] + 1.0)
    changed = prefill_attention(qb, kb, vb2, "f32")
    T = ps + 6
    assert np.abs(changed[:T] - want[:T]).max() > 1e-3   # frame 0 sees the last frame


def test_bf16_and_f16_decoding_matches_torch():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(allbits.view(np.int16).copy())
    ref_bf = t.view(torch.bfloat16).to(torch.float64).numpy()
    got_bf = bits_to_f64(allbits, "bf16")
    ok = ~np.isnan(ref_bf)
    assert np.array_equal(got_bf[ok], ref_bf[ok]) and np.isnan(got_bf[~ok]).all()
    ref_h = t.view(torch.float16).to(torch.float64).numpy()
    got_h = bits_to_f64(allbits, "f16")
    ok = ~np.isnan(ref_h)
    assert np.array_equal(got_h[ok], ref_h[ok])


# --------------------------------------------------- planted mistakes
class _EvictToFront(OraclePagedKV):
    """Planted mistake: evicted pages go to the front of the free list."""

    def _evict(self, st, window, commit_always):
        moved = 0
        while len(st.live) > window:
            st.free.appendleft(st.live.popleft())
            moved += 1
        if moved or commit_always:
            st.undo.clear()
        return moved


class _FullSpecialPages(OraclePagedKV):
    """Planted mistake: every non-last special page counted as full (page_size)."""

    def visible_ranges(self, block=0):
        idx, first, valid = super().visible_ranges(block)
        n_patch = len(self.blocks[block].scale) + len(self.blocks[block].live)
        valid = [self.page_size if (i >= n_patch and i < len(valid) - 1) else n
                 for i, n in enumerate(valid)]
        return idx, first, valid


class _LiveBeforeScale(OraclePagedKV):
    """Planted mistake: live window listed before the scale pages."""

    def visible_page_table(self, block=0):
        idx, indptr, lpl, valid = super().visible_page_table(block)
        st = self.blocks[block]
        ns, nl = len(st.scale), len(st.live)
        return idx[ns:ns + nl] + idx[:ns] + idx[ns + nl:], indptr, lpl, valid


class _CameraRunOffByOne(OraclePagedKV):
    """Planted mistake: the evicted frames' camera run starts one frame late."""

    def visible_ranges(self, block=0):
        idx, first, valid = super().visible_ranges(block)
        if self.camera_stream and idx and idx[-1] >= self.first_camera_page and valid[-1] > 1:
            first[-1] += 1
            valid[-1] -= 1
        return idx, first, valid


class _EvictedSpecialsKept(OraclePagedKV):
    """Planted mistake: without cross-frame specials, the evicted frames'
    specials are still attended (the default table)."""

    def visible_ranges(self, block=0):
        if not self.cross_frame_special:
            self.cross_frame_special = True
            try:
                return super().visible_ranges(block)
            finally:
                self.cross_frame_special = False
        return super().visible_ranges(block)


def test_planted_mistakes_are_caught():
    assert _check_policy_tables(_CameraRunOffByOne) != []
    assert _check_policy_tables(_EvictedSpecialsKept) != []
    assert _check_transparency(_CameraRunOffByOne, seed=7, n=16, cam=True) > 1e-6
    assert _check_transparency(_EvictedSpecialsKept, seed=7, n=16, cross=False) > 1e-6
    assert _check_hand_tables(_EvictToFront) != []
    assert _check_hand_tables(_LiveBeforeScale) != []
    assert _check_transparency(_FullSpecialPages) > 1e-6

    def wrong_scale(q, k, v):
        return dense_attention(q, k, v, sm_scale=math.sqrt(q.shape[2]))

    def swapped_kv(q, k, v):
        return dense_attention(q, v, k)

    def no_max(q, k, v):            # forgets to normalise by the row sum
        out = np.empty_like(q)
        for h in range(q.shape[1]):
            s = q[:, h] @ k[:, h].T / math.sqrt(q.shape[2])
            p = np.exp(s - s.max(axis=1, keepdims=True))
            out[:, h] = p @ v[:, h]
        return out

    for bad in (wrong_scale, swapped_kv, no_max):
        assert max(_check_attention(bad).values()) > 1e-3
