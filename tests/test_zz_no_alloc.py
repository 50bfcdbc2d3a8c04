"""kvc_paged_attention_static -- the entry point for callers that cannot
allocate device memory (for example code inside a host framework that owns
all GPU memory and lends out only the KV cache and the Q / output buffers, so
it has no workspace to give kvc_create).  It keeps its scratch in an array
inside the library.  Checked here through the C ABI, each time on two calls in
a row (the second sees the first call's leftovers in the array):

* bf16, head_dim 64, 999-row pages, against the CPU oracle and against what
  kvc_run gives for the same cache and queries;
* the fp32 tiny geometry (H=2, D=32, 16-row pages) against the oracle at 1e-4;
* head_dim 128 (32-row KV tiles) against the oracle;
* a query count whose split-KV partials fit the array for two splits only, so
  that the split count is cut by the array's size;
* the size limits, which are rejected before any device work.

This file is named to be collected last, so that a run that stops at the first
failure has run every other test before it.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ABS, REL_RMS = 2e-2, 5e-3          # the bf16 tolerance of the parity tests
F32_TOL = 1e-4                         # the fp32 tolerance of the parity tests


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _diff(got, want):
    """(max-abs, relative RMS) of a device tensor against a float64 array or tensor."""
    g = got.detach().to("cpu", torch.float64).numpy()
    w = want.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(want) else want
    return float(np.abs(g - w).max()), float(np.linalg.norm(g - w) / np.linalg.norm(w))


class _Pair:
    """A device cache (through the library) and the oracle fed the same frames."""

    def __init__(self, kvc, H, D, ps, dtype, scale_frames=8, window=64, headroom=16, max_frames=64,
                 seed=3, wid=77):
        from oracle import OraclePagedKV
        self.kvc, self.H, self.D, self.ps, self.dtype = kvc, H, D, ps, dtype
        self.seed, self.wid = seed, wid
        self.scale_frames, self.window = scale_frames, window
        self.c = kvc.PagedKVCache(1, H, D, ps, dtype, scale_frames=scale_frames, sliding_window=window,
                                  headroom=headroom, max_total_frames=max_frames)
        self.orc = OraclePagedKV(1, ps, H, D, dtype, scale_frames, window, headroom, max_frames)

    def frame(self, f):
        from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
        q, k, v = frame_qkv(self.seed, self.wid, f, 0, self.ps, self.H, self.D, self.dtype)
        self.c.append_frame(0, k.cuda(), v.cuda())
        self.orc.append_frame(0, to_bits(k), to_bits(v))
        self.c.evict_frames(0)
        self.orc.evict_frames(0, self.scale_frames, self.window)
        self.c.plan()
        return q

    def pages(self):
        """The visible page list the library planned, checked against the oracle's."""
        ids, _, _ = self.kvc.kvc_get_plan(self.c.h)
        _, valid, _ = self.kvc.kvc_read_device_plan(self.c.h, self.c._stream())
        o_ids, _, _, o_valid = self.orc.visible_page_table(0)
        assert list(ids) == list(o_ids) and list(valid) == list(o_valid)
        return ids, valid

    def static(self, qd, out, ids, valid):
        self.kvc.kvc_paged_attention_static(self.c.cache.data_ptr(), self.dtype, self.H, self.D, self.ps,
                                            ids, valid, qd.data_ptr(), out.data_ptr(), qd.shape[0], 0.0,
                                            self.c._stream())

    def want(self, q, rows=None):
        from oracle import paged_attention
        from streaming_paged_kv_gb300.inputs import to_bits
        return paged_attention(self.orc, 0, to_bits(q), rows=rows)


def test_static_scratch_matches_oracle_and_kvc_run_two_calls_in_a_row(kvc):
    p = _Pair(kvc, 16, 64, 999, "bf16", scale_frames=2, window=3, headroom=2)
    checked = 0
    for f in range(7):
        q = p.frame(f)
        if f < 5:
            continue
        qd = q.cuda()
        ref = torch.empty_like(qd)
        p.c.run(0, qd, ref)
        ids, valid = p.pages()
        want = p.want(q)
        for _ in range(2):                      # two calls in a row share the array
            out = torch.full_like(qd, float("nan"))
            p.static(qd, out, ids, valid)
            torch.cuda.synchronize()
            for mx, rel in (_diff(out, want), _diff(out, ref)):
                assert mx <= MAX_ABS and rel <= REL_RMS, (f, mx, rel)
            checked += 1
    assert checked == 4
    p.c.close()


def test_static_scratch_f32_tiny_against_oracle(kvc):
    p = _Pair(kvc, 2, 32, 16, "f32", scale_frames=2, window=4, headroom=2, max_frames=16, seed=0, wid=1)
    for f in range(12):
        q = p.frame(f)
        if f not in (0, 5, 11):
            continue
        ids, valid = p.pages()
        want = p.want(q)
        qd = q.cuda()
        for _ in range(2):
            out = torch.full_like(qd, float("nan"))
            p.static(qd, out, ids, valid)
            torch.cuda.synchronize()
            mx, _ = _diff(out, want)
            assert mx <= F32_TOL, (f, mx)
    p.c.close()


def test_static_scratch_head_dim_128(kvc):
    # 32-row KV tiles: a 256-row page is 8 tiles.
    p = _Pair(kvc, 8, 128, 256, "bf16", scale_frames=2, window=4, headroom=2, seed=5, wid=2)
    for f in range(9):
        q = p.frame(f)
    ids, valid = p.pages()
    want = p.want(q)
    qd = q.cuda()
    for _ in range(2):
        out = torch.full_like(qd, float("nan"))
        p.static(qd, out, ids, valid)
        torch.cuda.synchronize()
        mx, rel = _diff(out, want)
        assert mx <= MAX_ABS and rel <= REL_RMS, (mx, rel)
    p.c.close()


def test_static_scratch_split_count_cut_by_the_array(kvc):
    """2900 query rows x 16 heads: one split's partials (O and log-sum-exp,
    fp32) take 2900 * 16 * 65 * 4 B = 12.1 MB, so the 32 MiB array holds two
    splits; the wave model alone would take three or more (23 query tiles x
    16 heads = 368 CTAs per split on the GPU's SMs)."""
    p = _Pair(kvc, 16, 64, 256, "bf16", seed=9, wid=2)
    for f in range(20):
        p.frame(f)
    ids, valid = p.pages()
    rng = np.random.default_rng(12)
    q = torch.from_numpy(rng.standard_normal((2900, 16, 64)).astype(np.float32)).to(torch.bfloat16)
    rows = list(range(0, 2900, 7)) + [2899]
    want = p.want(q, rows)
    qd = q.cuda()
    sel = torch.as_tensor(rows, device="cuda")
    for _ in range(2):
        out = torch.full_like(qd, float("nan"))
        p.static(qd, out, ids, valid)
        torch.cuda.synchronize()
        assert not torch.isnan(out).any()
        mx, rel = _diff(out[sel], want)
        assert mx <= MAX_ABS and rel <= REL_RMS, (mx, rel)
    p.c.close()


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
