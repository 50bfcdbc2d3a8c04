"""Phase 1 (batch mode) through the C ABI against the oracle.

kvc_prefill appends the first frames to an empty block and attends all their
queries over the block's visible tokens, which are exactly those frames'
tokens; the oracle computes the dense bidirectional attention of the frames
from their own Q/K/V ([KVC] "FlashInferAttention Layer Implementation",
Phase 1; [SLOTS] "scale frames永不驱逐").  Checked: outputs (tolerance of the
parity tests), cache bytes and bookkeeping after the prefill, streaming on top
of a prefilled cache, and the error cases leaving the bookkeeping unchanged.
"""

import numpy as np
import pytest
import torch

from gpu_engine import TOL, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc as mod
    return mod


def _frames(seed, wid, n, layer, ps, H, D, dtype, head_scale=None):
    from streaming_paged_kv_gb300.inputs import frame_qkv
    return [frame_qkv(seed, wid, f, layer, ps, H, D, dtype, head_scale) for f in range(n)]


def _cat(frames, i):
    return torch.cat([fr[i] for fr in frames])


def _prefill_case(kvc, F, ps, H, D, dtype, scale_frames, window, headroom, rows=None, kernel=0,
                  n_layers=1, head_scale=None):
    from oracle import OraclePagedKV, prefill_attention
    from streaming_paged_kv_gb300.inputs import to_bits
    T = ps + 6
    c = kvc.PagedKVCache(n_layers, H, D, ps, dtype, scale_frames, window, headroom, 64,
                         max_query_tokens=F * T)
    if kernel:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, kernel)
    orc = OraclePagedKV(n_layers, ps, H, D, dtype, scale_frames, window, headroom, 64)
    results = []
    for layer in range(n_layers):
        fr = _frames(3, 40 + F, F, layer, ps, H, D, dtype, head_scale)
        q, k, v = (_cat(fr, i).cuda() for i in range(3))
        out = torch.empty_like(q)
        c.prefill(layer, q, k, v, out)
        for f in range(F):
            orc.append_frame(layer, to_bits(fr[f][1]), to_bits(fr[f][2]))
        qb = [to_bits(x[0]) for x in fr]
        want = prefill_attention(qb, [to_bits(x[1]) for x in fr], [to_bits(x[2]) for x in fr], dtype,
                                 rows=rows)
        got = out if rows is None else out[torch.as_tensor(rows, device=out.device)]
        torch.cuda.synchronize()
        results.append(compare(got, want, dtype))
        assert c.stats(layer) == orc.stats(layer)
        assert np.array_equal(to_bits(c.cache_view(layer).cpu()), orc.mirror[layer])
    return c, orc, results


def test_tiny_f32_prefill_then_stream(kvc):
    """Two scale frames prefilled (CUDA-core kernel, fp32), then four streamed
    frames attend over the prefilled cache as usual."""
    from oracle import paged_attention
    from streaming_paged_kv_gb300.inputs import frame_qkv, to_bits
    c, orc, res = _prefill_case(kvc, 2, 16, 2, 32, "f32", 2, 4, 2)
    assert res[0][0] <= TOL["f32"][0], res
    for f in range(2, 6):
        q, k, v = frame_qkv(3, 42, f, 0, 16, 2, 32, "f32")
        c.append_frame(0, k.cuda(), v.cuda())
        c.evict_frames(0)
        orc.append_frame(0, to_bits(k), to_bits(v))
        orc.evict_frames(0, 2, 4)
        c.plan()
        qd = q.cuda()
        out = torch.empty_like(qd)
        c.run(0, qd, out)
        torch.cuda.synchronize()
        mx, rel = compare(out, paged_attention(orc, 0, to_bits(q)), "f32")
        assert mx <= TOL["f32"][0], (f, mx)
    c.close()


@pytest.mark.parametrize("kernel", [1, 2])
def test_s224_prefill_eight_scale_frames_two_layers(kvc, kernel):
    """8 x 262 = 2096 queries over the same 2096 keys, every row compared."""
    c, orc, res = _prefill_case(kvc, 8, 256, 16, 64, "bf16", 8, 64, 16, kernel=kernel, n_layers=2)
    for mx, rel in res:
        assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], res
    c.close()


def test_s518_prefill_full_size_sampled_rows(kvc):
    """The 518x378 Phase-1 shape: 8 x 1005 = 8040 queries over 8040 keys, K
    scaled per head; sampled rows include every frame's first and last rows."""
    from streaming_paged_kv_gb300.inputs import k_head_scale
    T = 1005
    rows = sorted(set(list(range(0, 8 * T, 97)) + [f * T for f in range(8)] + [f * T + T - 1 for f in range(8)]))
    c, orc, res = _prefill_case(kvc, 8, 999, 16, 64, "bf16", 8, 64, 16, rows=rows,
                                head_scale=k_head_scale(0, 3, 16))
    mx, rel = res[0]
    assert mx <= TOL["bf16"][0] and rel <= TOL["bf16"][1], res
    c.close()


def test_prefill_errors_leave_bookkeeping_unchanged(kvc):
    from streaming_paged_kv_gb300.inputs import frame_qkv
    ps, H, D, T = 16, 2, 32, 22
    c = kvc.PagedKVCache(2, H, D, ps, "f32", 2, 4, 2, 16, max_query_tokens=3 * T)
    fr = _frames(1, 9, 4, 0, ps, H, D, "f32")
    q, k, v = (_cat(fr, i).cuda() for i in range(3))
    out = torch.empty_like(q)
    # More queries than max_query_tokens.
    with pytest.raises(kvc.KvcError) as e:
        c.prefill(0, q, k, v, out)
    assert e.value.code == "INVALID_ARG"
    assert c.stats(0)["frame_count"] == 0
    # Block 1 before block 0: no plan yet.
    q3, k3, v3, o3 = q[:3 * T], k[:3 * T], v[:3 * T], out[:3 * T]
    with pytest.raises(kvc.KvcError) as e:
        c.prefill(1, q3, k3, v3, o3)
    assert e.value.code == "NO_PLAN"
    assert c.stats(1)["frame_count"] == 0 and c.deques(1) == c.deques(0)
    # Block 0, then block 1 with the same frames: fine.
    c.prefill(0, q3, k3, v3, o3)
    ref = o3.clone()
    c.prefill(1, q3, k3, v3, o3)
    torch.cuda.synchronize()
    assert torch.equal(ref, o3)
    # A block that already holds frames.
    with pytest.raises(kvc.KvcError) as e:
        c.prefill(0, q3, k3, v3, o3)
    assert e.value.code == "INVALID_ARG"
    assert c.stats(0)["frame_count"] == 3
    # After clean, block 0 can be prefilled again; block 1 with a different
    # frame count no longer matches the plan.
    c.clean()
    c.prefill(0, q3, k3, v3, o3)
    with pytest.raises(kvc.KvcError) as e:
        c.prefill(1, q[:2 * T], k[:2 * T], v[:2 * T], out[:2 * T])
    assert e.value.code == "STALE_PLAN"
    assert c.stats(1)["frame_count"] == 0 and c.stats(1)["free_pages"] == 8
    c.close()
