"""Per-frame attention over the visible cache, in float64 on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The paged kernel computes, for every query row t and head h,

    O[t, h, :] = sum_j softmax_j( Q[t, h, :] . K[j, h, :] * sm_scale ) V[j, h, :]

over the visible tokens j, non-causally (the frame also attends to itself),
with as many KV heads as query heads and no positional encoding inside the
kernel ([KVC] "Kernel-Level Execution Flow": the plan passes causal=False,
pos_encoding_mode="NONE", num_qo_heads == num_kv_heads).  That is exactly
dense scaled-dot-product attention over the K/V gathered from the visible
pages -- what the manager itself does for fp32 inputs ([PERF] "Force-FP32
Fallback Avoidance": gather K/V into dense tensors and run
scaled_dot_product_attention).  The default scale is 1/sqrt(head_dim).
"""

import numpy as np


def bits_to_f64(bits, dtype):
    """Exact float64 values of stored elements given as raw bits."""
    bits = np.asarray(bits)
    if dtype == "bf16":
        # A bf16 value is the upper half of the float32 with the same sign,
        # exponent and leading mantissa bits.
        with np.errstate(invalid="ignore"):
            return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "f32":
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def dense_attention(q, k, v, sm_scale=None):
    """Softmax attention in float64.

    q: [Nq, H, D], k and v: [Nkv, H, D] (float64 values).  Returns [Nq, H, D].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, h, d = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    out = np.empty((nq, h, v.shape[2]), dtype=np.float64)
    for head in range(h):
        s = (q[:, head, :] @ k[:, head, :].T) * sm_scale          # [Nq, Nkv]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, head, :] = p @ v[:, head, :]
    return out


def paged_attention(cache, block, q_bits, sm_scale=None, rows=None, plan_block=0):
    """Attention of one frame's queries (raw bits ``[Nq, H, D]``) over block
    ``block``'s visible pages, as planned on ``plan_block``.

    ``rows`` optionally selects query rows (for sampled checks on big inputs).
    """
    k_bits, v_bits = cache.gather_visible(block, plan_block)
    if k_bits.shape[0] == 0:
        raise ValueError("no visible tokens")
    q = bits_to_f64(q_bits, cache.dtype)
    if rows is not None:
        q = q[np.asarray(rows)]
    return dense_attention(q, bits_to_f64(k_bits, cache.dtype),
                           bits_to_f64(v_bits, cache.dtype), sm_scale)


def prefill_attention(q_frames, k_frames, v_frames, dtype, sm_scale=None, rows=None):
    """Phase 1, batch mode ([KVC] "FlashInferAttention Layer Implementation";
    [SLOTS] "scale frames永不驱逐"): the first frames go through standard dense
    attention as one block, bidirectionally -- every query of every frame over
    every key of every frame.  Inputs are the frames' raw bits, each
    ``[T, H, D]``; the result is ``[F*T, H, D]`` float64, frame after frame
    (only the query rows ``rows`` of that, if given).
    """
    q = np.concatenate([bits_to_f64(x, dtype) for x in q_frames])
    if rows is not None:
        q = q[np.asarray(rows)]
    k = np.concatenate([bits_to_f64(x, dtype) for x in k_frames])
    v = np.concatenate([bits_to_f64(x, dtype) for x in v_frames])
    return dense_attention(q, k, v, sm_scale)

