"""Seeded synthetic inputs: per-frame Q/K/V streams and keyframe decisions.

This module only draws random numbers.  It holds none of the cache's or the
attention's arithmetic and imports nothing else from this package, so that
both the CUDA path and the CPU oracle can be fed from it.

Every tensor comes from its own counter-keyed stream:
``Philox(SeedSequence([seed, workload_id, 1, frame, layer, tensor, part]))``
with ``tensor`` in {q: 0, k: 1, v: 2} and ``part`` 0 for the 6 special rows,
1 for the patch rows.  Values are N(0, 1) float32, optionally multiplied per
head (K only) by a seeded U(0.5, 2) factor, then rounded to the storage dtype
by round-to-nearest-even (``torch.Tensor.to``).  Keeping special and patch rows
in separate streams lets a checker regenerate the special tokens of every frame
without drawing the (much larger) patch tokens.
"""

import numpy as np
import torch

NUM_SPECIAL = 6
_TENSOR_ID = {"q": 0, "k": 1, "v": 2}
TORCH_DTYPE = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _rng(*key):
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(k) for k in key])))


def k_head_scale(seed, workload_id, num_heads):
    """Per-head factor u_h ~ U(0.5, 2) applied to K, fixed for a whole stream."""
    return _rng(seed, workload_id, 2).uniform(0.5, 2.0, size=num_heads).astype(np.float32)


def keyframe_decisions(seed, workload_id, n):
    """Seeded Bernoulli(0.5) accept (True) / reject (False) decisions."""
    return _rng(seed, workload_id, 3).random(n) < 0.5


def _rows(seed, workload_id, frame, layer, name, part, n_rows, num_heads, head_dim, scale):
    x = _rng(seed, workload_id, 1, frame, layer, _TENSOR_ID[name], part).standard_normal(
        (n_rows, num_heads, head_dim), dtype=np.float32)
    if scale is not None and name == "k":
        x *= scale[None, :, None]
    return x


def frame_tensor(seed, workload_id, frame, layer, name, page_size, num_heads, head_dim,
                 dtype="bf16", head_scale=None, part=None):
    """One frame's Q, K or V as a CPU tensor of ``dtype``.

    Shape ``[6 + page_size, H, D]`` (special rows first, then patch rows), or
    only the special rows (``part="special"``) or only the patch rows
    (``part="patch"``).
    """
    pieces = []
    if part in (None, "special"):
        pieces.append(_rows(seed, workload_id, frame, layer, name, 0, NUM_SPECIAL,
                            num_heads, head_dim, head_scale))
    if part in (None, "patch"):
        pieces.append(_rows(seed, workload_id, frame, layer, name, 1, page_size,
                            num_heads, head_dim, head_scale))
    x = np.concatenate(pieces, axis=0) if len(pieces) > 1 else pieces[0]
    return torch.from_numpy(x).to(TORCH_DTYPE[dtype])


def frame_qkv(seed, workload_id, frame, layer, page_size, num_heads, head_dim,
              dtype="bf16", head_scale=None):
    """``(q, k, v)`` CPU tensors ``[6 + page_size, H, D]`` of one frame and layer."""
    return tuple(frame_tensor(seed, workload_id, frame, layer, n, page_size, num_heads,
                              head_dim, dtype, head_scale) for n in ("q", "k", "v"))


def to_bits(t):
    """Raw element bits of a CPU tensor as a NumPy array (uint16 / uint32)."""
    t = t.contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    raise TypeError(t.dtype)
