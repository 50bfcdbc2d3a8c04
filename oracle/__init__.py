"""CPU oracle for the two-stream paged KV cache and its per-frame attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) use it.
It shares no code with the CUDA path (``streaming_paged_kv_gb300``): no common
helpers, tables or constants, and it imports nothing from there.

What it computes, in plain slow code:

* ``oracle.paged_kv.OraclePagedKV`` -- the page bookkeeping of every
  transformer block (scale / live-window / free deques of patch page IDs, the
  append-only special-token stream, deferred eviction, rollback, window reset)
  and a byte-exact NumPy mirror of the cache tensor
  ``[max_num_pages, 2, page_size, H, D]``.
* ``oracle.attention`` -- softmax attention of a frame's queries over the
  visible keys/values, gathered densely in page order and computed in float64;
  and Phase 1 (batch mode): dense bidirectional attention of the first frames
  as one block, from the frames' own Q/K/V.

Pages cited (by tag, then section):

* [KVC]   "How LingBot-Map Implements the KV Cache Mechanism for Streaming
          Inference with FlashInfer Integration"
* [PERF]  "How to Improve Streaming Inference Performance with FlashInfer KV
          Cache Backend"
* [SLOTS] "LingBot-Map KV缓存机制深度揭秘：scale frames与keyframes如何占用slot"
          (mhpq.cn; its sections are the inline headings quoted in Chinese)

Readings taken where the pages are silent:

1. Special packing is frame-aligned: frame s of the stream owns slots
   ``[6*(s % fpp), 6*(s % fpp) + 6)`` of special page ``P + s // fpp`` with
   ``fpp = page_size // 6``; a non-last special page holds ``6*fpp`` valid
   tokens, the last one ``last_page_len``.  **Parity unpinned by the pages**
   for the page table itself (the attention result does not depend on it).
2. Free-list order: ``[0, 1, ..., P-1]`` at construction and after a reset;
   allocation pops the left end, eviction pushes the right end, rollback pushes
   the left end.  **Parity unpinned by the pages** (pinned by self-consistency:
   rollback restores the free list exactly).
3. Append -> evict -> attend, so a committed keyframe sees
   ``scale_frames + sliding_window`` patch pages, itself included.
4. Any eviction that moves a page commits (clears the undo stack);
   ``execute_deferred_eviction`` always commits.
"""

from .paged_kv import OraclePagedKV, OracleError  # noqa: F401
from .attention import dense_attention, paged_attention, prefill_attention  # noqa: F401
