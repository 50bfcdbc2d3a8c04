"""The streaming workloads, their shapes and their per-frame call schedules.

A workload fixes the cache geometry and how a synthetic video stream drives
the cache API frame by frame.  The schedules restate the usage patterns of the
pages:

* ``stream``   -- every frame is a keyframe: per block ``append_frame``,
  ``evict_frames``, then attention ([KVC] "Streaming Forward Pass").
* ``defer``    -- after the scale frames, every frame is appended with eviction
  deferred, attends, and is then accepted (``execute_deferred_eviction``) or
  rolled back (``rollback_last_frame``) on a seeded coin flip
  ([SLOTS] "光流关键帧与回滚机制"; [PERF] "Deferred Eviction for Keyframe Decisions").
* ``windowed`` -- the cache is reset at every window start; a window has
  ``window_slots`` slots (``scale_frames`` scale + the rest keyframes) and one
  keyframe every ``keyframe_interval`` frames, so it spans
  ``scale + (slots - scale) * interval`` frames; non-keyframes attend over
  cache + themselves without being kept ([SLOTS] "窗口模式", "keyframes滑动窗口").

Pages cited by tag: [KVC] "How LingBot-Map Implements the KV Cache Mechanism
for Streaming Inference with FlashInfer Integration"; [PERF] "How to Improve
Streaming Inference Performance with FlashInfer KV Cache Backend"; [SLOTS]
"LingBot-Map KV缓存机制深度揭秘：scale frames与keyframes如何占用slot".
"""

from dataclasses import dataclass, replace

NUM_SPECIAL = 6


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    num_layers: int
    num_heads: int
    head_dim: int
    dtype: str
    page_size: int
    scale_frames: int
    sliding_window: int
    headroom: int
    max_total_frames: int
    n_frames: int
    mode: str = "stream"
    keyframe_interval: int = 1
    window_slots: int = 0
    k_head_scale: bool = False

    @property
    def tokens_per_frame(self):
        return NUM_SPECIAL + self.page_size

    @property
    def num_patch_pages(self):
        return self.scale_frames + self.sliding_window + self.headroom

    @property
    def window_frames(self):
        """Frames covered by one window in ``windowed`` mode."""
        return self.scale_frames + (self.window_slots - self.scale_frames) * self.keyframe_interval

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    # 1 layer, H=2, D=32, fp32, 16 patch tokens + 6 specials per frame (2 frames per special page).
    "tiny": Workload(1, "tiny", 1, 2, 32, "f32", 16, 2, 4, 2, 16, 12),
    # 224x224 frames: 16x16 = 256 patches.
    "s224": Workload(2, "s224", 24, 16, 64, "bf16", 256, 8, 64, 16, 2048, 200),
    # Same shapes, 12 layers, provisional frames accepted or rolled back by a coin flip.
    "defer": Workload(3, "defer", 12, 16, 64, "bf16", 256, 8, 64, 16, 2048, 400, mode="defer"),
    # 518x378 frames, patch 14: 37x27 = 999 patches, exact (non power of two) page size.
    "s518": Workload(4, "s518", 24, 16, 64, "bf16", 999, 8, 64, 16, 2048, 2048, k_head_scale=True),
    # 518x378 windowed: 128 slots = 8 scale + 120 keyframe slots, keyframe every 13 frames.
    "win518": Workload(5, "win518", 24, 16, 64, "bf16", 999, 8, 120, 16, 2048, 25000,
                       mode="windowed", keyframe_interval=13, window_slots=128),
    # The camera head's own cache beside the trunk's ([SLOTS] "特殊 token 流", last
    # sentence: the camera head keeps an isomorphic, independent KV cache with the
    # same scale / window parameters).  The pages give no shapes; reading: the same
    # per-frame token layout and width as the 518x378 trunk, 4 layers of its own,
    # K scaled per head like the trunk's.  Driven frame by frame with "s518".
    "cam518": Workload(6, "cam518", 4, 16, 64, "bf16", 999, 8, 64, 16, 2048, 2048, k_head_scale=True),
}

# Streams made of two caches driven in lockstep: (trunk, camera head).
PAIRED = {"camcache": ("s518", "cam518")}


def schedule(w, decisions=None):
    """Per-frame events ``(frame, kind)`` of workload ``w`` in stream order.

    kind is one of
      ``"clean"``  -- reset the cache (no frame is processed by this event),
      ``"key"``    -- append + evict on every block, plan on block 0, attend,
      ``"accept"`` -- provisional frame (deferred eviction), then execute,
      ``"reject"`` -- provisional frame (deferred eviction), then rollback.
    ``decisions[i]`` is the accept/reject coin of frame i in ``defer`` mode.
    """
    for f in range(w.n_frames):
        if w.mode == "stream":
            yield f, "key"
        elif w.mode == "defer":
            if f < w.scale_frames:
                yield f, "key"
            else:
                yield f, ("accept" if decisions[f] else "reject")
        elif w.mode == "windowed":
            j = f % w.window_frames
            if j == 0:
                yield f, "clean"
            if j < w.scale_frames or (j - w.scale_frames) % w.keyframe_interval == 0:
                yield f, "key"
            else:
                yield f, "reject"
        else:
            raise ValueError(w.mode)
