"""Drive a cache engine through a workload's per-frame schedule.

An engine exposes: append(block, frame), evict(block), set_defer(on),
execute(block), rollback(block), clean(), plan(), attend(block, frame) and
after_frame(frame, kind).  The call order per block follows the streaming
forward pass: append -> evict -> (plan on block 0) -> attend.
"""

from streaming_paged_kv_gb300.inputs import keyframe_decisions
from streaming_paged_kv_gb300.workloads import schedule


def drive(w, engine, seed=0, n_frames=None, blocks=None, attend=True):
    w = w if n_frames is None else w.with_(n_frames=n_frames)
    blocks = range(w.num_layers) if blocks is None else blocks
    decisions = keyframe_decisions(seed, w.wid, w.n_frames) if w.mode == "defer" else None
    for f, kind in schedule(w, decisions):
        if kind == "clean":
            engine.clean()
            continue
        provisional = kind in ("accept", "reject")
        if provisional:
            engine.set_defer(True)
        for i, b in enumerate(blocks):
            engine.append(b, f)
            engine.evict(b)
            if i == 0:
                engine.plan()
            if attend:
                engine.attend(b, f)
        if kind == "accept":
            for b in blocks:
                engine.execute(b)
        elif kind == "reject":
            for b in blocks:
                engine.rollback(b)
        if provisional:
            engine.set_defer(False)
        engine.after_frame(f, kind)
