#!/usr/bin/env python3
"""Streamed frames/s of the 24-layer 518x378 exact-page paged-attention stream.

A step is one streamed frame through every block: per block append_frame,
evict_frames, (plan on block 0) and the paged attention run, all through the
C ABI of libkvc.so.  The stream is the 518x378 workload (page_size 999, H=16,
D=64, bf16, 8 scale / 64 window / 16 headroom pages, 2048 frames).  The timed
steps are the LAST K frames of that 2048-frame stream: the frames before them
are streamed untimed (append + evict only, then W full warm-up frames), so the
number always describes the same part of the stream whatever K is; the
default K covers the whole stream after the warm-up.

Inputs are synthetic: a pool of seeded N(0,1) bf16 Q/K/V frames per layer,
resident in HBM before the timed region (K scaled per head by a seeded
U(0.5, 2) factor); frame f of layer b uses pool entry (f + b) mod pool.  Every
layer's visible K/V (~340 MB at full context) is larger than L2, so no flush is
needed between steps.

The attention launches' duration (for the roofline) comes from CUDA events
that the library records on the launching stream around one attention launch
per step (the middle layer's; every layer of a step launches the same shape),
so that the measurement adds two events per step instead of two per layer.

Output: one JSON line (see the keys below).  ``--impl reference`` times the CPU
oracle instead, on a bounded sample of the same workload.
"""

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "streamed frames/s (24-layer paged attn, 518x378); attn TFLOP/s vs GB300 roofline"
STREAM_METRIC = "streamed frames/s ({layers}-layer paged attn, {label}); attention vs GB300 roofline"
UNIT = "frames/s"
LABELS = {"s518": "518x378 exact-page stream", "s224": "224x224 stream",
          "defer": "224x224 keyframe + deferred-eviction stream", "win518": "518x378 windowed stream",
          "tiny": "tiny fp32 stream"}


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="timed frames (default: rest of the stream)")
    p.add_argument("--warmup", type=int, default=16)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="s518",
                   help="s518 (default, the streamed metric), s224, defer, phase1, batch224, win518 or camcache")
    p.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tcgen05")
    p.add_argument("--splits", type=int, default=0, help="tuning: force the KV split count (0 = the library's choice)")
    p.add_argument("--qtiles", type=int, default=0,
                   help="tuning: 128-row query tiles per CTA of the tensor-core kernel (0 = the library's choice)")
    p.add_argument("--pdl", type=int, default=1,
                   help="tuning: 1 programmatic dependent launch between the library's kernels (default), 0 off")
    p.add_argument("--pool", type=int, default=4, help="distinct input frames per layer")
    p.add_argument("--batch", type=int, default=8, help="streams of --workload batch224")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the compact lines of the other workloads after the default measurement")
    p.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work")
    p.add_argument("--layers", type=int, default=None,
                   help="profiling size only: override the number of layers")
    p.add_argument("--frames", type=int, default=None,
                   help="profiling size only: override the stream length")
    return p.parse_args()


_PEAKS = None


def peaks():
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rates
    of this GPU model (MEASURED_PEAKS.json), else one earlier GB300
    measurement, with a warning on stderr."""
    global _PEAKS
    if _PEAKS is not None:
        return _PEAKS
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        _PEAKS = {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                  "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        sys.stderr.write("bench.py: MEASURED_PEAKS.json not found or unreadable; the roofline fractions "
                         "use fallback peaks (6800 GB/s, 1900 / 1700 TFLOP/s bf16 burst / sustained)\n")
        _PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}
    return _PEAKS


def roof_bound(flops, bytes_alg):
    """'tensor' when the arithmetic intensity is at or above the ridge point of
    the burst bf16 peak over the copy bandwidth, else 'hbm'."""
    pk = peaks()
    return "tensor" if flops / max(bytes_alg, 1.0) >= pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"] else "hbm"


def attn_roofline(bound, flops, bytes_alg, attn_ms, attn_launches, step_ms, kernel, traffic=None):
    """Roofline of the attention launches of a timed region.

    achieved = algorithmic work (flops = 4 n_q N_kv H D, or bytes = visible K/V
    once + Q in + O out) / the launches' CUDA-event time; `frac` divides by
    the burst bf16 peak (a tensor-bound launch is a fraction of a second) or
    the copy bandwidth.  `frac_sustained` is the same against the sustained
    bf16 peak, and `step_frac` is the roofline time of all timed launches
    (max of flops / peak and bytes / bandwidth) over the whole timed region,
    so that everything outside the attention launches counts against it."""
    pk = peaks()
    n = max(attn_launches, 1)
    secs = attn_ms / 1e3
    tflops = flops / secs / 1e12 if attn_ms > 0 else None
    gbs = bytes_alg / secs / 1e9 if attn_ms > 0 else None
    roof_s = max(flops / (pk["bf16_tflops"] * 1e12), bytes_alg / (pk["hbm_gbs"] * 1e9))
    r = {"bound": bound}
    if bound == "tensor":
        r.update({"achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                  "frac": tflops / pk["bf16_tflops"] if tflops else None})
    else:
        r.update({"achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                  "frac": gbs / pk["hbm_gbs"] if gbs else None})
    r["traffic"] = traffic
    r["peak_kind"] = (f"bf16 dense burst ({pk['source']})" if bound == "tensor"
                      else f"HBM copy bandwidth ({pk['source']})")
    r["frac_sustained"] = tflops / pk["bf16_tflops_sustained"] if (tflops and bound == "tensor") else None
    r["peak_sustained"] = pk["bf16_tflops_sustained"] if bound == "tensor" else None
    r["step_frac"] = roof_s / (step_ms / 1e3) if step_ms > 0 else None
    r["attn_tflops"] = tflops
    r["attn_gbs"] = gbs
    r["kernel"] = kernel
    r["flops_per_launch"] = flops / n
    r["alg_bytes_per_launch"] = bytes_alg / n
    r["launch_ms"] = attn_ms / n
    r["outside_attn_ms_per_step"] = None
    return r


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        for line in open(self.file.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------- GPU stream
class Stream:
    """One device stream of the workload through the library."""

    def __init__(self, kvc, w, pool, seed, kernel, dev, splits=0, qtiles=0, pdl=1):
        import torch
        from streaming_paged_kv_gb300.inputs import k_head_scale
        self.torch, self.kvc, self.w = torch, kvc, w
        self.c = kvc.PagedKVCache(w.num_layers, w.num_heads, w.head_dim, w.page_size, w.dtype,
                                  w.scale_frames, w.sliding_window, w.headroom, w.max_total_frames,
                                  device=dev)
        if kernel:
            self.c.set_option(kvc.KVC_OPT_ATTN_KERNEL, kernel)
        if splits:
            self.c.set_option(kvc.KVC_OPT_NUM_SPLITS, splits)
        if qtiles:
            self.c.set_option(kvc.KVC_OPT_QUERY_TILES, qtiles)
        if not pdl:
            self.c.set_option(kvc.KVC_OPT_PDL, 0)
        T, H, D = w.tokens_per_frame, w.num_heads, w.head_dim
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        scale = torch.from_numpy(k_head_scale(seed, w.wid, H)).to(dev) if w.k_head_scale else None
        self.pool = []
        for i in range(pool):
            per_layer = []
            for b in range(w.num_layers):
                q = torch.randn(T, H, D, generator=g, device=dev).to(torch.bfloat16)
                k = torch.randn(T, H, D, generator=g, device=dev)
                if scale is not None:
                    k = k * scale[None, :, None]
                k = k.to(torch.bfloat16)
                v = torch.randn(T, H, D, generator=g, device=dev).to(torch.bfloat16)
                per_layer.append((q, k, v))
            self.pool.append(per_layer)
        self.out = [torch.empty(T, H, D, dtype=torch.bfloat16, device=dev) for _ in range(w.num_layers)]
        self.frame = 0

    def inputs(self, f, b):
        return self.pool[(f + b) % len(self.pool)][b]

    def fast_forward(self, n):
        """Append + evict only (no attention) for n frames."""
        c = self.c
        for _ in range(n):
            for b in range(self.w.num_layers):
                _, k, v = self.inputs(self.frame, b)
                c.append_frame(b, k, v)
                c.evict_frames(b)
            self.frame += 1

    def step(self):
        """One streamed frame: append, evict, plan (block 0), attention per block."""
        c = self.c
        for b in range(self.w.num_layers):
            q, k, v = self.inputs(self.frame, b)
            c.append_frame(b, k, v)
            c.evict_frames(b)
            if b == 0:
                c.plan()
            c.run(b, q, self.out[b])
        self.frame += 1

    def visible_tokens(self):
        s = self.c.stats(0)
        return self.w.page_size * (s["scale_pages"] + s["live_pages"]) + s["special_tokens"]


def kernel_code_hash(path):
    """sha256 of a CUDA source with its comments and blank lines removed, so
    that only a change of code (not of commentary) marks counters as stale."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


# The committed ncu summary whose DRAM counters stand for each workload's
# attention launch (same kernel and launch shape, one layer at a late frame).
TRAFFIC_PROFILES = {"s518": "attn_tc_s518_l1f200_full.md", "s224": "attn_tc_s224_l1f200_full.md"}


def profiled_traffic(alg_bytes_per_launch, workload_name="s518"):
    """DRAM bytes per attention launch from the workload's committed ncu
    summary, scaled to this run's average launch by algorithmic bytes -- or None
    when there is no summary for the workload or the kernel code differs from
    the one the counters were taken on."""
    import re
    if workload_name not in TRAFFIC_PROFILES:
        return None
    prof = os.path.join(ROOT, "profiles", TRAFFIC_PROFILES[workload_name])
    src = os.path.join(ROOT, "streaming_paged_kv_gb300", "csrc", "kvc_attn_tc.cu")
    try:
        text = open(prof, encoding="utf-8").read()
        sha = re.search(r"^kernel_code_sha256: ([0-9a-f]+)$", text, re.M).group(1)
        dram = float(re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M).group(1))
        alg = float(re.search(r"^alg_bytes_per_launch: (\d+)$", text, re.M).group(1))
        if kernel_code_hash(src) != sha:
            return None
        return dram * alg_bytes_per_launch / alg
    except Exception:
        return None


def workload(args):
    from streaming_paged_kv_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(num_layers=args.layers)
    if args.frames:
        w = w.with_(n_frames=args.frames)
    return w


def aggregate(ms, frames, world, device="cpu"):
    """Whole-job numbers of independent replicas: the slowest rank's time and
    the frames of all ranks (max and sum over ranks; identity for one rank)."""
    if world <= 1:
        return ms, frames
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    f = torch.tensor([float(frames)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), int(f.item())


def run_ours(args, rank, world):
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    w = workload(args)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else w.n_frames - args.warmup
    W = args.warmup
    K = max(1, min(K, w.n_frames))
    W = max(0, min(W, w.n_frames - K))
    st = Stream(kvc, w, args.pool, args.seed + rank, args.kernel, dev, args.splits, args.qtiles, args.pdl)
    st.fast_forward(w.n_frames - K - W)
    for _ in range(W):
        st.step()
    torch.cuda.synchronize()
    # Algorithmic work of the timed frames (attention only): replay the same
    # frames on a bookkeeping-only handle to get each frame's visible tokens.
    n_q, H, D = w.tokens_per_frame, w.num_heads, w.head_dim
    book = kvc.PagedKVCache(1, H, D, w.page_size, w.dtype, w.scale_frames, w.sliding_window,
                            w.headroom, w.max_total_frames, device=None)
    flops = bytes_alg = 0.0
    for f in range(w.n_frames):
        book.append_frame(0)
        book.evict_frames(0)
        if f >= w.n_frames - K:
            s = book.stats(0)
            nkv = w.page_size * (s["scale_pages"] + s["live_pages"]) + s["special_tokens"]
            flops += w.num_layers * 4.0 * n_q * nkv * H * D
            bytes_alg += w.num_layers * (2.0 * nkv * H * D * 2 + 2.0 * n_q * H * D * 2)
    book.close()
    kvc.kvc_get_counters(st.c.h, reset=True)
    st.c.set_option(kvc.KVC_OPT_TIMING, w.num_layers)   # one timed launch per frame
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    ev0.record()
    for _ in range(K):
        st.step()
    ev1.record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    ms, total_frames = aggregate(ev0.elapsed_time(ev1), K, world, dev)
    launches, attn_launches, attn_ms = kvc.kvc_get_counters(st.c.h, reset=True)
    st.c.set_option(kvc.KVC_OPT_TIMING, 0)
    status = kvc.kvc_device_status(st.c.h, st.c._stream())
    if status != 0:
        raise RuntimeError(f"device status {status}")
    value = total_frames / (ms / 1e3)
    bound = roof_bound(flops, bytes_alg)
    roofline = attn_roofline(bound, flops, bytes_alg, attn_ms, attn_launches, ms,
                             "paged attention (kvc_run attention launch)",
                             profiled_traffic(bytes_alg / max(attn_launches, 1), w.name))
    roofline["outside_attn_ms_per_step"] = (ms - attn_ms) / K
    roofline["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(st.c.h)))
    res = {
        "metric": METRIC if w.name == "s518" else STREAM_METRIC.format(label=LABELS.get(w.name, w.name),
                                                                        layers=w.num_layers),
        "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: {LABELS.get(w.name, w.name)}, {w.num_layers} layers, "
                               f"H={H}, D={D}, page_size={w.page_size}, {w.n_frames} frames; timed = "
                               f"last {K} frames",
                   "frames_timed": [w.n_frames - K, w.n_frames - 1],
                   "l2": ("no flush: every layer's visible K/V (>300 MB at full context) exceeds L2"
                          if w.name == "s518" else
                          "no flush: the 24 layers' visible K/V together exceed L2, and each layer is "
                          "read once per frame"),
                   "parallelism": f"replicas x{world} (independent streams, no collective)",
                   "wall_s": t_wall},
        "roofline": roofline,
        "attn_tflops": roofline["attn_tflops"],
        "gpu_launches": launches,
        "clocks": clk,
    }
    del st
    torch.cuda.empty_cache()
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, kvc, w, dev, rank, world, K, W)
    return res


PAIRED_METRIC = ("streamed frames/s (518x378: 24-layer trunk + 4-layer camera-head paged attn, two caches); "
                 "attn TFLOP/s vs GB300 roofline")


def run_paired(args, rank, world):
    """The trunk's cache and the camera head's own cache in one stream: per
    frame every trunk layer appends, evicts, plans (layer 0) and attends, then
    every camera-head layer does the same on its cache.  Timed: the last K
    frames of the 2048-frame stream, as for the trunk alone."""
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    from streaming_paged_kv_gb300.workloads import PAIRED, WORKLOADS
    tw, hw = (WORKLOADS[n] for n in PAIRED["camcache"])
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else 20
    W = max(args.warmup, 3)
    streams = [Stream(kvc, w, args.pool, args.seed + rank + 17 * i, args.kernel, dev, args.splits, args.qtiles)
               for i, w in enumerate((tw, hw))]
    for st in streams:
        st.fast_forward(tw.n_frames - K - W)
    for _ in range(W):
        for st in streams:
            st.step()
    torch.cuda.synchronize()
    n_q, H, D = tw.tokens_per_frame, tw.num_heads, tw.head_dim
    book = kvc.PagedKVCache(1, H, D, tw.page_size, tw.dtype, tw.scale_frames, tw.sliding_window,
                            tw.headroom, tw.max_total_frames, device=None)
    flops = bytes_alg = 0.0
    layers = tw.num_layers + hw.num_layers
    for f in range(tw.n_frames):
        book.append_frame(0)
        book.evict_frames(0)
        if f >= tw.n_frames - K:
            s_ = book.stats(0)
            nkv = tw.page_size * (s_["scale_pages"] + s_["live_pages"]) + s_["special_tokens"]
            flops += layers * 4.0 * n_q * nkv * H * D
            bytes_alg += layers * (2.0 * nkv * H * D * 2 + 2.0 * n_q * H * D * 2)
    book.close()
    for st in streams:
        kvc.kvc_get_counters(st.c.h, reset=True)
        st.c.set_option(kvc.KVC_OPT_TIMING, st.w.num_layers)   # one timed launch per frame
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(K):
        for st in streams:
            st.step()
    ev1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms, total_frames = aggregate(ev0.elapsed_time(ev1), K, world, dev)
    launches = attn_launches = 0
    attn_ms = 0.0
    for st in streams:
        l_, a_, m_ = kvc.kvc_get_counters(st.c.h, reset=True)
        launches, attn_launches, attn_ms = launches + l_, attn_launches + a_, attn_ms + m_
        st.c.set_option(kvc.KVC_OPT_TIMING, 0)
        if kvc.kvc_device_status(st.c.h, st.c._stream()) != 0:
            raise RuntimeError("device status")
    roof = attn_roofline(roof_bound(flops, bytes_alg), flops, bytes_alg, attn_ms, attn_launches, ms,
                         "paged attention (kvc_run attention launch, both caches)")
    roof["outside_attn_ms_per_step"] = (ms - attn_ms) / K
    roof["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(streams[0].c.h)))
    del streams
    torch.cuda.empty_cache()
    return {
        "metric": PAIRED_METRIC, "value": total_frames / (ms / 1e3), "unit": "frames/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"camcache: {tw.name} trunk ({tw.num_layers} layers) + {hw.name} camera head "
                               f"({hw.num_layers} layers), H={H}, D={D}, page_size={tw.page_size}; timed = last "
                               f"{K} frames of {tw.n_frames}",
                   "l2": "no flush: every layer's visible K/V exceeds L2",
                   "parallelism": f"replicas x{world} (independent streams, no collective)"},
        "roofline": roof, "attn_tflops": roof["attn_tflops"], "gpu_launches": launches, "clocks": clk,
    }


WINDOW_METRIC = ("windowed-stream frames/s (518x378, 24-layer paged attn, 128-slot window reset per window, "
                 "keyframe interval 13); attn TFLOP/s vs GB300 roofline")


def run_windowed(args, rank, world):
    """The windowed long stream: a window of 8 scale + 120 keyframe slots,
    reset with clean at its start; one frame in 13 after the scale frames is
    a keyframe (append, evict, plan, attend), the others attend over the cache
    plus themselves and are rolled back.  Timed: one whole window from a clean
    start, after warm-up frames of a first window; frames/s and the device
    time of every frame (p50 / p99)."""
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    from streaming_paged_kv_gb300.workloads import WORKLOADS, schedule
    w = WORKLOADS["win518"]
    if args.layers:
        w = w.with_(num_layers=args.layers)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K = min(args.steps or w.window_frames, w.window_frames)
    W = max(args.warmup, 3)
    st = Stream(kvc, w, args.pool, args.seed + rank, args.kernel, dev, args.splits, args.qtiles)
    c, L = st.c, w.num_layers
    book = kvc.PagedKVCache(1, w.num_heads, w.head_dim, w.page_size, w.dtype, w.scale_frames,
                            w.sliding_window, w.headroom, w.max_total_frames, device=None)

    def frame(f, kind, count=None):
        if kind == "clean":
            c.clean()
            book.clean()
            return
        prov = kind == "reject"
        if prov:
            c.set_defer_eviction(True)
            book.set_defer_eviction(True)
        book.append_frame(0)
        book.evict_frames(0)
        if count is not None:
            s_ = book.stats(0)
            count.append(w.page_size * (s_["scale_pages"] + s_["live_pages"]) + s_["special_tokens"])
        for b in range(L):
            q, k, v = st.inputs(f, b)
            c.append_frame(b, k, v)
            c.evict_frames(b)
            if b == 0:
                c.plan()
            c.run(b, q, st.out[b])
        if prov:
            for b in range(L):
                c.rollback_last_frame(b)
            book.rollback_last_frame(0)
            c.set_defer_eviction(False)
            book.set_defer_eviction(False)

    events = schedule(w)
    done = 0
    for f, kind in events:                      # warm-up: the first frames of a window
        frame(f, kind)
        if kind != "clean":
            done += 1
            if done == W:
                break
    torch.cuda.synchronize()
    timed = [(f, kind) for f, kind in schedule(w.with_(n_frames=w.window_frames))][:K + 1]
    kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, L)   # one timed launch per frame
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    nkv = []
    marks = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for f, kind in timed:
        if kind != "clean":
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            marks.append(e)
        frame(f, kind, nkv)
    ev1.record()
    marks.append(ev1)
    torch.cuda.synchronize()
    clk = clocks.stop()
    n_frames = len(nkv)
    ms, total_frames = aggregate(ev0.elapsed_time(ev1), n_frames, world, dev)
    launches, attn_launches, attn_ms = kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, 0)
    if kvc.kvc_device_status(c.h, c._stream()) != 0:
        raise RuntimeError("device status")
    per = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(n_frames))
    T, H, D = w.tokens_per_frame, w.num_heads, w.head_dim
    flops = sum(L * 4.0 * T * n * H * D for n in nkv)
    bytes_alg = sum(L * (2.0 * n * H * D * 2 + 2.0 * T * H * D * 2) for n in nkv)
    roof = attn_roofline(roof_bound(flops, bytes_alg), flops, bytes_alg, attn_ms, attn_launches, ms,
                         "paged attention (kvc_run attention launch)")
    roof["outside_attn_ms_per_step"] = (ms - attn_ms) / max(n_frames, 1)
    roof["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(c.h)))
    achieved = roof["attn_tflops"]
    book.close()
    del st
    torch.cuda.empty_cache()
    return {
        "metric": WINDOW_METRIC, "value": total_frames / (ms / 1e3), "unit": "frames/s", "n_gpus": world,
        "steps": n_frames, "warmup": W, "ms_per_step": ms / n_frames, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"win518: 518x378 windowed stream, {L} layers, H={H}, D={D}, page_size={w.page_size}, "
                               f"window {w.window_slots} slots ({w.window_frames} frames, keyframe interval "
                               f"{w.keyframe_interval}); timed = one window from its clean start",
                   "l2": "no flush: every layer's visible K/V exceeds L2 once the window fills",
                   "parallelism": f"replicas x{world} (independent streams, no collective)"},
        "frame_ms": {"p50": per[len(per) // 2], "p99": per[min(len(per) - 1, int(len(per) * 0.99))],
                     "max": per[-1]},
        "roofline": roof,
        "attn_tflops": achieved,
        "gpu_launches": launches,
        "clocks": clk,
    }


DEFER_METRIC = ("keyframe + deferred-eviction stream frames/s (12-layer paged attn, 224x224; each frame after the "
                "scale frames provisional, then accepted or rolled back); attention vs GB300 roofline")


def run_defer(args, rank, world):
    """The keyframe + deferred-eviction stream: after the scale frames every
    frame is appended with eviction deferred, planned and attended on every
    layer, then accepted (execute_deferred_eviction) or rolled back by a
    seeded coin.  The frames before the timed ones run untimed with the same
    decisions, so that the timed frames see the stream's own cache state."""
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    from streaming_paged_kv_gb300.inputs import keyframe_decisions
    from streaming_paged_kv_gb300.workloads import WORKLOADS, schedule
    w = WORKLOADS["defer"]
    if args.layers:
        w = w.with_(num_layers=args.layers)
    if args.frames:
        w = w.with_(n_frames=args.frames)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    events = list(schedule(w, keyframe_decisions(args.seed + rank, w.wid, w.n_frames)))
    K = max(1, min(args.steps or 60, len(events) - max(args.warmup, 3)))
    st = Stream(kvc, w, args.pool, args.seed + rank, args.kernel, dev, args.splits, args.qtiles)
    c, L = st.c, w.num_layers
    book = kvc.PagedKVCache(1, w.num_heads, w.head_dim, w.page_size, w.dtype, w.scale_frames,
                            w.sliding_window, w.headroom, w.max_total_frames, device=None)

    def frame(f, kind, count=None):
        prov = kind in ("accept", "reject")
        if prov:
            c.set_defer_eviction(True)
            book.set_defer_eviction(True)
        book.append_frame(0)
        book.evict_frames(0)
        if count is not None:
            s_ = book.stats(0)
            count.append(w.page_size * (s_["scale_pages"] + s_["live_pages"]) + s_["special_tokens"])
        for b in range(L):
            q, k, v = st.inputs(f, b)
            c.append_frame(b, k, v)
            c.evict_frames(b)
            if b == 0:
                c.plan()
            c.run(b, q, st.out[b])
        if kind == "accept":
            for b in range(L):
                c.execute_deferred_eviction(b)
            book.execute_deferred_eviction(0)
        elif kind == "reject":
            for b in range(L):
                c.rollback_last_frame(b)
            book.rollback_last_frame(0)
        if prov:
            c.set_defer_eviction(False)
            book.set_defer_eviction(False)

    for f, kind in events[:len(events) - K]:     # untimed, the warm-up frames included
        frame(f, kind)
    torch.cuda.synchronize()
    kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, L)   # one timed launch per frame
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    nkv = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for f, kind in events[len(events) - K:]:
        frame(f, kind, nkv)
    ev1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms, total_frames = aggregate(ev0.elapsed_time(ev1), K, world, dev)
    launches, attn_launches, attn_ms = kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, 0)
    if kvc.kvc_device_status(c.h, c._stream()) != 0:
        raise RuntimeError("device status")
    T, H, D = w.tokens_per_frame, w.num_heads, w.head_dim
    flops = sum(L * 4.0 * T * n * H * D for n in nkv)
    bytes_alg = sum(L * (2.0 * n * H * D * 2 + 2.0 * T * H * D * 2) for n in nkv)
    roof = attn_roofline(roof_bound(flops, bytes_alg), flops, bytes_alg, attn_ms, attn_launches, ms,
                         "paged attention (kvc_run attention launch)")
    roof["outside_attn_ms_per_step"] = (ms - attn_ms) / K
    roof["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(c.h)))
    kinds = [kind for _, kind in events[len(events) - K:]]
    book.close()
    del st
    torch.cuda.empty_cache()
    return {
        "metric": DEFER_METRIC, "value": total_frames / (ms / 1e3), "unit": "frames/s", "n_gpus": world,
        "steps": K, "warmup": len(events) - K, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"defer: 224x224 keyframe + deferred-eviction stream, {L} layers, H={H}, D={D}, "
                               f"page_size={w.page_size}, {w.n_frames} frames; timed = the last {K} frames "
                               f"({kinds.count('accept')} accepted, {kinds.count('reject')} rolled back)",
                   "l2": "no flush: a frame reads the visible K/V of 12 layers (about 1 GB) between two launches of a layer, above L2",
                   "parallelism": f"replicas x{world} (independent streams, no collective)"},
        "roofline": roof,
        "attn_tflops": roof["attn_tflops"],
        "gpu_launches": launches,
        "clocks": clk,
    }


PHASE1_METRIC = ("Phase-1 batch prefill frames/s (8 scale frames x 1005 tokens, dense bidirectional, "
                 "24-layer paged attn, 518x378); attn TFLOP/s vs GB300 roofline")


def run_phase1(args, rank, world):
    """Phase 1 (batch mode): every layer's first 8 frames attend to each other
    densely (8 x 1005 = 8040 queries over the same 8040 keys) and are appended
    (kvc_prefill).  One step = kvc_clean + the prefill of every layer."""
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    from streaming_paged_kv_gb300.inputs import frame_qkv, k_head_scale
    from streaming_paged_kv_gb300.workloads import WORKLOADS
    w = WORKLOADS["s518"]
    L = args.layers or w.num_layers
    F, T, H, D = w.scale_frames, w.tokens_per_frame, w.num_heads, w.head_dim
    n_q = F * T
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else 20
    W = max(args.warmup, 3)
    c = kvc.PagedKVCache(L, H, D, w.page_size, w.dtype, w.scale_frames, w.sliding_window, w.headroom,
                         w.max_total_frames, max_query_tokens=n_q)
    if args.kernel:
        c.set_option(kvc.KVC_OPT_ATTN_KERNEL, args.kernel)
    hs = k_head_scale(args.seed + rank, w.wid, H)
    inputs = []
    for layer in range(min(args.pool, L)):
        fr = [frame_qkv(args.seed + rank, w.wid, f, layer, w.page_size, H, D, w.dtype, hs) for f in range(F)]
        inputs.append(tuple(torch.cat([x[i] for x in fr]).to(dev) for i in range(3)))
    out = torch.empty_like(inputs[0][0])

    def step():
        c.clean()
        for layer in range(L):
            q, k, v = inputs[layer % len(inputs)]
            c.prefill(layer, q, k, v, out)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, L)   # one timed launch per step
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(K):
        step()
    ev1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms, total_steps = aggregate(ev0.elapsed_time(ev1), K, world, dev)
    launches, attn_launches, attn_ms = kvc.kvc_get_counters(c.h, reset=True)
    c.set_option(kvc.KVC_OPT_TIMING, 0)
    if kvc.kvc_device_status(c.h, c._stream()) != 0:
        raise RuntimeError("device status")
    flops = K * L * 4.0 * n_q * n_q * H * D
    bytes_alg = K * L * (2.0 * n_q * H * D * 2 + 2.0 * n_q * H * D * 2)
    roof = attn_roofline(roof_bound(flops, bytes_alg), flops, bytes_alg, attn_ms, attn_launches, ms,
                         "paged attention (kvc_run attention launch inside kvc_prefill)")
    roof["outside_attn_ms_per_step"] = (ms - attn_ms) / K
    roof["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(c.h)))
    achieved = roof["attn_tflops"]
    c.close()
    return {
        "metric": PHASE1_METRIC, "value": total_steps * F / (ms / 1e3), "unit": "frames/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"phase1_518: {F} scale frames x {T} tokens, {L} layers, H={H}, D={D}, "
                               f"page_size={w.page_size}; one step = clean + prefill of every layer",
                   "l2": "no flush: the layers' caches (33 MB of K/V each, 24 blocks) exceed L2 together",
                   "parallelism": f"replicas x{world} (independent streams, no collective)"},
        "roofline": roof,
        "attn_tflops": achieved,
        "gpu_launches": launches,
        "clocks": clk,
    }


BATCH_METRIC = ("batched streams frames/s (B independent 224x224 streams, one attention launch per layer, "
                "24-layer paged attn); attn TFLOP/s vs GB300 roofline")


def run_batch224(args, rank, world):
    """Several independent 224x224 streams (one handle each) advance in
    lockstep; per layer every stream appends, evicts and (block 0) plans, then
    one kvc_run_batch launch attends all of them.  Timed region: frames
    (steady state, full window) of every stream."""
    import torch
    from streaming_paged_kv_gb300 import build
    build.build()
    from streaming_paged_kv_gb300 import kvc
    from streaming_paged_kv_gb300.workloads import WORKLOADS
    w = WORKLOADS["s224"]
    if args.layers:
        w = w.with_(num_layers=args.layers)
    B = args.batch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else 60
    W = max(args.warmup, 3)
    start = w.n_frames - K - W        # the timed frames are the stream's last K
    streams = [Stream(kvc, w, args.pool, args.seed + rank * 64 + i, args.kernel, dev, args.splits, args.qtiles)
               for i in range(B)]
    for st in streams:
        st.fast_forward(start)
    T, H, D, L = w.tokens_per_frame, w.num_heads, w.head_dim, w.num_layers
    rows = [T] * B
    qcat = [[torch.cat([st.inputs(f, b)[0] for st in streams]) for b in range(L)] for f in range(args.pool)]
    out = torch.empty(B * T, H, D, dtype=torch.bfloat16, device=dev)

    def step():
        f = streams[0].frame
        for b in range(L):
            for st in streams:
                _, k, v = st.inputs(st.frame, b)
                st.c.append_frame(b, k, v)
                st.c.evict_frames(b)
                if b == 0:
                    st.c.plan()
            kvc.run_batch([st.c for st in streams], [b] * B, qcat[(f + b) % args.pool][b], out, rows)
        for st in streams:
            st.frame += 1

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    nkv = streams[0].visible_tokens()     # every stream is in the same steady state
    flops = K * L * B * 4.0 * T * nkv * H * D
    bytes_alg = K * L * B * (2.0 * nkv * H * D * 2 + 2.0 * T * H * D * 2)
    h0 = streams[0].c
    kvc.kvc_get_counters(h0.h, reset=True)
    h0.set_option(kvc.KVC_OPT_TIMING, L)   # one timed launch per step
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(K):
        step()
    ev1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms, total_steps = aggregate(ev0.elapsed_time(ev1), K, world, dev)
    _, attn_launches, attn_ms = kvc.kvc_get_counters(h0.h, reset=True)
    launches = sum(kvc.kvc_get_counters(st.c.h, reset=True)[0] for st in streams) + _
    h0.set_option(kvc.KVC_OPT_TIMING, 0)
    for st in streams:
        if kvc.kvc_device_status(st.c.h, st.c._stream()) != 0:
            raise RuntimeError("device status")
    roof = attn_roofline(roof_bound(flops, bytes_alg), flops, bytes_alg, attn_ms, attn_launches, ms,
                         "paged attention (one kvc_run_batch launch per layer)")
    roof["outside_attn_ms_per_step"] = (ms - attn_ms) / K
    roof["launch_shape"] = dict(zip(("q_tiles", "splits"), kvc.kvc_get_launch_shape(h0.h)))
    achieved = roof["attn_tflops"]
    res = {
        "metric": BATCH_METRIC, "value": total_steps * B / (ms / 1e3), "unit": "frames/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"batch224: {B} streams x 224x224 (H={H}, D={D}, page_size={w.page_size}), "
                               f"{L} layers, frames {start + W}..{start + W + K - 1} of each {w.n_frames}-frame "
                               f"stream ({nkv} visible tokens)",
                   "l2": "no flush: the streams' visible K/V per layer together exceed L2",
                   "parallelism": f"replicas x{world} (independent streams, no collective)"},
        "roofline": roof,
        "attn_tflops": achieved,
        "gpu_launches": launches,
        "clocks": clk,
    }
    del streams
    torch.cuda.empty_cache()
    return res


def run_e2e(args, kvc, w, dev, rank, world, K, W):
    """The same frames/s through the public API with host inputs, over the
    same frames of the stream as the device-timed number: every step copies
    that frame's Q/K/V of every layer from pinned host memory and reads every
    layer's output back to pinned host memory inside the timed region (on
    their own streams, overlapping the attention launches)."""
    import torch
    K = max(1, min(K, w.n_frames))
    W = max(0, min(W, w.n_frames - K))
    T, H, D, L = w.tokens_per_frame, w.num_heads, w.head_dim, w.num_layers
    c = kvc.PagedKVCache(L, H, D, w.page_size, w.dtype, w.scale_frames, w.sliding_window,
                         w.headroom, w.max_total_frames, device=dev)
    g = torch.Generator()
    g.manual_seed(args.seed + 1000 + rank)
    host = [[torch.randn(T, H, D, generator=g).to(torch.bfloat16).pin_memory() for _ in range(3)]
            for _ in range(L)]
    host_out = [torch.empty(T, H, D, dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    # Copies overlap the attention: inputs go up on one stream and outputs
    # come back on another, into double-buffered device tensors; events order
    # each buffer's reuse after the launch that read or wrote it.
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dq = [[torch.empty(T, H, D, dtype=torch.bfloat16, device=dev) for _ in range(3)] for _ in range(2)]
    dout = [torch.empty(T, H, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    fetched = [torch.cuda.Event() for _ in range(2)]
    for e in consumed + fetched:
        e.record(comp)
    seq = [0]

    def frame(attend=True):
        for b in range(L):
            p = seq[0] & 1
            seq[0] += 1
            with torch.cuda.stream(up):
                up.wait_event(consumed[p])           # the launch that last read dq[p] is done
                for i in range(3):
                    dq[p][i].copy_(host[b][i], non_blocking=True)
                uploaded[p].record(up)
            comp.wait_event(uploaded[p])
            c.append_frame(b, dq[p][1], dq[p][2])
            c.evict_frames(b)
            if attend:
                if b == 0:
                    c.plan()
                comp.wait_event(fetched[p])          # dout[p] has been copied back
                c.run(b, dq[p][0], dout[p])
            consumed[p].record(comp)
            if attend:
                with torch.cuda.stream(down):
                    down.wait_event(consumed[p])
                    host_out[b].copy_(dout[p], non_blocking=True)
                    fetched[p].record(down)

    for _ in range(w.n_frames - K - W):
        frame(attend=False)
    for _ in range(W):
        frame()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(K):
        frame()
    torch.cuda.synchronize()
    dt, total_frames = aggregate(time.perf_counter() - t0, K, world, dev)
    c.close()
    return {"value": total_frames / dt, "unit": UNIT, "h2d_bytes_per_step": L * 3 * T * H * D * 2,
            "d2h_bytes_per_step": L * T * H * D * 2, "steps": K,
            "frames_timed": [w.n_frames - K, w.n_frames - 1]}


def compact(r):
    """The headline fields of another workload's bench line."""
    roof = r.get("roofline", {})
    keep = ("bound", "achieved", "peak", "unit", "frac", "traffic", "frac_sustained", "step_frac", "attn_tflops",
            "launch_ms", "outside_attn_ms_per_step", "launch_shape")
    out = {"metric": r["metric"], "value": r["value"], "unit": r["unit"], "steps": r["steps"],
           "ms_per_step": r["ms_per_step"], "workload": r["config"]["workload"],
           "roofline": {k: roof.get(k) for k in keep}, "gpu_launches": r.get("gpu_launches"),
           "clocks": r.get("clocks")}
    if "frame_ms" in r:
        out["frame_ms"] = r["frame_ms"]
    return out


def run_extra(args, rank, world):
    """The other workloads' numbers, measured in the same run after the
    default one: the windowed long stream (one whole window from its clean
    start, with per-frame latency percentiles), the last 60 frames of the
    224x224 stream, the last 60 frames of the keyframe + deferred-eviction
    stream, 8 batched 224x224 streams (one attention launch per layer), the
    trunk's cache beside the camera head's own cache, and the Phase-1 prefill
    of the scale frames."""
    import torch
    extra = {}
    plans = (("win518", run_windowed, {"steps": None, "warmup": 5}),
             ("s224", run_ours, {"workload": "s224", "steps": 60, "warmup": 5, "no_e2e": True}),
             ("defer", run_defer, {"steps": 60, "warmup": 5}),
             ("batch224", run_batch224, {"steps": 60, "warmup": 5}),
             ("camcache", run_paired, {"steps": 20, "warmup": 5}),
             ("phase1", run_phase1, {"steps": 10, "warmup": 3}))
    for name, fn, over in plans:
        a = argparse.Namespace(**vars(args))
        a.layers = a.frames = None
        for k, v in over.items():
            setattr(a, k, v)
        try:
            extra[name] = compact(fn(a, rank, world))
        except Exception as e:             # one failed extra must not cost the headline line
            extra[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
            if world > 1:
                raise
        torch.cuda.empty_cache()
    return extra


# ------------------------------------------------------------- CPU oracle
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


class OracleStream:
    """The oracle at the end of the stream: bookkeeping of every frame and the
    cache mirror of one block, filled by appending one fixed frame repeatedly
    (values do not change the oracle's cost)."""

    def __init__(self, w, seed):
        import numpy as np
        from oracle import OraclePagedKV
        from streaming_paged_kv_gb300.inputs import frame_qkv, k_head_scale, to_bits
        self.np = np
        self.w = w
        hs = k_head_scale(seed, w.wid, w.num_heads) if w.k_head_scale else None
        q, k, v = frame_qkv(seed, w.wid, 0, 0, w.page_size, w.num_heads, w.head_dim, w.dtype, hs)
        self.q, self.k, self.v = to_bits(q), to_bits(k), to_bits(v)
        self.orc = OraclePagedKV(1, w.page_size, w.num_heads, w.head_dim, w.dtype, w.scale_frames,
                                 w.sliding_window, w.headroom, w.max_total_frames, mirror_blocks=(0,))
        for _ in range(w.n_frames):
            self.orc.append_frame(0, self.k, self.v)
            self.orc.evict_frames(0, w.scale_frames, w.sliding_window)

    def attention_seconds(self, rows):
        from oracle import paged_attention
        t0 = time.perf_counter()
        paged_attention(self.orc, 0, self.q, rows=rows)
        return time.perf_counter() - t0

    def bookkeeping_seconds_per_frame(self, n=64):
        import numpy as np
        from oracle import OraclePagedKV
        w = self.w
        o = OraclePagedKV(w.num_layers, w.page_size, w.num_heads, w.head_dim, w.dtype,
                          w.scale_frames, w.sliding_window, w.headroom, w.max_total_frames,
                          mirror_blocks=())
        t0 = time.perf_counter()
        for _ in range(n):
            for b in range(w.num_layers):
                o.append_frame(b, self.k, self.v)
                o.evict_frames(b, w.scale_frames, w.sliding_window)
            o.visible_page_table(0)
        return (time.perf_counter() - t0) / n


def cpu_baseline(w, seed, budget_s):
    """Oracle frames/s at the end of the stream, from a bounded row sample of
    one layer's attention, extrapolated to all rows and all layers."""
    os_ = OracleStream(w, seed)
    n_q = w.tokens_per_frame
    rows_done, secs = 0, 0.0
    chunk = 16
    while secs < budget_s and rows_done < n_q:
        rows = list(range(rows_done, min(n_q, rows_done + chunk)))
        secs += os_.attention_seconds(rows)
        rows_done += len(rows)
        chunk = min(chunk * 2, 128)
    per_layer = secs * n_q / rows_done
    book = os_.bookkeeping_seconds_per_frame(8)
    per_frame = per_layer * w.num_layers + book
    return {"value": 1.0 / per_frame, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"last frame of the {w.n_frames}-frame stream "
                      f"({sum(os_.orc.visible_page_table(0)[3])} visible tokens): "
                      f"{rows_done}/{n_q} query rows x {w.num_heads} heads of one layer in {secs:.1f} s, "
                      f"scaled to {n_q} rows x {w.num_layers} layers, plus "
                      f"{book * 1e3:.2f} ms bookkeeping per frame"}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of a
    frame at the end of the stream (a slice of one layer's query rows),
    extrapolated to a whole frame."""
    w = workload(args)
    K = args.steps if args.steps is not None else 8
    W = args.warmup if args.warmup is not None else 3
    K, W = max(1, K), max(0, W)
    os_ = OracleStream(w, args.seed)
    n_q = w.tokens_per_frame
    t1 = os_.attention_seconds(list(range(8))) / 8          # calibration: seconds per row
    total_budget = 90.0
    rows = int(max(1, min(n_q, total_budget / max(K + W, 1) / max(t1, 1e-6))))
    sel = list(range(rows))
    for _ in range(W):
        os_.attention_seconds(sel)
    book = os_.bookkeeping_seconds_per_frame(4)
    secs = 0.0
    for _ in range(K):
        secs += os_.attention_seconds(sel)
    per_frame = secs / K * n_q / rows * w.num_layers + book
    value = 1.0 / per_frame
    cb = {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
          "sample": f"per step: {rows}/{n_q} query rows x {w.num_heads} heads of one layer of the last "
                    f"frame, scaled to a {w.num_layers}-layer frame, plus bookkeeping"}
    # ms_per_step is what a step took (one sample); the whole-frame time is an
    # extrapolation from it and is reported beside it.
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": K, "warmup": W, "ms_per_step": secs / K * 1e3,
            "sample_s_per_step": secs / K, "extrapolated_ms_per_frame": per_frame * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: 518x378 exact-page stream, {w.num_layers} layers, "
                                   f"H={w.num_heads}, D={w.head_dim}, page_size={w.page_size}, "
                                   f"{w.n_frames} frames; oracle on a row sample of the last frame"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    if args.workload in ("phase1", "batch224", "win518", "camcache", "defer"):
        res = {"phase1": run_phase1, "batch224": run_batch224, "win518": run_windowed,
               "camcache": run_paired, "defer": run_defer}[args.workload](args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return 0
    res = run_ours(args, rank, world)
    if args.workload == "s518" and not args.no_extra and not (args.layers or args.frames):
        res["extra"] = run_extra(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(workload(args), args.seed, args.cpu_budget)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
