"""The host library (page allocator, deques, plan, error paths) under
AddressSanitizer and UndefinedBehaviorSanitizer, on the CPU.

kvc_host.cpp is compiled with -fsanitize=address,undefined and linked with the
regular build's kernel objects into a separate library; a child process loads
it (KVC_LIB) with the sanitizer runtime preloaded and drives bookkeeping-only
handles against the oracle: every workload schedule with deferral and
rollback, the special-token policies, and random op mixes that hit every
error path.  Any sanitizer report, or a mismatch with the oracle, fails the
child.
"""

import os
import platform
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os
import numpy as np
from oracle import OraclePagedKV, OracleError
from streaming_paged_kv_gb300 import kvc
maps = open("/proc/self/maps").read()
assert kvc.LIB_PATH == os.environ["KVC_LIB"] and "libkvc_sanitized.so" in maps and "libasan" in maps
from streaming_paged_kv_gb300.workloads import WORKLOADS, schedule

def check(lib, orc, tag):
    assert lib.deques(0) == tuple(orc.deques(0)), tag
    assert lib.stats(0) == orc.stats(0), tag

for name in ("tiny", "defer", "s518", "win518"):
    for cross, cam in ((True, False), (False, False), (True, True)):
        w = WORKLOADS[name]
        n = min(w.n_frames, 700) if name != "win518" else w.window_frames + 30
        pol = dict(cross_frame_special=cross, camera_only=cam)
        lib = kvc.PagedKVCache(1, w.num_heads, w.head_dim, w.page_size, w.dtype, w.scale_frames,
                               w.sliding_window, w.headroom, w.max_total_frames, device=None, **pol)
        orc = OraclePagedKV(1, w.page_size, w.num_heads, w.head_dim, w.dtype, w.scale_frames,
                            w.sliding_window, w.headroom, w.max_total_frames, mirror_blocks=(), **pol)
        z = np.zeros((w.tokens_per_frame, w.num_heads, w.head_dim), np.uint32 if w.dtype == "f32" else np.uint16)
        coins = np.random.default_rng(7).random(n) < 0.5
        for f, kind in schedule(w.with_(n_frames=n), coins):
            if kind == "clean":
                lib.clean(); orc.clean(); continue
            prov = kind in ("accept", "reject")
            lib.set_defer_eviction(prov); orc.set_defer_eviction(prov)
            lib.append_frame(0); orc.append_frame(0, z, z)
            lib.evict_frames(0, **pol); orc.evict_frames(0, w.scale_frames, w.sliding_window, **pol)
            lib.plan()
            assert tuple(lib.plan_ranges()) == tuple(orc.visible_ranges(0)), (name, f)
            if kind == "accept":
                lib.execute_deferred_eviction(0); orc.execute_deferred_eviction(0, w.scale_frames, w.sliding_window)
            elif kind == "reject":
                lib.rollback_last_frame(0); orc.rollback_last_frame(0)
            lib.set_defer_eviction(False); orc.set_defer_eviction(False)
            check(lib, orc, (name, f))
        lib.close()

rng = np.random.default_rng(99)
lib = kvc.PagedKVCache(2, 2, 32, 16, "f32", 2, 4, 2, 24, device=None)
orc = OraclePagedKV(2, 16, 2, 32, "f32", 2, 4, 2, 24, mirror_blocks=())
z = np.zeros((22, 2, 32), np.uint32)
for step in range(4000):
    op, b = int(rng.integers(0, 8)), int(rng.integers(0, 2))
    if op == 5:
        on = bool(rng.random() < 0.5)
        lib.set_defer_eviction(on); orc.set_defer_eviction(on); continue
    if op == 7 and rng.random() < 0.9:
        continue
    calls = {0: (lambda: lib.append_frame(b), lambda: orc.append_frame(b, z, z)),
             1: (lambda: lib.append_frame(b), lambda: orc.append_frame(b, z, z)),
             2: (lambda: lib.evict_frames(b), lambda: orc.evict_frames(b, 2, 4)),
             3: (lambda: lib.rollback_last_frame(b), lambda: orc.rollback_last_frame(b)),
             4: (lambda: lib.execute_deferred_eviction(b), lambda: orc.execute_deferred_eviction(b, 2, 4)),
             6: (lambda: lib.plan(), lambda: None),
             7: (lambda: lib.clean(), lambda: orc.clean())}
    le = oe = None
    try:
        calls[op][0]()
    except kvc.KvcError as e:
        le = e.code
    try:
        calls[op][1]()
    except OracleError as e:
        oe = e.code
    if op != 6:
        assert le == oe, (step, op, le, oe)
for bad in (dict(page_size=5), dict(scale_frames=2000), dict(head_dim=48)):
    args = dict(num_blocks=1, num_heads=16, head_dim=64, page_size=256)
    args.update(bad)
    try:
        kvc.kvc_required_bytes(kvc.make_config(**args))
        raise SystemExit("accepted a bad config")
    except kvc.KvcError:
        pass
lib.close()
print("SANITIZED-OK")
'''


def _tool(name):
    return shutil.which(name)


def test_host_library_under_asan_and_ubsan(tmp_path):
    gxx = _tool("g++")
    if not gxx:
        pytest.skip("no g++")
    asan = subprocess.run([gxx, "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("no AddressSanitizer runtime")
    sys.path.insert(0, ROOT)
    from streaming_paged_kv_gb300 import build
    build.build(checked=False)                       # the regular build's kernel objects
    cuda = os.path.dirname(os.path.dirname(build.nvcc()))
    objdir = os.path.join(build.PKG, "_build", platform.machine())
    lib = str(tmp_path / "libkvc_sanitized.so")
    host_obj = str(tmp_path / "kvc_host.o")
    san = ["-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer"]
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-g", "-fPIC", *san, "-I", build.INCLUDE, "-I", build.CSRC,
                        "-I", os.path.join(cuda, "include"), "-c", os.path.join(build.CSRC, "kvc_host.cpp"),
                        "-o", host_obj], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    kernels = [os.path.join(objdir, f + ".o") for f in ("kvc_kernels.cu", "kvc_attn_tc.cu", "kvc_static.cu")]
    r = subprocess.run([gxx, "-shared", *san, "-o", lib, host_obj, *kernels, "-L", os.path.join(cuda, "lib64"),
                        "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, KVC_LIB=lib, LD_PRELOAD=asan, PYTHONPATH=ROOT,
               ASAN_OPTIONS="detect_leaks=0:verify_asan_link_order=0:abort_on_error=0",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, cwd=ROOT, env=env,
                       timeout=600)
    out = r.stdout + r.stderr
    assert r.returncode == 0 and "SANITIZED-OK" in out, out[-4000:]
    assert "AddressSanitizer" not in out and "runtime error" not in out, out[-4000:]
