"""CPU baselines the GPU forward is reported beside (measurement only, never on the GPU path).

* ``recurrence_f32``: the fp32 per-token recurrence of the gated delta rule in C with
  OpenMP over (sequence, v head) chains (gdn_cpu_recurrence.c) - the CPU operator
  that "Exp 2026-07-13 - Linear-Attention Scans on the NPU" (§4) found faster than its
  NPU scan.  Built by ``build()`` with the host's gcc (no architecture flags, so the
  same source builds on x86-64 and Arm).
* ``oracle_pool``: the fp64 oracle timed over v heads in a spawn-started process pool
  (the same parallelisation over chains).

Host facts recorded beside the numbers: ``cpu_model()`` and ``host_cores()``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "gdn_cpu_recurrence.c")
_LIB = os.path.join(_DIR, "libgdn_cpu.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libgdn_cpu.so next to its source (gcc -O3 -fopenmp); returns its path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp"
    r = subprocess.run(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed on {_SRC}:\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.gdn_cpu_recurrence_f32.restype = I
        lib.gdn_cpu_recurrence_f32.argtypes = [P] * 8 + [I] * 6 + [F, P, I]
        lib.gdn_cpu_max_threads.restype = I
        lib.gdn_cpu_max_threads.argtypes = []
        _lib = lib
    return _lib


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def recurrence_f32(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, threads=None):
    """fp32 per-token recurrence on the host; returns (o [.., Hv, dv], hT [N, Hv, dk, dv]).

    q, k [rows, T, Hqk, dk]; v [rows, T, Hv, dv]; g, beta [rows, T, Hv]; h0 [N, Hv, dk, dv]
    or None; cu_seqlens int32 [N + 1] (rows = 1) or None (N = rows).  Any float dtype in,
    converted to fp32 once.
    """
    lib = _load()
    q, k, v, g, beta, h0 = (_f32(a) for a in (q, k, v, g, beta, h0))
    rows, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = rows if cu is None else len(cu) - 1
    o = np.empty((rows, T, Hv, dv), dtype=np.float32)
    hT = np.empty((N, Hv, dk, dv), dtype=np.float32)
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.gdn_cpu_recurrence_f32(ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(h0), ptr(o),
                                    ptr(hT), N, T, Hqk, Hv, dk, dv, float(scale), ptr(cu),
                                    int(threads or host_cores()))
    if rc != 0:
        raise MemoryError("gdn_cpu_recurrence_f32: no memory for a state buffer")
    return o, hT


def time_recurrence_f32(x, scale, threads, groups=None, reps=1):
    """Seconds of one recurrence_f32 call over the inputs ``x`` (numpy dict: q, k, v, g,
    beta, h0, cu_seqlens), best of ``reps``.  ``groups`` keeps only the first that many
    q/k heads and the v heads that read them (the grouped map stays exact); None = all."""
    q, k, v, g, beta, h0 = (x[n] for n in ("q", "k", "v", "g", "beta", "h0"))
    if groups is not None:
        rep = v.shape[2] // q.shape[2]
        q, k = q[:, :, :groups], k[:, :, :groups]
        v, g, beta = v[:, :, :groups * rep], g[:, :, :groups * rep], beta[:, :, :groups * rep]
        h0 = None if h0 is None else h0[:, :groups * rep]
    args = [_f32(a) for a in (q, k, v, g, beta, h0)]
    best = None
    for _ in range(reps):
        t = time.perf_counter()
        recurrence_f32(*args[:5], scale, args[5], x.get("cu_seqlens"), threads)
        dt = time.perf_counter() - t
        best = dt if best is None else min(best, dt)
    return best


def _oracle_head(args):
    """One v head of the fp64 oracle (a pool worker); returns its seconds."""
    q, k, v, g, beta, scale, h0, op = args
    import oracle
    fwd = {"ssd": oracle.ssd_recurrent, "kda": oracle.kda_recurrent}.get(op, oracle.gdn_recurrent)
    t = time.perf_counter()
    fwd(q, k, v, g, beta, scale, h0)
    return time.perf_counter() - t


def oracle_pool(x, scale, n_tok, workers, op="gdn"):
    """Wall seconds of the fp64 oracle over the first ``n_tok`` tokens of every v head of
    row 0, one head per task in a pool of ``workers`` spawn-started processes."""
    import multiprocessing as mp
    q, k, v, g, beta, h0 = (x[n] for n in ("q", "k", "v", "g", "beta", "h0"))
    Hqk, Hv = q.shape[2], v.shape[2]
    rep = Hv // Hqk
    tasks = []
    for hv in range(Hv):
        hq = hv // rep
        sl = slice(0, n_tok)
        tasks.append((np.asarray(q[:1, sl, hq:hq + 1], np.float64),
                      np.asarray(k[:1, sl, hq:hq + 1], np.float64),
                      np.asarray(v[:1, sl, hv:hv + 1], np.float64),
                      np.asarray(g[:1, sl, hv:hv + 1], np.float64),
                      np.asarray(beta[:1, sl, hv:hv + 1], np.float64), scale,
                      None if h0 is None else np.asarray(h0[:1, hv:hv + 1], np.float64), op))
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_head, tasks[:workers])  # warm the workers (imports)
        t = time.perf_counter()
        pool.map(_oracle_head, tasks)
        return time.perf_counter() - t
