"""Benchmark: GDN chunked-prefill tokens/s per layer on GB300, with roofline fraction.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

One step = one gdn_chunk_fwd call (every operator of the chunkwise forward)
over one batch of the headline workload (16 heads of 128, 4096 tokens, bf16;
see linear_attention_prefill_gb300/workloads.py).  Inputs are resident in HBM
when timing starts; L2 (129 MB) is flushed by writing a 320 MB buffer before
every timed step, outside the timed events.  Each step is timed with CUDA events
on the launching stream; the job time is the max over ranks.  Under torchrun
every rank runs its own batch (weak scaling, no collective on the data path).

Prints one JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload instead.

CPU baselines (rank 0, N = 1, outside every timed GPU region): the fp64 oracle over
v heads in a spawn-started process pool on the host cores (``cpu_baseline``), which
also checks the GPU output of the timed calls on that sample (``parity``), and the
fp32 per-token recurrence in C with OpenMP on all host cores and on one core
(``cpu_baseline.fp32_recurrence``).
"""
from __future__ import annotations

import os

# the CPU oracle legs time one core: keep BLAS from spawning threads
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import csv
import io
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_prefill_gb300 import roofline  # noqa: E402
from linear_attention_prefill_gb300.sharding import rank_seed, reduce_timing  # noqa: E402
from linear_attention_prefill_gb300.workloads import HEADLINE, WORKLOADS, make_decode_inputs, make_inputs  # noqa: E402

METRIC = "GDN chunked-prefill tokens/s per layer on 1 GB300; % of TC/HBM roofline"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 320 * 2 ** 20
# One forward call is two launches on the caller's stream (the chunk-parallel prep
# kernel, then the chunk-serial chain kernel that also writes o), in bf16 and fp32
# alike.  The roofline block times the call, and the launch list in profiles/ gives
# each kernel's share.
KERNEL_NAME = "gdn_chunk_fwd (gdn_prep_kernel + gdn_chain_kernel)"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy peak is the roofline's)
KERNEL_NAMES = {"ssd": "ssd_chunk_fwd (gdn_prep_kernel + gdn_chain_kernel, no erase term)",
                "kda": "kda_chunk_fwd (kda_prep_kernel + gdn_chain_kernel in KDA mode)",
                "gdn_prologue": "gdn_chunk_fwd_prologue (gdn_prep_kernel with the fused prologue + "
                                "gdn_chain_kernel)",
                "f32": "gdn_chunk_fwd_f32 (gdn_prep_f32_kernel + gdn_chain_f32_kernel)",
                "ssd_f32": "ssd_chunk_fwd_f32 (gdn_prep_f32_kernel + gdn_chain_f32_kernel, no erase "
                           "term)"}


def kernel_name(w, chain="dv_tile") -> str:
    if w.dtype == "f32":
        return KERNEL_NAMES["ssd_f32" if w.op == "ssd" else "f32"]
    if chain == "tc":
        fn = "gdn_chunk_fwd_prologue" if w.prologue else f"{w.op}_chunk_fwd"
        return f"{fn} (gdn_prep_tc_kernel + gdn_chain_tc_kernel)"
    return KERNEL_NAMES.get("gdn_prologue" if w.prologue else w.op, KERNEL_NAME)


def chain_of(lap, w, choice) -> str:
    """The chain kernel the bf16 forward of ``w`` runs ("tc" or "dv_tile"; "-" for fp32)
    under --chain ``choice``."""
    if w.dtype == "f32":
        return "-"
    forced = {"auto": None, "tc": True, "dv_tile": False}[choice]
    return lap.chain_kind(w.n_seqs, w.Hv, w.dk, w.dv, w.op, forced)


CHAIN_LABEL = {"tc": "tcgen05, one CTA per chain (state in registers, products in tensor memory)",
               "dv_tile": "mma.sync, one CTA per (chain, dv tile)",
               "-": "split-precision tf32 mma.sync (three products per step), one CTA per "
                    "(chain, 16 dv columns)"}


def launches_per_call(w) -> int:
    """Kernel launches of one forward call: a prep launch and a chain launch (bf16 and
    fp32 paths alike)."""
    return 2


def measured_traffic(workload: str):
    """DRAM bytes (read + write) per forward call, summed over its launches, from a
    committed ncu capture - only if it was taken on this exact kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_hash") != roofline.kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_call")


def config_of(w, world, extra=None, l2_flush="write"):
    cfg = {"workload": w.name, "seqlens": list(w.seqlens) if len(w.seqlens) <= 16 else len(w.seqlens),
           "T_total": w.T_total, "Hqk": w.Hqk, "Hv": w.Hv, "dk": w.dk, "dv": w.dv,
           "chunk": w.chunk, "h0": w.h0_std is not None, "global_batch": w.n_seqs * world,
           "seq_len": max(w.seqlens), "l2": f"flushed (320 MB {l2_flush}) before every timed step",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if extra:
        cfg.update(extra)
    return cfg


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 10]
        self.file.close()
        os.unlink(self.file.name)
        if not rows:
            return None
        mhz = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        max_mhz = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(max_mhz) if max_mhz else None, "reasons": reasons,
                "samples": len(rows)}


def run_decode(lap, w, dev, steps=1000):
    """Decode on workload ``w``'s state shape, continuing from its prefill: one forward
    gives hT, then ``steps`` one-token steps update it in place - timed as separate
    launches and as one CUDA graph of all the steps.  Returns µs per step and the HBM
    bandwidth that implies (state read + written, the token's q, k, v, g, beta and o)."""
    stepfn = {"ssd": lap.ssd_recurrent_step, "kda": lap.kda_recurrent_step}.get(
        w.op, lap.gdn_recurrent_step)
    fwd = {"ssd": lap.ssd_chunk_fwd, "kda": lap.kda_chunk_fwd}.get(w.op, lap.gdn_chunk_fwd)
    x = make_inputs(w, device=dev)
    _, h = fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=w.chunk,
               scale=w.scale, cu_seqlens=x["cu_seqlens"])
    del x
    toks = [make_decode_inputs(w, s, device=dev) for s in range(steps)]
    d = {n: torch.stack([t[n] for t in toks]) for n in ("q", "k", "v", "g", "beta")}
    del toks
    N, Hv = w.n_seqs, w.Hv
    o = torch.empty((steps, N, Hv, w.dv), dtype=d["q"].dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run_all():
        for s in range(steps):
            stepfn(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], h, o[s],
                   scale=w.scale)

    run_all()  # warm-up (and the state keeps evolving from the prefill's)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run_all()
    b.record(stream)
    torch.cuda.synchronize()
    plain = a.elapsed_time(b) * 1e3 / steps
    graph_us = None
    try:
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run_all()
        stream.wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_us = a.elapsed_time(b) * 1e3 / steps
    except RuntimeError:
        graph_us = None
    nbytes = roofline.decode_bytes(N, w.Hqk, Hv, w.dk, w.dv, 2 if w.dtype == "bf16" else 4,
                                   gate_per_channel=w.op == "kda")
    peaks, _ = roofline.load_peaks()
    out = {"workload": w.name, "from": "the prefill's final state", "steps": steps,
           "us_per_step": round(plain, 3),
           "us_per_step_cuda_graph": None if graph_us is None else round(graph_us, 3),
           "bytes_per_step": nbytes,
           "achieved_gbs_graph": None if graph_us is None else round(nbytes / graph_us / 1e3, 1)}
    if graph_us is not None:
        out["hbm_frac_graph"] = round(nbytes / graph_us / 1e3 / peaks["hbm_gbs"], 4)
    return out


def oracle_tokens_per_s(w, x_cpu, budget_s):
    """fp64 oracle (one core) on the first tokens of every head; returns (tok/s, sample)."""
    from oracle import gdn_recurrent, kda_recurrent, prologue, ssd_recurrent
    fwd = {"ssd": ssd_recurrent, "kda": kda_recurrent}.get(w.op, gdn_recurrent)
    if w.prologue:  # the oracle's prologue, then the recurrence
        def fwd(q, k, v, a, b, scale, h0, _f=fwd):
            qn, kn, g, beta = prologue(q, k, a, b)
            return _f(qn, kn, v, g, beta, scale, h0)
    H = w.Hv
    # calibrate: a few tokens of every head
    probe = 16
    t = time.perf_counter()
    sl = {k_: v_[:, :probe] for k_, v_ in x_cpu.items() if k_ in ("q", "k", "v", "g", "beta")}
    fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], w.scale, x_cpu["h0"][:1] if x_cpu["h0"] is not None else None)
    per_tok = (time.perf_counter() - t) / probe
    n_tok = int(max(probe, min(w.seqlens[0], budget_s / per_tok)))
    sl = {k_: v_[:, :n_tok] for k_, v_ in x_cpu.items() if k_ in ("q", "k", "v", "g", "beta")}
    h0 = x_cpu["h0"][:1] if x_cpu["h0"] is not None else None
    t = time.perf_counter()
    fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], w.scale, h0)
    dt = time.perf_counter() - t
    return n_tok / dt, f"first {n_tok} tokens of sequence 0, all {H} v heads, fp64 numpy, 1 thread", dt


def _oracle_head(args):
    """One v head of the fp64 oracle (a spawn-started pool worker).  The inputs and the
    output live in shared memory blocks named in ``args``; returns the seconds taken."""
    from multiprocessing import shared_memory
    op, names, shapes, hv, hq, n_tok, scale, has_h0 = args
    blocks = {n: shared_memory.SharedMemory(name=names[n]) for n in names}
    try:
        arr = {n: np.ndarray(shapes[n], dtype=np.float64, buffer=blocks[n].buf) for n in names}
        import oracle
        fwd = {"ssd": oracle.ssd_recurrent, "kda": oracle.kda_recurrent}.get(op,
                                                                           oracle.gdn_recurrent)
        sl = slice(0, n_tok)
        t = time.perf_counter()
        o, _ = fwd(arr["q"][:, sl, hq:hq + 1], arr["k"][:, sl, hq:hq + 1],
                   arr["v"][:, sl, hv:hv + 1], arr["g"][:, sl, hv:hv + 1],
                   arr["beta"][:, sl, hv:hv + 1], scale,
                   arr["h0"][:, hv:hv + 1] if has_h0 else None)
        dt = time.perf_counter() - t
        arr["o"][:n_tok, hv] = o[0, :, 0]
        return dt
    finally:
        for b in blocks.values():
            b.close()


def oracle_pool_rate(w, xc, budget_s, workers):
    """The fp64 oracle over the first n tokens of every v head of row 0, one head per task
    in a pool of ``workers`` spawn-started processes (inputs and output in shared memory),
    n sized so the pool's wall time is about ``budget_s``.  Returns (tokens/s of the layer,
    sample text, wall s, o [n, Hv, dv])."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    T = w.seqlens[0]
    src = {n: xc[n][:1, :T].float().numpy() for n in ("q", "k", "v", "g", "beta")}
    if xc["h0"] is not None:
        src["h0"] = xc["h0"][:1].numpy()
    src["o"] = np.zeros((T, w.Hv, w.dv))
    blocks, names, shapes = {}, {}, {}
    try:
        for n, a in src.items():
            b = shared_memory.SharedMemory(create=True, size=max(8, a.size * 8))
            np.ndarray(a.shape, dtype=np.float64, buffer=b.buf)[...] = a
            blocks[n], names[n], shapes[n] = b, b.name, a.shape
        rep = w.Hv // w.Hqk

        def tasks(n_tok):
            return [(w.op, names, shapes, hv, hv // rep, n_tok, w.scale, "h0" in src)
                    for hv in range(w.Hv)]
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            probe = min(T, 64)
            per_tok = max(pool.map(_oracle_head, tasks(probe)[:workers])) / probe
            waves = -(-w.Hv // workers)
            n_tok = int(max(probe, min(T, budget_s / (per_tok * waves))))
            t = time.perf_counter()
            pool.map(_oracle_head, tasks(n_tok))
            wall = time.perf_counter() - t
        o = np.ndarray(shapes["o"], dtype=np.float64, buffer=blocks["o"].buf)[:n_tok].copy()
    finally:
        for b in blocks.values():
            b.close()
            b.unlink()
    sample = (f"first {n_tok} tokens of sequence 0, all {w.Hv} v heads, fp64 numpy, "
              f"one head per task, {workers} processes")
    return n_tok / wall, sample, wall, o


def parity_sample(o_gpu, o_ref, dtype):
    """max |x - ref| / RMS(ref) raw and after half a bf16 ulp of |ref| per element, and the
    NMSE, of the GPU output against the oracle on the sampled tokens."""
    x = o_gpu.astype(np.float64)
    d = np.abs(x - o_ref)
    rms = float(np.sqrt(np.mean(o_ref ** 2))) or 1.0
    adj = d
    if dtype == "bf16":
        a = np.abs(o_ref)
        half_ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
        adj = np.maximum(d - half_ulp, 0.0)
    return {"max_abs_over_rms": float(d.max() / rms), "max_abs_over_rms_adjusted":
            float(adj.max() / rms), "nmse": float(np.sum(d ** 2) / np.sum(o_ref ** 2)),
            "tolerance": 2e-2 if dtype == "bf16" else 1e-4}


def fp32_recurrence_baseline(w, xc, budget_s):
    """The fp32 per-token recurrence (C, OpenMP) on all host cores and on one core; tokens/s
    of the layer.  All cores run row 0 whole when that fits the budget, else a prefix."""
    import cpu_baseline as cb
    cores = cb.host_cores()
    x = {n: (None if xc[n] is None else xc[n].float().numpy()) for n in
         ("q", "k", "v", "g", "beta", "h0")}
    x["cu_seqlens"] = None
    T = w.seqlens[0]
    probe = {n: (None if a is None else a[:, :min(T, 256)]) if n != "h0" else a for n, a in x.items()}
    probe["cu_seqlens"] = None
    t = cb.time_recurrence_f32(probe, w.scale, cores)
    n_tok = int(max(64, min(T, budget_s / max(t / min(T, 256), 1e-9))))
    xs = {n: (None if a is None else a[:, :n_tok]) if n not in ("h0", "cu_seqlens") else a
          for n, a in x.items()}
    t_all = cb.time_recurrence_f32(xs, w.scale, cores, reps=3)
    # one core: one q/k head and the v heads that read it, over the same tokens; the
    # layer's rate on one core counts all Hqk such groups
    t_group = cb.time_recurrence_f32(xs, w.scale, 1, groups=1, reps=2)
    return {"value": n_tok / t_all, "unit": UNIT, "cores": cores, "kind": "fp32 per-token recurrence "
            "(C, OpenMP over (sequence, v head) chains)", "cpu_model": cb.cpu_model(),
            "sample": f"first {n_tok} tokens of sequence 0, all {w.Hv} v heads",
            "one_core": {"value": n_tok / (t_group * w.Hqk), "unit": UNIT, "cores": 1,
                         "sample": f"the same tokens, one q/k head group of {w.Hv // w.Hqk} v "
                                   f"heads, timed and scaled to the layer's {w.Hqk} groups"}}


def cpu_inputs(w, x):
    """The same tensors on the host (first sequence row only) for the oracle legs."""
    out = {}
    for k_ in ("q", "k", "v", "g", "beta"):
        out[k_] = x[k_][:1].detach().cpu()
    out["h0"] = None if x["h0"] is None else x["h0"][:1].detach().cpu()
    return out


def oracle_workers(w):
    """Processes for the oracle pool: the host's cores, at most one per v head."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, w.Hv))


def bench_reference(args, w, rank, world):
    if rank != 0:
        return
    x = make_inputs(w, device="cpu")
    xc = cpu_inputs(w, x)
    workers = oracle_workers(w)
    times, rates = [], []
    sample = ""
    if w.prologue:
        for _ in range(args.warmup):
            oracle_tokens_per_s(w, xc, 0.05)
        for _ in range(args.steps):
            r, sample, dt = oracle_tokens_per_s(w, xc, args.ref_step_s)
            rates.append(r)
            times.append(dt)
        workers = 1
    else:
        for _ in range(args.warmup):
            oracle_pool_rate(w, xc, 0.05, workers)
        for _ in range(args.steps):
            r, sample, dt, _ = oracle_pool_rate(w, xc, args.ref_step_s, workers)
            rates.append(r)
            times.append(dt)
    value = len(rates) / sum(1.0 / r for r in rates)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, 1), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_cuda(args, w, rank, world, local_rank):
    import linear_attention_prefill_gb300 as lap
    lap.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    x = make_inputs(w, device=dev, seed=rank_seed(w.seed, rank))
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if args.l2_flush == "read":  # a reduction over the buffer: L2 left holding clean lines
        flush.zero_()
        sink = torch.empty((), dtype=torch.float32, device=dev)

        def flush_l2():
            torch.sum(flush, dim=0, out=sink)
    else:
        def flush_l2():
            flush.zero_()
    o = torch.empty_like(x["v"])
    hT = torch.empty((w.n_seqs, w.Hv, w.dk, w.dv), dtype=torch.float32, device=dev)

    fwd = {"ssd": lap.ssd_chunk_fwd, "kda": lap.kda_chunk_fwd}.get(w.op, lap.gdn_chunk_fwd)
    if w.prologue:  # raw q, k and gate inputs through the fused prologue
        def fwd(q, k, v, a, b, h0, o, hT, **kw):
            return lap.gdn_chunk_fwd_prologue(q, k, v, a, b, None, None, h0, o, hT, **kw)
    chain = chain_of(lap, w, args.chain)
    # fp32 and KDA have one chain each (config.chain names the one that ran)
    extra = ({} if w.dtype == "f32" or w.op == "kda" or args.chain == "auto"
             else {"tc_chain": args.chain == "tc"})

    def step():
        fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o, hT, chunk=w.chunk,
            scale=w.scale, cu_seqlens=x["cu_seqlens"], stream=stream, **extra)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.25)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        flush_l2()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = [a.elapsed_time(b) for a, b in evs]
    clk = clocks.stop()
    # a bounded device-side wait that gave up, or an operand out of range, voids the run
    lap.gdn_device_status(stream)
    local_ms = sum(ms)
    job_ms, job_tokens = reduce_timing(local_ms, float(w.T_total * args.steps))
    value = job_tokens / (job_ms / 1e3)
    launches = launches_per_call(w) * args.steps

    # end to end through the public API from pinned host memory: every step copies its
    # inputs in and o, hT out; consecutive steps run on two streams so the upload of
    # one overlaps the compute and download of the previous (HostPipeline)
    host = {k_: (None if x[k_] is None else x[k_].detach().cpu().pin_memory())
            for k_ in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens")}
    pipe = lap.HostPipeline(chunk=w.chunk, device=dev,
                            op="gdn_prologue" if w.prologue else w.op, depth=2,
                            scale=w.scale, **extra)
    for _ in range(max(2, args.warmup)):
        pipe.submit(host)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    bi = bo = 0
    for _ in range(e2e_steps):
        _, _, _, bi, bo = pipe.submit(host)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_ms, e2e_tok = reduce_timing(e2e_s * 1e3, float(w.T_total * e2e_steps))
    e2e_value = e2e_tok / (e2e_ms / 1e3)

    decode = run_decode(lap, WORKLOADS[args.decode_workload], dev) if args.decode else None
    lap.gdn_device_status(stream)  # the end-to-end and decode runs as well

    if rank != 0:
        return
    peaks, src = roofline.load_peaks()
    model = roofline.workload_model(w, peaks)
    avg_s = statistics.mean(ms) / 1e3
    achieved = model["bytes"] / avg_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": job_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_of(w, world, {"chain": CHAIN_LABEL[chain]}, args.l2_flush),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": measured_traffic(w.name + (":tc" if chain == "tc" else "")),
                     "peak_source": src,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": kernel_name(w, chain),
                     "algorithmic_bytes": model["bytes"],
                     "algorithmic_flops": model["flops"],
                     "tensor_frac": round(model["flops"] / avg_s / 1e12 / peaks["bf16_tflops"], 4),
                     "t_roof_us": round(model["t_roof"] * 1e6, 2),
                     "roofline_frac": round(model["t_roof"] / avg_s, 4)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "streams": 2},
        "gpu_launches": launches,
        "clocks": clk,
        "kernel_ms": {"median": statistics.median(ms), "min": min(ms), "max": max(ms)},
    }
    if decode is not None:
        line["decode"] = decode
    if world == 1 and args.cpu_baseline:
        xc = cpu_inputs(w, x)
        o_cpu = o[:1].float().cpu().numpy()
        if w.prologue:
            rate, sample, _ = oracle_tokens_per_s(w, xc, args.cpu_baseline_s)
            cores = 1
            par = None
        else:
            cores = oracle_workers(w)
            rate, sample, _, o_ref = oracle_pool_rate(w, xc, args.cpu_baseline_s, cores)
            par = parity_sample(o_cpu[0, :o_ref.shape[0]], o_ref, w.dtype)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample}
        if w.op == "gdn" and not w.prologue:
            line["cpu_baseline"]["fp32_recurrence"] = fp32_recurrence_baseline(
                w, xc, args.cpu_baseline_s / 2)
        if par is not None:
            line["parity"] = dict(par, sample=sample)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-baseline-s", type=float, default=10.0)
    ap.add_argument("--ref-step-s", type=float, default=0.5)
    ap.add_argument("--no-decode", dest="decode", action="store_false")
    ap.add_argument("--l2-flush", default="write", choices=["write", "read"],
                    help="how L2 is flushed before each timed step: writing a 320 MB buffer "
                         "(default), or reading it, which leaves no dirty lines behind - for DRAM "
                         "traffic captures with ncu --cache-control none")
    ap.add_argument("--chain", default="auto", choices=["auto", "tc", "dv_tile"],
                    help="chunk-serial kernel of the bf16 forward: the library's own choice "
                         "(default), the tensor-memory chain, or the dv-tile chain")
    ap.add_argument("--decode-workload", default="long_64k_weak", choices=sorted(WORKLOADS),
                    help="state shape of the decode measurement (continues from its prefill)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        bench_reference(args, w, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        bench_cuda(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
