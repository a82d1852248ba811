"""Algorithmic byte and FLOP model of the GDN chunked-prefill forward.

Bytes: every tensor that must cross HBM once and only once - q, k, v, o in the
input dtype, g and beta in fp32 (one scalar per token and v head), and the
fp32 [dk, dv] state per (sequence, v head) read (h0) and written (hT).  This is
the "ideal resident" global-memory traffic of "Empowering Hybrid Attention
Models on NPUs", Figure 4(a): at T=2048, H=10, d=128 with FP16 Q/K/V/O and
FP32 gates and state it gives 21.41 MiB for GDN, and 31.33 MiB once the gate
is per channel as in KDA (checked by a golden test).

FLOPs: per token and v head, counting only the triangles the method needs
(strictly lower KK^T, lower-with-diagonal QK^T and its product with V_new,
lower-triangular Tm in the W/U products, the solve, and the three dk x dv
state products: W h, Q h and the update), times 2.
"""
from __future__ import annotations

import json
import os

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}

# sm_103a: 152 SMs, 128 fp32 lanes per SM, one FMA (2 FLOP) per lane per clock.
SM_COUNT = 152
FP32_LANES_PER_SM = 128


def load_peaks(path=None):
    """Measured peaks (HBM GB/s, dense bf16 TFLOP/s); falls back to fixed figures.

    Returns (peaks dict, source) with source "measured" or "fallback".
    """
    if path is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        if pk.get("hbm_gbs") and pk.get("bf16_tflops"):
            return pk, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def io_bytes(T_total, n_seqs, Hqk, Hv, dk, dv, elem_bytes, h0_read=False, hT_written=True,
             gate_per_channel=False):
    """Bytes that must cross HBM once: q, k, v, o, g, beta, h0, hT."""
    per_token = 2 * Hqk * dk * elem_bytes + 2 * Hv * dv * elem_bytes
    per_token += Hv * 4 * (dk if gate_per_channel else 1)   # g
    per_token += Hv * 4                                       # beta
    state = n_seqs * Hv * dk * dv * 4
    return T_total * per_token + state * (int(h0_read) + int(hT_written))


def macs_per_token_head(chunk, dk, dv):
    """Multiply-adds per token per v head (triangles only)."""
    C = chunk
    kkt = (C - 1) / 2 * dk
    qkt = (C + 1) / 2 * dk
    wu = (C + 1) / 2 * (dk + dv)
    solve = C * C / 6
    state = 3 * dk * dv
    pv = (C + 1) / 2 * dv
    return kkt + qkt + wu + solve + state + pv


def ssd_macs_per_token_head(chunk, dk, dv):
    """The SSD scan's four stages: C B^T gram, intra-chunk output, Q h, state update."""
    C = chunk
    return (C + 1) / 2 * dk + (C + 1) / 2 * dv + 2 * dk * dv


def flops(T_total, Hv, chunk, dk, dv, op="gdn"):
    # KDA has GDN's products (its per-channel gate adds exponentials, not MACs)
    per = ssd_macs_per_token_head if op == "ssd" else macs_per_token_head
    return 2.0 * T_total * Hv * per(chunk, dk, dv)


def decode_bytes(n_seqs, Hqk, Hv, dk, dv, elem_bytes, gate_per_channel=False):
    """One decode step: the fp32 state read and written, plus one token of q, k, v, o, g, beta
    (g per key channel for KDA)."""
    return (n_seqs * Hv * dk * dv * 4 * 2
            + n_seqs * (2 * Hqk * dk + 2 * Hv * dv) * elem_bytes
            + n_seqs * Hv * 4 * ((dk if gate_per_channel else 1) + 1))


def fp32_alu_tflops(sm_mhz):
    return SM_COUNT * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def workload_model(w, peaks):
    """Bytes, FLOPs and roofline time of one forward call of workload ``w``."""
    eb = 4 if w.dtype == "f32" else 2
    b = io_bytes(w.T_total, w.n_seqs, w.Hqk, w.Hv, w.dk, w.dv, eb,
                 h0_read=w.h0_std is not None, hT_written=True,
                 gate_per_channel=getattr(w, "op", "gdn") == "kda")
    f = flops(w.T_total, w.Hv, w.chunk, w.dk, w.dv, getattr(w, "op", "gdn"))
    t_hbm = b / (peaks["hbm_gbs"] * 1e9)
    if w.dtype == "f32":
        tc = fp32_alu_tflops(peaks.get("sm_max_mhz", 2070.0)) * 1e12
    else:
        tc = peaks["bf16_tflops"] * 1e12
    t_fl = f / tc
    return dict(bytes=b, flops=f, t_hbm=t_hbm, t_flop=t_fl, t_roof=max(t_hbm, t_fl),
                bound="hbm" if t_hbm >= t_fl else ("alu" if w.dtype == "f32" else "tensor"))


# ---- measured DRAM traffic (ncu) ---------------------------------------------------
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_hash() -> str:
    """Hash of every CUDA source of the library: a traffic figure is shown only for
    the exact sources it was measured on."""
    import hashlib
    csrc = os.path.join(ROOT, "linear_attention_prefill_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_ncu_csv(path, launches_per_call):
    """DRAM bytes per forward call from an ncu --csv launch list that holds
    dram__bytes_read.sum and dram__bytes_write.sum for whole calls of
    ``launches_per_call`` consecutive launches; returns (bytes per call, per-kernel
    read/write means)."""
    import csv
    rows = []
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        rows.append(r)
    launches = {}
    for r in rows:
        d = launches.setdefault(int(r["ID"]), {"kernel": r["Kernel Name"]})
        if r["Metric Name"] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            d[r["Metric Name"]] = float(r["Metric Value"].replace(",", ""))
    ids = sorted(launches)
    calls = len(ids) // launches_per_call
    if calls == 0:
        raise ValueError(f"{path}: fewer than {launches_per_call} launches")
    per_call = []
    kernels = {}
    for c in range(calls):
        tot = 0.0
        for i in ids[c * launches_per_call:(c + 1) * launches_per_call]:
            d = launches[i]
            rd, wr = d.get("dram__bytes_read.sum", 0.0), d.get("dram__bytes_write.sum", 0.0)
            tot += rd + wr
            k = kernels.setdefault(d["kernel"].split("(")[0], [0.0, 0.0, 0])
            k[0] += rd
            k[1] += wr
            k[2] += 1
        per_call.append(tot)
    kern = {k: {"dram_read": int(v[0] / v[2]), "dram_write": int(v[1] / v[2])}
            for k, v in kernels.items()}
    return int(sum(per_call) / len(per_call)), kern


CACHE_NOTES = {
    "cold": "ncu flushes L2 before each profiled launch; mean over the profiled calls",
    "none": "ncu --cache-control none (no flush between the launches of a call); L2 flushed "
            "by reading a 320 MB buffer before each call (bench.py --l2-flush read); mean over "
            "the profiled calls",
}


def write_traffic(csv_path, workload, kernel, launches_per_call, source, cache="none"):
    """Record a workload's measured DRAM bytes per call in profiles/traffic.json, stamped
    with the current kernel source hash."""
    per_call, kern = traffic_from_ncu_csv(csv_path, launches_per_call)
    try:
        with open(TRAFFIC_JSON) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data[workload] = {"kernel": kernel, "kernel_source_hash": kernel_source_hash(),
                      "dram_bytes_per_call": per_call, "kernels": kern,
                      "cache": CACHE_NOTES[cache], "source": source}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(data, f, indent=1)
    return per_call


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser(description="record measured DRAM traffic per forward call "
                                             "from an ncu --csv launch list")
    ap.add_argument("csv")
    ap.add_argument("--workload", required=True)
    ap.add_argument("--kernel", required=True, help="what one call launches")
    ap.add_argument("--launches-per-call", type=int, default=2)
    ap.add_argument("--source", default="", help="the profiles/ summary of the capture")
    ap.add_argument("--cache", default="none", choices=sorted(CACHE_NOTES),
                    help="how the capture treated L2")
    a = ap.parse_args()
    print(write_traffic(a.csv, a.workload, a.kernel, a.launches_per_call, a.source, a.cache))
