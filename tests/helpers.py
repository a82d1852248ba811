"""Shared helpers for the GPU parity tests: run the oracle on chosen chains of the
very tensors handed to the kernel, the error measures of the tolerance, and a
record of every comparison (printed at the end of the run by conftest.py)."""
import numpy as np
import torch

from oracle import gdn_recurrent, kda_recurrent, qk_head, ssd_recurrent

# max |x - x_ref| / RMS(x_ref): bf16 inputs with fp32 accumulation, and the fp32 path.
# o is stored in the input dtype; for bf16 the comparison first allows half an ulp of the
# exact value's own bf16 storage (see rel_err).  The fp32 final state has no allowance.
TOL = {"bf16": 2e-2, "f32": 1e-4}

# (test, quantity, raw max-abs/RMS, max-abs/RMS after the storage allowance, NMSE)
RECORDS = []


def half_ulp(x, dtype):
    """Half a unit in the last place of |x| in ``dtype`` ("bf16": 8 significant bits)."""
    if dtype != "bf16":
        return np.zeros_like(x)
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def rel_err(x, ref, out_dtype=None):
    """max |x - ref| / RMS(ref).

    With ``out_dtype="bf16"`` ``x`` is a stored bf16 result: storing the exact value
    ``ref`` in bf16 alone moves it by up to half an ulp of |ref|, so that much is taken
    off each element's difference before the arithmetic error is measured.  The
    allowance depends on the reference only, so a wrong x cannot widen it.
    """
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    d = np.abs(x - ref)
    if out_dtype is not None:
        d = np.maximum(d - half_ulp(ref, out_dtype), 0.0)
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0.0:
        return float(d.max())
    return float(d.max() / rms)


def nmse(x, ref):
    """sum (x - ref)^2 / sum ref^2 (the normalised mean squared error)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sum(ref ** 2)
    return float(np.sum((x - ref) ** 2) / den) if den > 0 else float(np.sum((x - ref) ** 2))


def record(name, quantity, x, ref, out_dtype=None):
    """Measure x against ref (raw, allowance-adjusted, NMSE), keep the record, return the
    allowance-adjusted error."""
    raw = rel_err(x, ref)
    adj = rel_err(x, ref, out_dtype) if out_dtype else raw
    RECORDS.append((name, quantity, raw, adj, nmse(x, ref)))
    return adj


def to_np(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy().astype(np.float64)


def oracle_heads(x, heads, seqs=None, op="gdn", head_map="grouped"):
    """fp64 oracle for v heads ``heads`` (and sequences ``seqs``) of inputs ``x``.

    Slices each chain's own q/k head (GQA map ``head_map``) and v head so the oracle
    touches only what it checks.  Returns {(n, hv): (o [L, dv], hT [dk, dv])}.
    """
    q, k, v, g, beta, h0, cu = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                x["cu_seqlens"])
    B, T, Hqk, _ = q.shape
    Hv = v.shape[2]
    if cu is None:
        spans = [(b, b, 0, T) for b in range(B)]
    else:
        c = cu.cpu().numpy()
        spans = [(n, 0, int(c[n]), int(c[n + 1])) for n in range(len(c) - 1)]
    if seqs is not None:
        spans = [spans[i] for i in seqs]
    out = {}
    for n, b, t0, t1 in spans:
        for hv in heads:
            hq = qk_head(hv, Hqk, Hv, head_map)
            sl = slice(t0, t1)
            h0n = None if h0 is None else to_np(h0[n:n + 1, hv:hv + 1])
            fwd = {"gdn": gdn_recurrent, "ssd": ssd_recurrent, "kda": kda_recurrent}[op]
            o, hT = fwd(to_np(q[b:b + 1, sl, hq:hq + 1]), to_np(k[b:b + 1, sl, hq:hq + 1]),
                        to_np(v[b:b + 1, sl, hv:hv + 1]), to_np(g[b:b + 1, sl, hv:hv + 1]),
                        to_np(beta[b:b + 1, sl, hv:hv + 1]), x["scale"], h0n)
            out[(n, hv)] = (o[0, :, 0], hT[0, 0])
    return out


def check_heads(x, o, hT, heads, dtype, seqs=None, tol=None, op="gdn", head_map="grouped",
                name=None):
    """Compare the kernel's o / hT with the oracle (``op`` "gdn", "ssd" or "kda") on the chosen
    chains; records raw max-abs/RMS, the allowance-adjusted error and the NMSE of each, asserts
    the adjusted errors are within the tolerance and returns them."""
    tol = TOL[dtype] if tol is None else tol
    ref = oracle_heads(x, heads, seqs, op, head_map)
    cu = x["cu_seqlens"]
    B, T = x["q"].shape[:2]
    if cu is not None:
        cu = cu.cpu().numpy()
    spans = ([(b, b, 0, T) for b in range(B)] if cu is None else
             [(n, 0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)])
    worst_o = worst_h = 0.0
    o_parts, or_parts, h_parts, hr_parts = [], [], [], []
    for (n, hv), (o_ref, h_ref) in ref.items():
        _, b, t0, t1 = spans[n]
        o_parts.append(to_np(o[b, t0:t1, hv]))
        or_parts.append(o_ref)
        if hT is not None:
            h_parts.append(to_np(hT[n, hv]))
            hr_parts.append(h_ref)
    name = name or _current_test()
    if o_parts:
        worst_o = record(name, "o", np.concatenate([p.ravel() for p in o_parts]),
                         np.concatenate([p.ravel() for p in or_parts]), out_dtype=dtype)
    if h_parts:
        worst_h = record(name, "hT", np.concatenate([p.ravel() for p in h_parts]),
                         np.concatenate([p.ravel() for p in hr_parts]))
    assert worst_o <= tol, f"o error {worst_o:.3e} > {tol}"
    assert worst_h <= tol, f"hT error {worst_h:.3e} > {tol}"
    return worst_o, worst_h


def _current_test():
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
