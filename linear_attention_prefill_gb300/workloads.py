"""Seeded synthetic workloads for the Gated DeltaNet chunked-prefill forward.

This module only draws inputs.  It holds none of the method's arithmetic, so the
CUDA path and the fp64 oracle can both take their inputs from here without
sharing any computation.

Input recipe (the kernel sweep of "Empowering Hybrid Attention Models on NPUs",
§7.1 setup: chunk 64, FP16/bf16 Q/K/V with FP32 gates and states; head counts
16/32 of Figure 13; sequences up to 64K tokens of Figure 16; a 128x128 fp32
state per head, §5 "adding a 64-KiB state"):

* q, k ~ N(0, 1), then L2-normalised along the head dimension in fp32 and
  rounded once to the input dtype (the kernel and the oracle both see the
  rounded values);
* v ~ N(0, 1) rounded to the input dtype;
* beta = sigmoid(N(0, 1)) in fp32 (already squashed: the kernel takes beta);
* g = -softplus(N(mu, 1)) * s in fp32 (a log-decay <= 0; mu and s per workload);
  for Kimi Delta Attention (op "kda") one such draw per key channel, g [B, T, Hv, dk];
* h0 ~ N(0, sigma) in fp32 where a workload carries state, else absent.

All draws come from one ``torch.Generator`` seeded per workload, on the device
the tensors are made on.  Draws on CPU and on CUDA differ; every test takes the
oracle's inputs from the very tensors it passes to the kernel.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic problem: shapes, dtype, distributions, seed."""

    name: str
    seqlens: tuple          # lengths of the sequences; more than one => packed varlen
    Hqk: int
    Hv: int
    dk: int
    dv: int
    chunk: int
    dtype: str              # "bf16" or "f32": dtype of q, k, v and o
    g_mu: float = 0.0       # g = -softplus(N(g_mu, 1)) * g_scale
    g_scale: float = 1.0
    h0_std: Optional[float] = None   # None: no initial state (zeros)
    op: str = "gdn"                  # "gdn" (gated delta rule), "ssd" (Mamba-2 scan) or
                                     # "kda" (delta rule with a per-channel gate)
    varlen: bool = False    # True: one packed [1, T_total, ...] batch with cu_seqlens
    seed: int = 0
    decode_steps: int = 0   # one-token steps that continue from the final state
    prologue: bool = False  # raw inputs for the fused prologue (see make_inputs)

    @property
    def T_total(self) -> int:
        return int(sum(self.seqlens))

    @property
    def n_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def scale(self) -> float:
        return 1.0 if self.op == "ssd" else float(self.dk) ** -0.5

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


# The five workloads the measurements are quoted on.
WORKLOADS = {
    # tiny fp32 case that the oracle finishes in well under a second
    "tiny_f32": Workload("tiny_f32", (256,), 2, 2, 64, 64, 64, "f32", seed=1),
    # one GDN layer of a 0.8B-class hybrid model: 16 heads of 128, 4K prompt
    "layer_16h_4k": Workload("layer_16h_4k", (4096,), 16, 16, 128, 128, 64, "bf16", seed=2),
    # GQA: each qk head shared by two v heads; carried initial state, final state returned
    "gqa_32v_8k_state": Workload("gqa_32v_8k_state", (8192,), 16, 32, 128, 128, 64, "bf16",
                                 h0_std=0.1, seed=3),
    # 8 packed sequences of 512..2048 tokens with per-sequence initial state
    "varlen_8seq": Workload("varlen_8seq", _varlen_lengths(8, 512, 2048, 4), 16, 32, 128, 128, 64,
                            "bf16", g_mu=0.5, h0_std=0.1, varlen=True, seed=4),
    # long context, strong decay (weak-decay and chunk-128 variants below)
    "long_64k_strong": Workload("long_64k_strong", (65536,), 32, 32, 128, 128, 64, "bf16",
                                g_mu=1.0, seed=5, decode_steps=1000),
}
WORKLOADS["long_64k_weak"] = WORKLOADS["long_64k_strong"].replace(
    name="long_64k_weak", g_mu=0.0, g_scale=0.01)
WORKLOADS["long_64k_strong_c128"] = WORKLOADS["long_64k_strong"].replace(
    name="long_64k_strong_c128", chunk=128)
WORKLOADS["long_64k_weak_c128"] = WORKLOADS["long_64k_weak"].replace(
    name="long_64k_weak_c128", chunk=128)

# Mamba-2 SSD scan of a 2.7B-class model ("Exp 2026-07-13 — Linear-Attention Scans on the
# NPU", §3: head_dim 64, d_state 128, chunks of 64; 80 heads sharing one B/C group), 4K prompt.
# The headline layer fed raw: unnormalised q, k and the gate inputs a, b of the fused
# prologue (g = -softplus(a), beta = sigmoid(b): the same distributions as the headline).
WORKLOADS["layer_16h_4k_prologue"] = WORKLOADS["layer_16h_4k"].replace(
    name="layer_16h_4k_prologue", prologue=True)

WORKLOADS["ssd_80h_4k"] = Workload("ssd_80h_4k", (4096,), 1, 80, 128, 64, 64, "bf16", seed=6,
                                   op="ssd")

# Kimi Delta Attention layer (the pages' KDA kernels at 16 heads, Figure 13; head dim 128 and
# the per-channel fp32 gate of Figure 4), 4K prompt.
WORKLOADS["kda_16h_4k"] = Workload("kda_16h_4k", (4096,), 16, 16, 128, 128, 64, "bf16", seed=7,
                                   op="kda")

# The workload the headline throughput is quoted on.
HEADLINE = "layer_16h_4k"


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def cu_seqlens_of(seqlens) -> np.ndarray:
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return cu


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw one batch of inputs for workload ``w`` on ``device``.

    Returns a dict with q, k ([B, T, Hqk, dk]), v ([B, T, Hv, dv]), g ([B, T, Hv]
    fp32, or [B, T, Hv, dk] for KDA), beta ([B, T, Hv] fp32) - for a prologue workload
    q, k unnormalised and g, beta the raw gate inputs a, b - h0 ([N, Hv, dk, dv] fp32 or None), cu_seqlens (int32
    [N+1] on ``device`` for varlen workloads, else None), and the sizes
    B, T, N, scale.  A varlen batch is one packed row: B = N sequences,
    tensors [1, T_total, ...].
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    if w.varlen:
        B, T = 1, w.T_total
    else:
        assert len(set(w.seqlens)) == 1, "fixed-length batch needs equal lengths"
        B, T = w.n_seqs, w.seqlens[0]
    N = w.n_seqs

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    if w.prologue:  # raw rows: N(0, 1) times a per-row factor exp(N(0, 1))
        q = (randn(B, T, w.Hqk, w.dk) * torch.exp(randn(B, T, w.Hqk, 1))).to(dt)
        k = (randn(B, T, w.Hqk, w.dk) * torch.exp(randn(B, T, w.Hqk, 1))).to(dt)
    else:
        q = _unit_rows(randn(B, T, w.Hqk, w.dk)).to(dt)
        k = _unit_rows(randn(B, T, w.Hqk, w.dk)).to(dt)
    v = randn(B, T, w.Hv, w.dv).to(dt)
    if w.prologue:  # the raw gate inputs a (in g) and b (in beta)
        beta = randn(B, T, w.Hv)
        g = randn(B, T, w.Hv) + w.g_mu
    elif w.op == "ssd":
        # dt = softplus(N(0, 1)) is the input step (beta); g = dt * A with A = -exp(N(0, 0.3))
        # per head
        beta = torch.nn.functional.softplus(randn(B, T, w.Hv))
        g = -beta * torch.exp(0.3 * randn(w.Hv))
    elif w.op == "kda":
        beta = torch.sigmoid(randn(B, T, w.Hv))
        g = -torch.nn.functional.softplus(randn(B, T, w.Hv, w.dk) + w.g_mu) * w.g_scale
    else:
        beta = torch.sigmoid(randn(B, T, w.Hv))
        g = -torch.nn.functional.softplus(randn(B, T, w.Hv) + w.g_mu) * w.g_scale
    h0 = None
    if w.h0_std is not None:
        h0 = randn(N, w.Hv, w.dk, w.dv) * w.h0_std
    cu = None
    if w.varlen:
        cu = torch.from_numpy(cu_seqlens_of(w.seqlens)).to(device)
    return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), h0=h0,
                cu_seqlens=cu, B=w.n_seqs if w.varlen else B, T=T, N=N, scale=w.scale)


def make_decode_inputs(w: Workload, step: int, device="cpu") -> dict:
    """One decode token per sequence, same distributions, seeded by (seed, step)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1_000_003 + 7919 * (step + 1))
    dt = torch_dtype(w.dtype)
    N = w.n_seqs

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    q = _unit_rows(randn(N, w.Hqk, w.dk)).to(dt)
    k = _unit_rows(randn(N, w.Hqk, w.dk)).to(dt)
    v = randn(N, w.Hv, w.dv).to(dt)
    if w.op == "ssd":
        beta = torch.nn.functional.softplus(randn(N, w.Hv))
        g = -beta * torch.exp(0.3 * randn(w.Hv))
    elif w.op == "kda":
        beta = torch.sigmoid(randn(N, w.Hv))
        g = -torch.nn.functional.softplus(randn(N, w.Hv, w.dk) + w.g_mu) * w.g_scale
    else:
        beta = torch.sigmoid(randn(N, w.Hv))
        g = -torch.nn.functional.softplus(randn(N, w.Hv) + w.g_mu) * w.g_scale
    return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), N=N, scale=w.scale)
