"""Python binding of libgdn.so: argument marshalling only.

The functions carry the C ABI's names.  They take torch tensors (device memory
and streams are torch's), check dtypes, devices, shapes and contiguity, pass
raw pointers and sizes to the library and turn a non-OK status into an
exception.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind: without libgdn.so every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT = range(5)
# flags of gdn_chunk_fwd_ex / gdn_recurrent_step_ex (include/gdn.h)
GDN_FLAG_HEAD_MAP_MODULO, GDN_FLAG_CHECK_INPUTS, GDN_FLAG_TC_CHAIN = 1, 2, 4
GDN_FLAG_DV_TILE_CHAIN = 8

# name -> (restype, argtypes) of every symbol include/gdn.h declares
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_FWD_ARGS = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P]
_STEP_ARGS = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]
_SZ = ctypes.c_size_t
_U = ctypes.c_uint
SIGNATURES = {
    "gdn_chunk_fwd": (_I, _FWD_ARGS),
    "gdn_chunk_fwd_ex": (_I, _FWD_ARGS[:-1] + [_U, _P, _SZ, _P]),
    "gdn_chunk_fwd_noalloc": (_I, _FWD_ARGS),
    "gdn_chunk_fwd_workspace_size": (_SZ, [_I] * 8),
    "gdn_chunk_fwd_f32": (_I, _FWD_ARGS),
    "gdn_recurrent_step": (_I, _STEP_ARGS),
    "gdn_recurrent_step_ex": (_I, _STEP_ARGS[:-1] + [_U, _P]),
    "gdn_recurrent_step_f32": (_I, _STEP_ARGS),
    "gdn_chunk_fwd_prologue": (_I, _FWD_ARGS[:5] + [_P, _P] + _FWD_ARGS[5:]),
    "gdn_chunk_fwd_prologue_ex": (_I, _FWD_ARGS[:5] + [_P, _P] + _FWD_ARGS[5:-1] + [_U, _P, _SZ, _P]),
    "gdn_recurrent_step_prologue": (_I, _STEP_ARGS[:5] + [_P, _P] + _STEP_ARGS[5:]),
    "ssd_chunk_fwd": (_I, _FWD_ARGS),
    "ssd_chunk_fwd_ex": (_I, _FWD_ARGS[:-1] + [_U, _P, _SZ, _P]),
    "ssd_chunk_fwd_f32": (_I, _FWD_ARGS),
    "ssd_recurrent_step": (_I, _STEP_ARGS),
    "ssd_recurrent_step_f32": (_I, _STEP_ARGS),
    "kda_chunk_fwd": (_I, _FWD_ARGS),
    "kda_chunk_fwd_ex": (_I, _FWD_ARGS[:-1] + [_U, _P, _SZ, _P]),
    "kda_chunk_fwd_workspace_size": (_SZ, [_I] * 8),
    "kda_recurrent_step": (_I, _STEP_ARGS),
    "gdn_device_status": (_I, [_P]),
    "gdn_selftest_expired_wait": (_I, [ctypes.c_longlong, _P]),
    "gdn_status_string": (ctypes.c_char_p, [_I]),
    "gdn_last_error": (ctypes.c_char_p, []),
    "gdn_abi_version": (_I, []),
    "gdn_chunk_fwd_chain_kind": (_I, [_I, _I, _I, _I, _I, _U]),
}

_lib = None
_lock = threading.Lock()


class GdnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgdn.so not found at {path}: build it first "
                    "(python -m linear_attention_prefill_gb300._build)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().gdn_status_string(status).decode()


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, load_library().gdn_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, name, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, chunk=64, varlen=False) -> int:
    """Bytes of workspace the bf16 forward needs (0 for rejected sizes)."""
    return int(load_library().gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, chunk,
                                                           int(bool(varlen))))


def chain_kind(n_seqs, Hv, dk, dv, op="gdn", tc_chain=None) -> str:
    """The chunk-serial kernel a bf16 forward of ``op`` ("gdn", "gdn_prologue", "ssd" or
    "kda") runs for n_seqs sequences of Hv v heads: "tc" (tensor-memory chain) or
    "dv_tile"."""
    if op == "kda":
        return "dv_tile"
    k = load_library().gdn_chunk_fwd_chain_kind(n_seqs, Hv, dk, dv, int(op != "ssd"),
                                                _flags(tc_chain=tc_chain))
    if k < 0:
        raise ValueError(f"no chain for n_seqs={n_seqs}, Hv={Hv}, dk={dk}, dv={dv}")
    return "tc" if k == 1 else "dv_tile"


def gdn_chunk_fwd(q, k, v, g, beta, h0=None, o=None, hT=None, *, chunk: int = 64,
                  scale: Optional[float] = None, cu_seqlens=None, output_final_state=True,
                  stream=None, workspace=None, head_map: str = "grouped",
                  check_inputs: bool = False, tc_chain: Optional[bool] = None):
    """Chunked-prefill forward of the gated delta rule; returns (o, hT).

    q, k [B, T, Hqk, dk]; v [B, T, Hv, dv] (bf16 or fp32, all the same);
    g, beta [B, T, Hv] fp32; h0 [N, Hv, dk, dv] fp32 or None.  With
    cu_seqlens (int32 [N+1] on the device) the batch is one packed row, B = 1.
    o and hT may be passed preallocated; hT may be h0 (in place).  The bf16
    path runs gdn_chunk_fwd_ex with ``workspace`` (a uint8 device tensor of at
    least gdn_chunk_fwd_workspace_size bytes) or a fresh one from torch's
    caching allocator, and the flags: ``head_map`` "grouped" (hv // (Hv // Hqk))
    or "modulo" (hv % Hqk), ``check_inputs`` (a device pass over g, beta and
    cu_seqlens, reported by gdn_device_status), ``tc_chain`` (None: the library
    picks the chain kind from the number of chains; True: the chunk-serial
    operators on tcgen05, one CTA per chain; False: the dv-tile chain).
    ``scale`` defaults to dk^-0.5.
    """
    flags = _flags(head_map, check_inputs, tc_chain)
    if flags and q.dtype != torch.bfloat16:
        raise TypeError("head_map, check_inputs and tc_chain apply to the bf16 forward")
    return _chunk_fwd("gdn", q, k, v, g, beta, h0, o, hT, chunk,
                      k.shape[-1] ** -0.5 if scale is None else scale, cu_seqlens,
                      output_final_state, stream, workspace, flags=flags)


def _flags(head_map="grouped", check_inputs=False, tc_chain=None) -> int:
    """The _ex flag word; ``tc_chain`` None lets the library pick the chain kind, True
    forces the tensor-memory chain, False the dv-tile chain."""
    if head_map not in ("grouped", "modulo"):
        raise ValueError(f"head_map must be 'grouped' or 'modulo', got {head_map!r}")
    if tc_chain not in (None, True, False):
        raise ValueError(f"tc_chain must be None, True or False, got {tc_chain!r}")
    return ((GDN_FLAG_HEAD_MAP_MODULO if head_map == "modulo" else 0)
            | (GDN_FLAG_CHECK_INPUTS if check_inputs else 0)
            | (0 if tc_chain is None else GDN_FLAG_TC_CHAIN if tc_chain else GDN_FLAG_DV_TILE_CHAIN))


def gdn_chunk_fwd_prologue(q, k, v, a, b, A_log=None, dt_bias=None, h0=None, o=None, hT=None, *,
                           chunk: int = 64, scale: Optional[float] = None, cu_seqlens=None,
                           output_final_state=True, stream=None, workspace=None,
                           head_map: str = "grouped", check_inputs: bool = False,
                           tc_chain: Optional[bool] = None):
    """gdn_chunk_fwd with the fused prologue (bf16): q, k unnormalised; raw gates a, b
    [B, T, Hv] fp32; A_log, dt_bias [Hv] fp32 or None.  g = -exp(A_log) softplus(a +
    dt_bias), beta = sigmoid(b), q and k divided by sqrt(sum x^2 + 1e-6).  Returns (o, hT)."""
    dev = q.device
    Hv = v.shape[2]
    for t, name in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if t is not None:
            _need(t, name, torch.float32, dev, (Hv,))
    return _chunk_fwd("gdn", q, k, v, a, b, h0, o, hT, chunk,
                      k.shape[-1] ** -0.5 if scale is None else scale, cu_seqlens,
                      output_final_state, stream, workspace, prologue=(A_log, dt_bias),
                      flags=_flags(head_map, check_inputs, tc_chain))


def ssd_chunk_fwd(q, k, v, g, beta, h0=None, o=None, hT=None, *, chunk: int = 64,
                  scale: float = 1.0, cu_seqlens=None, output_final_state=True, stream=None,
                  workspace=None, head_map: str = "grouped", check_inputs: bool = False,
                  tc_chain: Optional[bool] = None):
    """Chunked Mamba-2 SSD scan (the same recurrence without the erase term):
    S_t = exp(g_t) S_{t-1} + beta_t v_t k_t^T, o_t = S_t (scale q_t), with
    C -> q, B -> k, x -> v, dt A -> g, dt -> beta.  Arguments as gdn_chunk_fwd;
    ``scale`` defaults to 1.  Returns (o, hT)."""
    flags = _flags(head_map, check_inputs, tc_chain)
    if flags and q.dtype != torch.bfloat16:
        raise TypeError("head_map, check_inputs and tc_chain apply to the bf16 forward")
    return _chunk_fwd("ssd", q, k, v, g, beta, h0, o, hT, chunk, scale, cu_seqlens,
                      output_final_state, stream, workspace, flags=flags)


def kda_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, chunk=64, varlen=False) -> int:
    """Bytes of workspace the KDA forward needs (0 for rejected sizes)."""
    return int(load_library().kda_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, chunk,
                                                           int(bool(varlen))))


def kda_chunk_fwd(q, k, v, g, beta, h0=None, o=None, hT=None, *, chunk: int = 64,
                  scale: Optional[float] = None, cu_seqlens=None, output_final_state=True,
                  stream=None, workspace=None, head_map: str = "grouped",
                  check_inputs: bool = False):
    """Chunked-prefill forward of Kimi Delta Attention (bf16, dk = 128); returns (o, hT).

    h_t = (I - beta_t k_t k_t^T) diag(exp g_t) h_{t-1} + beta_t k_t v_t^T,
    o_t = h_t^T (scale q_t).  As gdn_chunk_fwd, except g is [B, T, Hv, dk] fp32:
    one log-decay per key channel.  Runs kda_chunk_fwd_ex with ``workspace`` or a
    fresh one.  ``scale`` defaults to dk^-0.5.
    """
    return _chunk_fwd("kda", q, k, v, g, beta, h0, o, hT, chunk,
                      k.shape[-1] ** -0.5 if scale is None else scale, cu_seqlens,
                      output_final_state, stream, workspace,
                      flags=_flags(head_map, check_inputs))


def _chunk_fwd(op, q, k, v, g, beta, h0, o, hT, chunk, scale, cu_seqlens, output_final_state,
               stream, workspace, prologue=None, flags=0):
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdn_chunk_fwd runs on a CUDA device")
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q, k, v must be bf16 or fp32")
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    _need(q, "q", dt, dev)
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev, (B, T, Hv, dv))
    _need(g, "g", torch.float32, dev, (B, T, Hv, dk) if op == "kda" else (B, T, Hv))
    _need(beta, "beta", torch.float32, dev, (B, T, Hv))
    if op == "kda" and dt != torch.bfloat16:
        raise TypeError("the KDA forward takes bf16 q, k, v")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if B != 1:
            raise ValueError("with cu_seqlens the batch must be one packed row (B == 1)")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev, (N, Hv, dk, dv))
    if o is None:
        o = torch.empty((B, T, Hv, dv), dtype=dt, device=dev)
    _need(o, "o", dt, dev, (B, T, Hv, dv))
    if hT is None and output_final_state:
        hT = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=dev)
    if hT is not None:
        _need(hT, "hT", torch.float32, dev, (N, Hv, dk, dv))
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
            N, T, Hqk, Hv, dk, dv, chunk, float(scale), _ptr(cu_seqlens))
    if prologue is not None:
        if dt != torch.bfloat16:
            raise TypeError("the fused prologue takes bf16 q, k, v")
        args = args[:5] + (_ptr(prologue[0]), _ptr(prologue[1])) + args[5:]
        need = gdn_chunk_fwd_workspace_size(N, T, Hqk, Hv, dk, dv, chunk, cu_seqlens is not None)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
        _check(lib.gdn_chunk_fwd_prologue_ex(*args, int(flags), _ptr(workspace),
                                             workspace.numel(), _stream_handle(stream, dev)))
        return o, hT
    if dt == torch.float32:
        _check(getattr(lib, f"{op}_chunk_fwd_f32")(*args, _stream_handle(stream, dev)))
        return o, hT
    size_fn = kda_chunk_fwd_workspace_size if op == "kda" else gdn_chunk_fwd_workspace_size
    need = size_fn(N, T, Hqk, Hv, dk, dv, chunk, cu_seqlens is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    _check(getattr(lib, f"{op}_chunk_fwd_ex")(*args, int(flags), _ptr(workspace),
                                              workspace.numel(), _stream_handle(stream, dev)))
    return o, hT


def gdn_recurrent_step(q, k, v, g, beta, h, o=None, *, scale: Optional[float] = None,
                       stream=None, head_map: str = "grouped", check_inputs: bool = False):
    """One decode token of the gated delta rule; updates h in place and returns o.

    q, k [N, Hqk, dk]; v [N, Hv, dv]; g, beta [N, Hv] fp32; h [N, Hv, dk, dv] fp32.
    ``head_map`` and ``check_inputs`` as in gdn_chunk_fwd (bf16: gdn_recurrent_step_ex).
    """
    flags = _flags(head_map, check_inputs)
    if flags and q.dtype != torch.bfloat16:
        raise TypeError("head_map and check_inputs apply to the bf16 step")
    return _step("gdn", q, k, v, g, beta, h, o, k.shape[-1] ** -0.5 if scale is None else scale,
                 stream, flags=flags)


def gdn_recurrent_step_prologue(q, k, v, a, b, h, A_log=None, dt_bias=None, o=None, *,
                                scale: Optional[float] = None, stream=None):
    """One decode token with the fused prologue (bf16; see gdn_chunk_fwd_prologue)."""
    return _step("gdn", q, k, v, a, b, h, o, k.shape[-1] ** -0.5 if scale is None else scale,
                 stream, prologue=(A_log, dt_bias))


def ssd_recurrent_step(q, k, v, g, beta, h, o=None, *, scale: float = 1.0, stream=None):
    """One decode token of the Mamba-2 SSD recurrence; updates h in place, returns o."""
    return _step("ssd", q, k, v, g, beta, h, o, scale, stream)


def kda_recurrent_step(q, k, v, g, beta, h, o=None, *, scale: Optional[float] = None,
                       stream=None):
    """One decode token of Kimi Delta Attention (g [N, Hv, dk]); updates h, returns o."""
    if q.dtype != torch.bfloat16:
        raise TypeError("the KDA decode step takes bf16 q, k, v")
    return _step("kda", q, k, v, g, beta, h, o, k.shape[-1] ** -0.5 if scale is None else scale,
                 stream)


def _step(op, q, k, v, g, beta, h, o, scale, stream, prologue=None, flags=0):
    lib = load_library()
    dev = q.device
    dt = q.dtype
    N, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    _need(q, "q", dt, dev)
    _need(k, "k", dt, dev, q.shape)
    _need(v, "v", dt, dev, (N, Hv, dv))
    _need(g, "g", torch.float32, dev, (N, Hv, dk) if op == "kda" else (N, Hv))
    _need(beta, "beta", torch.float32, dev, (N, Hv))
    _need(h, "h", torch.float32, dev, (N, Hv, dk, dv))
    if o is None:
        o = torch.empty((N, Hv, dv), dtype=dt, device=dev)
    _need(o, "o", dt, dev, (N, Hv, dv))
    if prologue is not None:
        if dt != torch.bfloat16:
            raise TypeError("the fused prologue takes bf16 q, k, v")
        for t, name in zip(prologue, ("A_log", "dt_bias")):
            if t is not None:
                _need(t, name, torch.float32, dev, (Hv,))
        _check(lib.gdn_recurrent_step_prologue(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(prologue[0]), _ptr(prologue[1]),
            _ptr(h), _ptr(o), N, Hqk, Hv, dk, dv, float(scale), _stream_handle(stream, dev)))
        return o
    if flags:
        _check(lib.gdn_recurrent_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h),
                                         _ptr(o), N, Hqk, Hv, dk, dv, float(scale), int(flags),
                                         _stream_handle(stream, dev)))
        return o
    fn = getattr(lib, f"{op}_recurrent_step" + ("" if dt == torch.bfloat16 else "_f32"))
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h), _ptr(o), N, Hqk, Hv,
              dk, dv, float(scale), _stream_handle(stream, dev)))
    return o


def gdn_selftest_expired_wait(limit_cycles: int = 1 << 20, stream=None):
    """Enqueue the timeout-path diagnostic (a bounded wait that is bound to expire)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load_library().gdn_selftest_expired_wait(int(limit_cycles), _stream_handle(stream, dev)))


def gdn_device_status(stream=None):
    """Raise GdnError for what the kernels recorded since the last check: a bounded
    device-side wait that gave up (GDN_ERR_TIMEOUT); a KDA log-decay below -10, an fp16
    operand out of range, or an input-check violation (GDN_ERR_INVALID_ARG)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load_library().gdn_device_status(_stream_handle(stream, dev)))


def gdn_chunk_fwd_host(inputs: dict, chunk: int = 64, device="cuda", stream=None, out=None,
                       op: str = "gdn", **fwd_kw):
    """End-to-end call from pinned host memory: copy inputs in, run, copy o and hT out
    (``op`` "ssd" runs ssd_chunk_fwd, "kda" kda_chunk_fwd, "gdn_prologue"
    gdn_chunk_fwd_prologue on raw q, k and gate inputs instead).

    ``inputs`` holds pinned CPU tensors q, k, v, g, beta and optionally h0 and
    cu_seqlens.  ``out`` may hold preallocated pinned (o, hT) host tensors and
    device buffers to reuse; ``fwd_kw`` (scale, tc_chain, ...) passes on to the forward.
    Returns (o_host, hT_host, bytes_in, bytes_out).
    """
    dev = torch.device(device)
    bufs = out.setdefault("dev", {}) if out is not None else {}
    d = {}
    nbytes_in = 0
    for name in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
        t = inputs.get(name)
        if t is None:
            d[name] = None
            continue
        buf = bufs.get(name)
        if buf is None or buf.shape != t.shape or buf.dtype != t.dtype:
            buf = bufs[name] = torch.empty(t.shape, dtype=t.dtype, device=dev)
        buf.copy_(t, non_blocking=True)
        d[name] = buf
        nbytes_in += t.numel() * t.element_size()
    fwd = {"ssd": ssd_chunk_fwd, "kda": kda_chunk_fwd,
           "gdn_prologue": lambda q, k, v, a, b, h0, o, hT, **kw: gdn_chunk_fwd_prologue(
               q, k, v, a, b, None, None, h0, o, hT, **kw)}.get(op, gdn_chunk_fwd)
    if "workspace" not in bufs:
        B, T, Hqk, dk = d["q"].shape
        Hv, dv = d["v"].shape[2], d["v"].shape[3]
        N = d["cu_seqlens"].numel() - 1 if d["cu_seqlens"] is not None else B
        size_fn = kda_chunk_fwd_workspace_size if op == "kda" else gdn_chunk_fwd_workspace_size
        need = size_fn(N, T, Hqk, Hv, dk, dv, chunk, d["cu_seqlens"] is not None)
        bufs["workspace"] = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    o_dev, hT_dev = fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], bufs.get("o"),
                        bufs.get("hT"), chunk=chunk, cu_seqlens=d["cu_seqlens"], stream=stream,
                        workspace=bufs["workspace"], **fwd_kw)
    bufs["o"], bufs["hT"] = o_dev, hT_dev
    if out is not None and "o_host" in out:
        o_h, hT_h = out["o_host"], out["hT_host"]
    else:
        o_h = torch.empty(o_dev.shape, dtype=o_dev.dtype, pin_memory=True)
        hT_h = torch.empty(hT_dev.shape, dtype=hT_dev.dtype, pin_memory=True)
        if out is not None:
            out["o_host"], out["hT_host"] = o_h, hT_h
    o_h.copy_(o_dev, non_blocking=True)
    hT_h.copy_(hT_dev, non_blocking=True)
    nbytes_out = o_h.numel() * o_h.element_size() + hT_h.numel() * hT_h.element_size()
    return o_h, hT_h, nbytes_in, nbytes_out


class HostPipeline:
    """Forward calls streamed from pinned host memory, copies overlapped across calls.

    Each call copies its inputs host -> device, runs the forward and copies o and
    hT device -> host, all on one of ``depth`` streams with its own device buffers,
    workspace and pinned outputs; consecutive calls go to different streams, so the
    upload of call i + 1 overlaps the compute and the download of call i (the host
    link carries one direction of each at once).  ``submit`` returns the pinned
    (o, hT) of that call and a CUDA event that completes when they are filled.
    ``fwd_kw`` (scale, tc_chain, ...) passes on to every forward call.
    """

    def __init__(self, chunk: int = 64, device="cuda", op: str = "gdn", depth: int = 2,
                 **fwd_kw):
        self.dev = torch.device(device)
        self.chunk, self.op, self.fwd_kw = chunk, op, fwd_kw
        self.slots = [dict(stream=torch.cuda.Stream(self.dev), bufs={}) for _ in range(depth)]
        self.n = 0

    def submit(self, inputs: dict):
        slot = self.slots[self.n % len(self.slots)]
        self.n += 1
        bufs = slot["bufs"]
        with torch.cuda.stream(slot["stream"]):
            o_h, hT_h, nbytes_in, nbytes_out = gdn_chunk_fwd_host(
                inputs, chunk=self.chunk, device=self.dev, stream=slot["stream"], out=bufs,
                op=self.op, **self.fwd_kw)
            done = torch.cuda.Event()
            done.record(slot["stream"])
        return o_h, hT_h, done, nbytes_in, nbytes_out
