"""Gated DeltaNet forward on one GB300: Python binding of libgdn's C ABI.

Three entry points, same names as the C ABI (``include/gdn.h``):

* ``gdn_gating(A_log, a, b, dt_bias) -> (g, beta)``
* ``gdn_chunk_fwd(q, k, v, g, beta, ...) -> (o, final_state)``
* ``gdn_recurrent_decode(q, k, v, ..., ssm_pool, ssm_indices) -> o``

This module only marshals arguments: it checks devices, dtypes and
contiguity, allocates outputs with ``torch.empty`` and passes raw pointers and
the current CUDA stream to the shared library.  Every step of the computation
runs in libgdn's CUDA kernels; if the library is missing the calls raise, there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = ["gdn_gating", "gdn_chunk_fwd", "gdn_recurrent_decode", "chunk_fwd_workspace_size", "chunk_fwd_kernel_launches",
           "gdn_chunk_fwd_noalloc", "NOALLOC_SCRATCH_BYTES", "gdn_causal_conv1d_fwd",
           "gdn_causal_conv1d_update", "gdn_causal_conv1d_update_spec", "gdn_conv_decode_pack",
           "gdn_recurrent_decode_bf16",
           "gdn_recurrent_decode_mtp", "gdn_chunk_bwd", "chunk_bwd_workspace_size",
           "gdn_chunk_fwd_gated", "chunk_gated_delta_rule", "GDNError", "lib_path", "load_library", "status_string", "DEV_BAD_CU_SEQLENS",
           "DEV_BAD_SLOT", "DEV_WAIT_TIMEOUT", "DEV_DRAIN_TIMEOUT", "EXPORTED_SYMBOLS",
           "testing_force_wait_expiry"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libgdn.so")
_lib = None
_lock = threading.Lock()

GDN_OK, GDN_EINVAL, GDN_EUNSUPPORTED, GDN_ECUDA, GDN_EWORKSPACE, GDN_ESCRATCH_LIMIT = 0, 1, 2, 3, 4, 5
DEV_BAD_CU_SEQLENS, DEV_BAD_SLOT, DEV_WAIT_TIMEOUT, DEV_DRAIN_TIMEOUT = 1, 2, 4, 8

#: Every symbol include/gdn.h declares (checked by the tests).
EXPORTED_SYMBOLS = ("gdn_status_string", "gdn_version", "gdn_gating", "gdn_chunk_fwd_workspace_size",
                    "gdn_chunk_fwd_kernel_launches",
                    "gdn_chunk_fwd", "gdn_recurrent_decode", "gdn_chunk_fwd_noalloc",
                    "gdn_causal_conv1d_fwd", "gdn_causal_conv1d_update", "gdn_conv_decode_pack",
                    "gdn_recurrent_decode_bf16", "gdn_recurrent_decode_mtp", "gdn_chunk_bwd_workspace_size",
                    "gdn_chunk_bwd", "gdn_chunk_fwd_gated", "gdn_testing_force_wait_expiry",
                    "gdn_causal_conv1d_update_spec")

#: Size of the fixed scratch buffer behind gdn_chunk_fwd_noalloc (bytes).
NOALLOC_SCRATCH_BYTES = 32 << 20


class GDNError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {status_string(code)} (status {code})")
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libgdn.so (built by ``build.py``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libgdn.so not found at {_LIB_PATH}; build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.gdn_status_string.argtypes = [I]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = I
        lib.gdn_testing_force_wait_expiry.argtypes = [I]
        lib.gdn_testing_force_wait_expiry.restype = I
        lib.gdn_gating.argtypes = [P, P, P, P, I64, I, P, P, P]
        lib.gdn_gating.restype = I
        lib.gdn_chunk_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.gdn_chunk_fwd_workspace_size.restype = SZ
        lib.gdn_chunk_fwd_kernel_launches.argtypes = [I, I, I, I, I, I, I, I]
        lib.gdn_chunk_fwd_kernel_launches.restype = I
        lib.gdn_chunk_fwd.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, P, P, SZ, P, P]
        lib.gdn_chunk_fwd.restype = I
        lib.gdn_chunk_fwd_gated.argtypes = [P, P, P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, P, P, P,
                                            P, SZ, P, P]
        lib.gdn_chunk_fwd_gated.restype = I
        lib.gdn_recurrent_decode.argtypes = [P, P, P, P, P, P, P, P, P, F, I, P, I, P, I, I, I, I, I,
                                             P, P, P]
        lib.gdn_recurrent_decode.restype = I
        lib.gdn_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, P, P, P]
        lib.gdn_chunk_fwd_noalloc.restype = I
        lib.gdn_causal_conv1d_fwd.argtypes = [P, P, P, P, I, I, P, P, P, I, I, I64, I, I, P, P, P]
        lib.gdn_causal_conv1d_fwd.restype = I
        lib.gdn_causal_conv1d_update.argtypes = [P, P, I, I, P, P, P, I, I, I, I, P, P, P]
        lib.gdn_causal_conv1d_update.restype = I
        lib.gdn_causal_conv1d_update_spec.argtypes = [P, P, I, I, P, P, P, P, P, I, I, I, I, I, I, P, P, P]
        lib.gdn_causal_conv1d_update_spec.restype = I
        lib.gdn_conv_decode_pack.argtypes = [P, P, I, I, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P]
        lib.gdn_conv_decode_pack.restype = I
        lib.gdn_recurrent_decode_bf16.argtypes = [P, P, P, P, P, P, P, P, P, F, I, P, I, P, I, I, I, I, I,
                                                  P, P, P]
        lib.gdn_recurrent_decode_bf16.restype = I
        lib.gdn_recurrent_decode_mtp.argtypes = [P, P, P, P, P, P, P, P, P, F, I, P, I, P, I, I, P, P, I, P,
                                                 I, I, I, I, P, P, P]
        lib.gdn_recurrent_decode_mtp.restype = I
        lib.gdn_chunk_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.gdn_chunk_bwd_workspace_size.restype = SZ
        lib.gdn_chunk_bwd.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P,
                                      P, SZ, P, P]
        lib.gdn_chunk_bwd.restype = I
        _lib = lib
        return lib


def status_string(code: int) -> str:
    try:
        return load_library().gdn_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def testing_force_wait_expiry(on: bool) -> bool:
    """Testing hook of the C ABI (gdn_testing_force_wait_expiry): while on, the
    first bounded wait of every decode block and chunk-forward chain runs out
    and the kernels take their failure path.  Returns the previous setting."""
    return bool(load_library().gdn_testing_force_wait_expiry(1 if on else 0))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, dtype, device, ndim=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (the library does not copy)")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def _scale_arg(scale) -> float:
    return -1.0 if scale is None else float(scale)


def gdn_gating(A_log: torch.Tensor, a: torch.Tensor, b: torch.Tensor, dt_bias: torch.Tensor,
               g: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None):
    """g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b); fp32 [Ttok, HV].

    A_log, dt_bias: fp32 [HV]; a, b: bf16 [Ttok, HV].  ``g``/``beta`` may be
    passed to write into existing fp32 buffers."""
    dev = a.device
    HV = A_log.numel()
    _check(A_log, "A_log", torch.float32, dev)
    _check(dt_bias, "dt_bias", torch.float32, dev)
    _check(a, "a", torch.bfloat16, dev)
    _check(b, "b", torch.bfloat16, dev)
    if a.shape != b.shape or a.numel() % max(HV, 1) != 0 or a.shape[-1] != HV or dt_bias.numel() != HV:
        raise ValueError("gdn_gating: a, b must be [Ttok, HV] and A_log, dt_bias [HV]")
    Ttok = a.numel() // HV
    if g is None:
        g = torch.empty(a.shape, dtype=torch.float32, device=dev)
    if beta is None:
        beta = torch.empty(a.shape, dtype=torch.float32, device=dev)
    _check(g, "g", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    rc = load_library().gdn_gating(_ptr(A_log), _ptr(a), _ptr(b), _ptr(dt_bias), Ttok, HV,
                                   _ptr(g), _ptr(beta), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_gating", rc)
    return g, beta


def chunk_fwd_workspace_size(B, T, H, HV, K, V, N, varlen) -> int:
    return int(load_library().gdn_chunk_fwd_workspace_size(B, T, H, HV, K, V, N, int(bool(varlen))))


def chunk_fwd_kernel_launches(B, T, H, HV, K, V, N, varlen) -> int:
    """Kernels gdn_chunk_fwd launches for these sizes on the current device."""
    return int(load_library().gdn_chunk_fwd_kernel_launches(B, T, H, HV, K, V, N, int(bool(varlen))))


def _prefill_args(fn, q, k, v, initial_state, output_final_state, cu_seqlens, num_seqs, dev_status, o,
                  final_state, workspace):
    """Checks and output allocation shared by the prefill entry points."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, dev)
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise ValueError(f"{fn}: q, k must be [B,T,H,K] and v [B,T,HV,V]")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev, ndim=1)
        N = int(num_seqs) if num_seqs is not None else cu_seqlens.numel() - 1
    else:
        N = B
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, dev)
        if tuple(initial_state.shape) != (N, HV, K, V):
            raise ValueError(f"initial_state must be [N,HV,K,V] = {(N, HV, K, V)}")
    if o is None:
        o = torch.empty((B, T, HV, V), dtype=torch.bfloat16, device=dev)
    _check(o, "o", torch.bfloat16, dev)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, HV, K, V), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev)
    ws_bytes = chunk_fwd_workspace_size(B, T, H, HV, K, V, N, cu_seqlens is not None)
    if ws_bytes > 0 and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    return (B, T, H, K, HV, V, N), o, final_state, workspace


def gdn_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, scale: Optional[float] = None,
                  initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                  cu_seqlens: Optional[torch.Tensor] = None, use_qk_l2norm: bool = True,
                  num_seqs: Optional[int] = None, dev_status: Optional[torch.Tensor] = None,
                  o: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None
                  ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked prefill.  q, k bf16 [B,T,H,K]; v bf16 [B,T,HV,V]; g, beta fp32
    [B,T,HV]; initial_state fp32 [N,HV,K,V] or None; cu_seqlens int32 [N+1]
    (device) with B = 1, or None.  Returns (o bf16 [B,T,HV,V], final_state fp32
    [N,HV,K,V] or None).  ``num_seqs`` gives N for varlen input without a
    device-to-host read (default: cu_seqlens.numel() - 1, a host-side size)."""
    dims, o, final_state, workspace = _prefill_args("gdn_chunk_fwd", q, k, v, initial_state, output_final_state,
                                                    cu_seqlens, num_seqs, dev_status, o, final_state, workspace)
    B, T, H, K, HV, V, N = dims
    for t, n in ((g, "g"), (beta, "beta")):
        _check(t, n, torch.float32, q.device)
    if tuple(g.shape) != (B, T, HV) or tuple(beta.shape) != (B, T, HV):
        raise ValueError(f"gdn_chunk_fwd: g and beta must be [B,T,HV] = {(B, T, HV)}")
    rc = load_library().gdn_chunk_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _scale_arg(scale), _ptr(initial_state),
        _ptr(cu_seqlens), N, B, T, H, HV, K, V, int(bool(use_qk_l2norm)), _ptr(o),
        _ptr(final_state), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _ptr(dev_status), _stream(q.device))
    if rc != GDN_OK:
        raise GDNError("gdn_chunk_fwd", rc)
    return o, final_state


def gdn_chunk_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, A_log: torch.Tensor,
                        a: torch.Tensor, b: torch.Tensor, dt_bias: torch.Tensor, scale: Optional[float] = None,
                        initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                        cu_seqlens: Optional[torch.Tensor] = None, use_qk_l2norm: bool = True,
                        num_seqs: Optional[int] = None, return_gates: bool = False,
                        dev_status: Optional[torch.Tensor] = None, o: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Chunked prefill with the gating fused in: A_log, dt_bias fp32 [HV]; a, b
    bf16 [B,T,HV] (the raw gate projections).  Returns (o, final_state), or
    (o, final_state, g, beta) with ``return_gates`` (fp32 [B,T,HV], e.g. for
    the backward).  Other arguments as in ``gdn_chunk_fwd``."""
    dims, o, final_state, workspace = _prefill_args("gdn_chunk_fwd_gated", q, k, v, initial_state,
                                                    output_final_state, cu_seqlens, num_seqs, dev_status, o,
                                                    final_state, workspace)
    B, T, H, K, HV, V, N = dims
    dev = q.device
    for t, n, dt in ((A_log, "A_log", torch.float32), (dt_bias, "dt_bias", torch.float32),
                     (a, "a", torch.bfloat16), (b, "b", torch.bfloat16)):
        _check(t, n, dt, dev)
    if tuple(A_log.shape) != (HV,) or tuple(dt_bias.shape) != (HV,):
        raise ValueError(f"gdn_chunk_fwd_gated: A_log and dt_bias must be [HV] = {(HV,)}")
    if tuple(a.shape) != (B, T, HV) or tuple(b.shape) != (B, T, HV):
        raise ValueError(f"gdn_chunk_fwd_gated: a and b must be [B,T,HV] = {(B, T, HV)}")
    g_out = beta_out = None
    if return_gates:
        g_out = torch.zeros((B, T, HV), dtype=torch.float32, device=dev)
        beta_out = torch.zeros((B, T, HV), dtype=torch.float32, device=dev)
    rc = load_library().gdn_chunk_fwd_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(A_log), _ptr(a), _ptr(b), _ptr(dt_bias), _scale_arg(scale),
        _ptr(initial_state), _ptr(cu_seqlens), N, B, T, H, HV, K, V, int(bool(use_qk_l2norm)), _ptr(o),
        _ptr(final_state), _ptr(g_out), _ptr(beta_out), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_chunk_fwd_gated", rc)
    if return_gates:
        return o, final_state, g_out, beta_out
    return o, final_state


def gdn_chunk_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                          beta: torch.Tensor, scale: Optional[float] = None,
                          initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                          cu_seqlens: Optional[torch.Tensor] = None, use_qk_l2norm: bool = True,
                          num_seqs: Optional[int] = None, dev_status: Optional[torch.Tensor] = None,
                          o: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None
                          ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """gdn_chunk_fwd for callers that cannot allocate device memory at call time
    (for example a serving runtime whose device memory is all reserved by its own
    pool).  The library keeps the workspace in a fixed buffer of
    NOALLOC_SCRATCH_BYTES per GPU; larger inputs raise GDNError with
    GDN_ESCRATCH_LIMIT.  The C call allocates nothing; pass ``o`` and
    ``final_state`` to keep this wrapper from allocating its outputs either.
    Calls sharing a device must not overlap on the GPU."""
    dev = q.device
    for t, n_, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                      (g, "g", torch.float32), (beta, "beta", torch.float32)):
        _check(t, n_, dt, dev)
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise ValueError("gdn_chunk_fwd_noalloc: q, k must be [B,T,H,K] and v [B,T,HV,V]")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if tuple(g.shape) != (B, T, HV) or tuple(beta.shape) != (B, T, HV):
        raise ValueError(f"gdn_chunk_fwd_noalloc: g and beta must be [B,T,HV] = {(B, T, HV)}")
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev, ndim=1)
        N = int(num_seqs) if num_seqs is not None else cu_seqlens.numel() - 1
    else:
        N = B
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, dev)
        if tuple(initial_state.shape) != (N, HV, K, V):
            raise ValueError(f"initial_state must be [N,HV,K,V] = {(N, HV, K, V)}")
    if o is None:
        o = torch.empty((B, T, HV, V), dtype=torch.bfloat16, device=dev)
    _check(o, "o", torch.bfloat16, dev)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, HV, K, V), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev)
    rc = load_library().gdn_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _scale_arg(scale), _ptr(initial_state),
        _ptr(cu_seqlens), N, B, T, H, HV, K, V, int(bool(use_qk_l2norm)), _ptr(o), _ptr(final_state),
        _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_chunk_fwd_noalloc", rc)
    return o, final_state


def gdn_recurrent_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         ssm_pool: torch.Tensor, ssm_indices: torch.Tensor,
                         g: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None,
                         A_log: Optional[torch.Tensor] = None, a: Optional[torch.Tensor] = None,
                         b: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                         scale: Optional[float] = None, use_qk_l2norm: bool = True,
                         dev_status: Optional[torch.Tensor] = None,
                         o: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One-token decode against ``ssm_pool`` [P,HV,K,V] fp32 (updated in place).

    q, k bf16 [R,1,H,K]; v bf16 [R,1,HV,V]; ssm_indices int32 [R] (-1 = PAD).
    Gates: either g, beta fp32 [R,HV], or A_log, dt_bias fp32 [HV] with a, b bf16
    [R,HV] (fused gating).  Returns o bf16 [R,1,HV,V]."""
    if ssm_pool is None or ssm_indices is None:
        raise ValueError("gdn_recurrent_decode: ssm_pool and ssm_indices are required")
    dev = q.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (ssm_pool, "ssm_pool", torch.float32), (ssm_indices, "ssm_indices", torch.int32)):
        _check(t, n, dt, dev)
    if q.dim() != 4 or q.shape[1] != 1 or k.shape != q.shape or v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise ValueError("gdn_recurrent_decode: q, k must be [R,1,H,K] and v [R,1,HV,V]")
    R, _, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if ssm_pool.dim() != 4 or tuple(ssm_pool.shape[1:]) != (HV, K, V):
        raise ValueError(f"ssm_pool must be [P,{HV},{K},{V}]")
    if ssm_indices.numel() != R:
        raise ValueError("ssm_indices must have one entry per request")
    for t, n, dt in ((g, "g", torch.float32), (beta, "beta", torch.float32),
                     (A_log, "A_log", torch.float32), (dt_bias, "dt_bias", torch.float32),
                     (a, "a", torch.bfloat16), (b, "b", torch.bfloat16)):
        _check(t, n, dt, dev)
    if o is None:
        o = torch.empty((R, 1, HV, V), dtype=torch.bfloat16, device=dev)
    _check(o, "o", torch.bfloat16, dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev)
    rc = load_library().gdn_recurrent_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(a), _ptr(b), _ptr(dt_bias),
        _scale_arg(scale), int(bool(use_qk_l2norm)), _ptr(ssm_pool), ssm_pool.shape[0],
        _ptr(ssm_indices), R, H, HV, K, V, _ptr(o), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_recurrent_decode", rc)
    return o


# Short aliases mirroring the pages' Python names.
chunk_gated_delta_rule = gdn_chunk_fwd
fused_gdn_gating = gdn_gating


# ------------------------------------------------------------------ conv1d
_ACT = {None: 0, "none": 0, "silu": 1, "swish": 1}


def _act_code(activation) -> int:
    if activation not in _ACT:
        raise ValueError(f"activation must be None or 'silu', got {activation!r}")
    return _ACT[activation]


def gdn_causal_conv1d_fwd(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor],
                          conv_states: Optional[torch.Tensor], query_start_loc: torch.Tensor,
                          cache_indices: Optional[torch.Tensor] = None,
                          has_initial_state: Optional[torch.Tensor] = None, activation="silu",
                          out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None):
    """Packed causal conv1d prefill; see ``gdn_causal_conv1d_fwd`` in include/gdn.h.

    x [dim, total] bf16 (channel-first), weight [dim, W], bias [dim] or None,
    conv_states [P, dim, S] (updated in place), query_start_loc int32 [N + 1],
    cache_indices int32 [N], has_initial_state bool [N].  Returns out [dim, total].
    """
    dev = x.device
    _check(x, "x", torch.bfloat16, dev, 2)
    _check(weight, "weight", torch.bfloat16, dev, 2)
    _check(bias, "bias", torch.bfloat16, dev, 1)
    _check(conv_states, "conv_states", torch.bfloat16, dev, 3)
    _check(query_start_loc, "query_start_loc", torch.int32, dev, 1)
    _check(cache_indices, "cache_indices", torch.int32, dev, 1)
    if has_initial_state is not None:
        _check(has_initial_state, "has_initial_state", torch.bool, dev, 1)
    dim, total = x.shape
    W = weight.shape[1]
    P, S = (conv_states.shape[0], conv_states.shape[2]) if conv_states is not None else (0, max(W - 1, 1))
    N = query_start_loc.shape[0] - 1
    if out is None:
        out = torch.empty_like(x)
    rc = load_library().gdn_causal_conv1d_fwd(
        _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_states), P, S, _ptr(query_start_loc),
        _ptr(cache_indices), _ptr(has_initial_state), N, dim, total, W, _act_code(activation), _ptr(out),
        _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_causal_conv1d_fwd", rc)
    return out


def gdn_causal_conv1d_update(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
                             bias: Optional[torch.Tensor], conv_state_indices: torch.Tensor, activation="silu",
                             out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None):
    """One-token conv against the state pool; see include/gdn.h.  x [R, dim] bf16,
    conv_state [P, dim, S] (in place), conv_state_indices int32 [R] (-1 = PAD).
    Returns out [R, dim]."""
    dev = x.device
    _check(x, "x", torch.bfloat16, dev, 2)
    _check(conv_state, "conv_state", torch.bfloat16, dev, 3)
    _check(weight, "weight", torch.bfloat16, dev, 2)
    _check(bias, "bias", torch.bfloat16, dev, 1)
    _check(conv_state_indices, "conv_state_indices", torch.int32, dev, 1)
    R, dim = x.shape
    if out is None:
        out = torch.empty_like(x)
    rc = load_library().gdn_causal_conv1d_update(
        _ptr(x), _ptr(conv_state), conv_state.shape[0], conv_state.shape[2], _ptr(weight), _ptr(bias),
        _ptr(conv_state_indices), R, dim, weight.shape[1], _act_code(activation), _ptr(out), _ptr(dev_status),
        _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_causal_conv1d_update", rc)
    return out


def gdn_causal_conv1d_update_spec(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
                                  bias: Optional[torch.Tensor], conv_state_indices: torch.Tensor,
                                  num_accepted_tokens: Optional[torch.Tensor], query_start_loc: torch.Tensor,
                                  mtp_step: int, activation="silu", out: Optional[torch.Tensor] = None,
                                  dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Multi-token (MTP) decode conv; see include/gdn.h.  x [Ttot, dim] bf16;
    conv_state [P, dim, state_len] bf16 (in place, state_len >= width - 1 +
    mtp_step); conv_state_indices int32 [N]; num_accepted_tokens int32 [N] or
    None; query_start_loc int32 [N + 1].  Returns out [Ttot, dim]."""
    dev = x.device
    _check(x, "x", torch.bfloat16, dev, 2)
    _check(conv_state, "conv_state", torch.bfloat16, dev, 3)
    _check(weight, "weight", torch.bfloat16, dev, 2)
    _check(bias, "bias", torch.bfloat16, dev, 1)
    _check(conv_state_indices, "conv_state_indices", torch.int32, dev, 1)
    _check(num_accepted_tokens, "num_accepted_tokens", torch.int32, dev, 1)
    _check(query_start_loc, "query_start_loc", torch.int32, dev, 1)
    Ttot, dim = x.shape
    N = conv_state_indices.shape[0]
    if query_start_loc.shape[0] != N + 1:
        raise ValueError("query_start_loc must hold N + 1 offsets")
    if out is None:
        out = torch.empty_like(x)
    rc = load_library().gdn_causal_conv1d_update_spec(
        _ptr(x), _ptr(conv_state), conv_state.shape[0], conv_state.shape[2], _ptr(weight), _ptr(bias),
        _ptr(conv_state_indices), _ptr(num_accepted_tokens), _ptr(query_start_loc), N, Ttot, int(mtp_step), dim,
        weight.shape[1], _act_code(activation), _ptr(out), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_causal_conv1d_update_spec", rc)
    return out


def gdn_conv_decode_pack(mixed_qkv: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
                         bias: Optional[torch.Tensor], conv_state_indices: torch.Tensor, H: int, HV: int, K: int,
                         V: int, activation="silu", dev_status: Optional[torch.Tensor] = None):
    """Decode conv over the packed q | k | v channels, returned split as
    q, k [R, 1, H, K] and v [R, 1, HV, V] (the inputs gdn_recurrent_decode takes)."""
    dev = mixed_qkv.device
    _check(mixed_qkv, "mixed_qkv", torch.bfloat16, dev, 2)
    _check(conv_state, "conv_state", torch.bfloat16, dev, 3)
    _check(weight, "weight", torch.bfloat16, dev, 2)
    _check(bias, "bias", torch.bfloat16, dev, 1)
    _check(conv_state_indices, "conv_state_indices", torch.int32, dev, 1)
    R = mixed_qkv.shape[0]
    q = torch.empty(R, 1, H, K, dtype=torch.bfloat16, device=dev)
    k = torch.empty(R, 1, H, K, dtype=torch.bfloat16, device=dev)
    v = torch.empty(R, 1, HV, V, dtype=torch.bfloat16, device=dev)
    rc = load_library().gdn_conv_decode_pack(
        _ptr(mixed_qkv), _ptr(conv_state), conv_state.shape[0], conv_state.shape[2], _ptr(weight), _ptr(bias),
        _ptr(conv_state_indices), R, H, HV, K, V, weight.shape[1], _act_code(activation), _ptr(q), _ptr(k),
        _ptr(v), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_conv_decode_pack", rc)
    return q, k, v


# ------------------------------------------------------- decode variants
def _gate_args(g, beta, A_log, a, b, dt_bias, dev):
    for t, n, dt in ((g, "g", torch.float32), (beta, "beta", torch.float32),
                     (A_log, "A_log", torch.float32), (dt_bias, "dt_bias", torch.float32),
                     (a, "a", torch.bfloat16), (b, "b", torch.bfloat16)):
        _check(t, n, dt, dev)


def gdn_recurrent_decode_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ssm_pool: torch.Tensor,
                              ssm_indices: torch.Tensor, g=None, beta=None, A_log=None, a=None, b=None,
                              dt_bias=None, scale=None, use_qk_l2norm: bool = True, o=None, dev_status=None):
    """gdn_recurrent_decode against a bf16 state pool [P, HV, K, V] (updated in place)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, dev, 4)
    _check(ssm_pool, "ssm_pool", torch.bfloat16, dev, 4)
    _check(ssm_indices, "ssm_indices", torch.int32, dev, 1)
    _gate_args(g, beta, A_log, a, b, dt_bias, dev)
    R, _, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if o is None:
        o = torch.empty((R, 1, HV, V), dtype=torch.bfloat16, device=dev)
    rc = load_library().gdn_recurrent_decode_bf16(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(a), _ptr(b), _ptr(dt_bias),
        _scale_arg(scale), int(bool(use_qk_l2norm)), _ptr(ssm_pool), ssm_pool.shape[0], _ptr(ssm_indices), R,
        H, HV, K, V, _ptr(o), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_recurrent_decode_bf16", rc)
    return o


def gdn_recurrent_decode_mtp(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ssm_pool: torch.Tensor,
                             cu_seqlens: torch.Tensor, read_indices: torch.Tensor, write_indices: torch.Tensor,
                             num_accepted_tokens: Optional[torch.Tensor] = None, g=None, beta=None, A_log=None,
                             a=None, b=None, dt_bias=None, scale=None, use_qk_l2norm: bool = True, o=None,
                             dev_status=None):
    """Multi-token decode; see include/gdn.h.  q, k [Ttot, H, K], v [Ttot, HV, V] bf16;
    ssm_pool fp32 [P, HV, K, V] (in place); cu_seqlens int32 [N + 1]; read / write
    indices int32 [N, ld]; num_accepted_tokens int32 [N] or None.  Returns o [Ttot, HV, V]."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, dev, 3)
    _check(ssm_pool, "ssm_pool", torch.float32, dev, 4)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _check(read_indices, "read_indices", torch.int32, dev, 2)
    _check(write_indices, "write_indices", torch.int32, dev, 2)
    _check(num_accepted_tokens, "num_accepted_tokens", torch.int32, dev, 1)
    _gate_args(g, beta, A_log, a, b, dt_bias, dev)
    if read_indices.shape != write_indices.shape:
        raise ValueError("read_indices and write_indices must have the same shape [N, ld]")
    Tt, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    N, ld = read_indices.shape
    if o is None:
        o = torch.empty((Tt, HV, V), dtype=torch.bfloat16, device=dev)
    rc = load_library().gdn_recurrent_decode_mtp(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(a), _ptr(b), _ptr(dt_bias),
        _scale_arg(scale), int(bool(use_qk_l2norm)), _ptr(ssm_pool), ssm_pool.shape[0], _ptr(cu_seqlens), N, Tt,
        _ptr(read_indices), _ptr(write_indices), ld, _ptr(num_accepted_tokens), H, HV, K, V, _ptr(o),
        _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_recurrent_decode_mtp", rc)
    return o


# ----------------------------------------------------------------- backward
def chunk_bwd_workspace_size(B, T, H, HV, K, V, N, varlen) -> int:
    return int(load_library().gdn_chunk_bwd_workspace_size(B, T, H, HV, K, V, N, int(bool(varlen))))


def gdn_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  do: torch.Tensor, scale=None, initial_state: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None, dht: Optional[torch.Tensor] = None,
                  use_qk_l2norm: bool = True, workspace: Optional[torch.Tensor] = None,
                  dev_status: Optional[torch.Tensor] = None):
    """Gradients of gdn_chunk_fwd; see include/gdn.h.  Returns
    (dq, dk, dv, dg, dbeta, dh0) as fp32 tensors (dh0 None without initial_state)."""
    dev = q.device
    _check(q, "q", torch.bfloat16, dev, 4)
    _check(k, "k", torch.bfloat16, dev, 4)
    _check(v, "v", torch.bfloat16, dev, 4)
    _check(g, "g", torch.float32, dev, 3)
    _check(beta, "beta", torch.float32, dev, 3)
    _check(do, "do", torch.bfloat16, dev, 4)
    _check(initial_state, "initial_state", torch.float32, dev, 4)
    _check(dht, "dht", torch.float32, dev, 4)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else B
    if tuple(k.shape) != (B, T, H, K) or tuple(v.shape[:2]) != (B, T) or tuple(do.shape) != (B, T, HV, V):
        raise ValueError("gdn_chunk_bwd: q, k [B,T,H,K], v and do [B,T,HV,V] must agree")
    if tuple(g.shape) != (B, T, HV) or tuple(beta.shape) != (B, T, HV):
        raise ValueError(f"gdn_chunk_bwd: g and beta must be [B,T,HV] = {(B, T, HV)}")
    for t, n in ((initial_state, "initial_state"), (dht, "dht")):
        if t is not None and tuple(t.shape) != (N, HV, K, V):
            raise ValueError(f"gdn_chunk_bwd: {n} must be [N,HV,K,V] = {(N, HV, K, V)}")
    dq = torch.empty(B, T, H, K, dtype=torch.float32, device=dev)
    dk = torch.empty_like(dq)
    dv = torch.empty(B, T, HV, V, dtype=torch.float32, device=dev)
    dg = torch.empty(B, T, HV, dtype=torch.float32, device=dev)
    dbeta = torch.empty_like(dg)
    dh0 = torch.empty(N, HV, K, V, dtype=torch.float32, device=dev) if initial_state is not None else None
    need = chunk_bwd_workspace_size(B, T, H, HV, K, V, N, cu_seqlens is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    rc = load_library().gdn_chunk_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _scale_arg(scale), _ptr(initial_state), _ptr(cu_seqlens),
        N, B, T, H, HV, K, V, int(bool(use_qk_l2norm)), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
        _ptr(dbeta), _ptr(dh0), _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(dev))
    if rc != GDN_OK:
        raise GDNError("gdn_chunk_bwd", rc)
    return dq, dk, dv, dg, dbeta, dh0


class _ChunkGatedDeltaRule(torch.autograd.Function):
    """gdn_chunk_fwd forward, gdn_chunk_bwd backward (marshalling only)."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, scale, output_final_state, cu_seqlens, use_qk_l2norm,
                num_seqs):
        o, ht = gdn_chunk_fwd(q, k, v, g, beta, scale=scale, initial_state=initial_state,
                              output_final_state=output_final_state, cu_seqlens=cu_seqlens,
                              use_qk_l2norm=use_qk_l2norm, num_seqs=num_seqs)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens)
        ctx.scale, ctx.l2 = scale, use_qk_l2norm
        if ht is None:
            return o
        return o, ht

    @staticmethod
    def backward(ctx, do, dht=None):
        q, k, v, g, beta, h0, cu = ctx.saved_tensors
        do = do.to(torch.bfloat16).contiguous()
        dht = None if dht is None else dht.float().contiguous()
        dq, dk, dv, dg, dbeta, dh0 = gdn_chunk_bwd(q, k, v, g, beta, do, scale=ctx.scale, initial_state=h0,
                                                   cu_seqlens=cu, dht=dht, use_qk_l2norm=ctx.l2)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dg, dbeta,
                None if dh0 is None else dh0, None, None, None, None, None)


def chunk_gated_delta_rule(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                           beta: torch.Tensor, scale: Optional[float] = None,
                           initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                           cu_seqlens: Optional[torch.Tensor] = None, use_qk_l2norm_in_kernel: bool = True,
                           num_seqs: Optional[int] = None):
    """Differentiable chunked prefill with the argument names of the pages'
    chunk_gated_delta_rule (FastDeploy PR "support fla triton kernel for
    qwen3.5", Usage section 1).  Returns (o, final_state) (final_state None
    unless ``output_final_state``); autograd runs gdn_chunk_bwd and yields
    gradients for q, k, v (in their bf16 dtype), g, beta and initial_state
    (fp32)."""
    out = _ChunkGatedDeltaRule.apply(q, k, v, g, beta, initial_state, scale, output_final_state, cu_seqlens,
                                     use_qk_l2norm_in_kernel, num_seqs)
    if isinstance(out, tuple):
        return out
    return out, None
