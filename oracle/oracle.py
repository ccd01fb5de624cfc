"""Oracle for the Gated DeltaNet forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this module.  The product library never does, and this
module imports nothing from the product package.

Contents
--------
* ``gating``, ``recurrent``, ``decode``, ``decode_mtp``: thin ctypes
  front-ends to the plain C fp64 oracle in ``gdn_oracle.c`` (the per-token
  definitions; see that file for the passages each one follows).
* ``decode_bf16_pool``: ``decode`` on a pool stored in bf16 (the step runs on
  the stored values, the new state is rounded back to bf16 by ``round_bf16``,
  ties to even).
* Independent numpy restatements used only to pin the C oracle:
    - ``gating_scalar``: the gating formula evaluated with Python's ``math``.
    - ``transition_product``: the recurrence written as
      S_t = a_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
      (the same update, factored the other way round).
    - ``attention_form``: the whole sequence as one chunk, solved with a dense
      LU: (I + A) Delta = diag(beta) V - diag(beta e^gamma) K S0, then
      o = scale (diag(e^gamma) Q S0 + (Q K^T * causal decay) Delta).
    - ``chunked_wy``: the six-step chunked algorithm of "NPU Training
      Operators - GDN", section "Operator semantics" (chunk-local cumsum ->
      beta K K^T with gate decay -> triangular solve -> w/u recompute ->
      inter-chunk state propagation -> output), in fp64 with a dense
      triangular solve, for any chunk size C.  It is a self-check of the
      derivation only, never compared against the GPU path.

Parity pinning: every function above is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants and brute force; nothing on the pages prints
absolute output values, so no pin comes from a printed worked example.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i = ctypes.POINTER(ctypes.c_int)
            lib.oracle_gating.argtypes = [d, d, d, d, ctypes.c_long, ctypes.c_int, d, d]
            lib.oracle_gating.restype = None
            lib.oracle_recurrent.argtypes = [
                d, d, d, d, d, ctypes.c_double, d, i, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, d, d, i, ctypes.c_int, ctypes.c_int]
            lib.oracle_recurrent.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [
                d, d, d, d, d, ctypes.c_double, ctypes.c_int, d, ctypes.c_int, i,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                d, i]
            lib.oracle_decode.restype = ctypes.c_int
            CI = ctypes.c_int
            lib.oracle_decode_mtp.argtypes = [
                d, d, d, d, d, ctypes.c_double, CI, d, CI, i, CI, i, i, CI, i, CI, CI, CI, CI, d, i]
            lib.oracle_decode_mtp.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of a numpy array or a (CPU) torch tensor of any float dtype."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only to widen bf16 exactly
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int)) if a is not None else None


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------
# C front-ends
# --------------------------------------------------------------------------

def gating(A_log, a, b, dt_bias):
    """g, beta (fp64, shape of a) from the gating formula; a, b: [Ttok, HV]."""
    A_log, a, b, dt_bias = map(_f64, (A_log, a, b, dt_bias))
    Ttok, HV = a.shape
    g = np.empty_like(a)
    beta = np.empty_like(a)
    _load().oracle_gating(_dp(A_log), _dp(a), _dp(b), _dp(dt_bias), Ttok, HV, _dp(g), _dp(beta))
    return g, beta


def recurrent(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
              use_qk_l2norm=True, output_final_state=True, items=None, nthreads=None):
    """Per-token fp64 recurrence over dense [B,T,...] or varlen (cu_seqlens) input.

    Shapes: q, k [B,T,H,K]; v [B,T,HV,V]; g, beta [B,T,HV];
    initial_state [N,HV,K,V] or None.  Returns (o [B,T,HV,V], final [N,HV,K,V] or None).
    ``items``: optional iterable of (n, hv) pairs to compute; other outputs stay NaN.
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = len(cu) - 1
    else:
        N = B
    h0 = _f64(initial_state) if initial_state is not None else None
    o = np.full((B, T, HV, V), np.nan)
    ht = np.full((N, HV, K, V), np.nan) if output_final_state else None
    it = None
    n_items = 0
    if items is not None:
        it = np.ascontiguousarray(np.array([n * HV + hv for n, hv in items], dtype=np.int32))
        n_items = len(it)
    sc = float(scale) if scale is not None else -1.0
    rc = _load().oracle_recurrent(
        _dp(q), _dp(k), _dp(v), _dp(g), _dp(beta), sc, _dp(h0), _ip(cu), N, B, T, H,
        HV, K, V, int(bool(use_qk_l2norm)), _dp(o), _dp(ht), _ip(it), n_items,
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_recurrent: inconsistent arguments")
    return o, ht


def decode(q, k, v, g, beta, pool, ssm_indices, scale=None, use_qk_l2norm=True):
    """Pool-indexed one-token decode.  q, k [R,H,K] (or [R,1,H,K]); v [R,HV,V];
    g, beta [R,HV]; pool [P,HV,K,V] (a copy is updated and returned).
    Returns (o [R,HV,V], new_pool, bad_index_flag)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    q = q.reshape(q.shape[0], -1, q.shape[-1])
    k = k.reshape(k.shape[0], -1, k.shape[-1])
    v = v.reshape(v.shape[0], -1, v.shape[-1])
    g = g.reshape(g.shape[0], -1)
    beta = beta.reshape(beta.shape[0], -1)
    R, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    pool = _f64(pool).copy()
    P = pool.shape[0]
    idx = np.ascontiguousarray(np.asarray(ssm_indices, dtype=np.int32))
    o = np.empty((R, HV, V))
    bad = ctypes.c_int(0)
    sc = float(scale) if scale is not None else -1.0
    rc = _load().oracle_decode(_dp(q), _dp(k), _dp(v), _dp(g), _dp(beta), sc,
                               int(bool(use_qk_l2norm)), _dp(pool), P, _ip(idx), R,
                               H, HV, K, V, _dp(o), ctypes.byref(bad))
    if rc != 0:
        raise ValueError("oracle_decode: inconsistent arguments")
    return o, pool, bad.value


def decode_mtp(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx, num_accepted=None, scale=None,
               use_qk_l2norm=True):
    """Multi-token decode (see ``oracle_decode_mtp`` in gdn_oracle.c).
    q, k [Ttot,H,K] (or [Ttot,1,H,K]); v [Ttot,HV,V]; g, beta [Ttot,HV];
    pool [P,HV,K,V] (a copy is updated and returned); cu_seqlens [N+1];
    read_idx / write_idx [N, ld]; num_accepted [N] or None.
    Returns (o [Ttot,HV,V], new_pool, bad_index_flag)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    q = q.reshape(q.shape[0], -1, q.shape[-1])
    k = k.reshape(k.shape[0], -1, k.shape[-1])
    v = v.reshape(v.shape[0], -1, v.shape[-1])
    g = g.reshape(g.shape[0], -1)
    beta = beta.reshape(beta.shape[0], -1)
    Tt, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    pool = _f64(pool).copy()
    P = pool.shape[0]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    ri = np.ascontiguousarray(np.asarray(read_idx, dtype=np.int32))
    wi = np.ascontiguousarray(np.asarray(write_idx, dtype=np.int32))
    N, ld = ri.shape
    na = None if num_accepted is None else np.ascontiguousarray(np.asarray(num_accepted, dtype=np.int32))
    o = np.zeros((Tt, HV, V))
    bad = ctypes.c_int(0)
    sc = float(scale) if scale is not None else -1.0
    rc = _load().oracle_decode_mtp(_dp(q), _dp(k), _dp(v), _dp(g), _dp(beta), sc, int(bool(use_qk_l2norm)),
                                   _dp(pool), P, _ip(cu), N, _ip(ri), _ip(wi), ld,
                                   None if na is None else _ip(na), H, HV, K, V, _dp(o), ctypes.byref(bad))
    if rc != 0:
        raise ValueError("oracle_decode_mtp: inconsistent arguments")
    return o, pool, bad.value


def round_bf16(x):
    """Round fp64 values to the nearest bf16 (8 significant bits, ties to even)
    and return them as fp64: the storage rounding of a bf16 state pool."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0), e - 8)


def decode_bf16_pool(q, k, v, g, beta, pool_bf16_values, ssm_indices, scale=None, use_qk_l2norm=True):
    """One-token decode against a pool stored in bf16: the step runs on the
    stored values (upcast), the output uses the updated state, and the state is
    stored back rounded to bf16.  pool_bf16_values holds the bf16 numbers as
    floats.  Returns (o, new_pool_values, bad_index_flag)."""
    pool = _f64(pool_bf16_values)
    o, new, bad = decode(q, k, v, g, beta, pool, ssm_indices, scale=scale, use_qk_l2norm=use_qk_l2norm)
    touched = sorted({int(s) for s in np.asarray(ssm_indices).ravel() if 0 <= int(s) < pool.shape[0]})
    for s in touched:
        new[s] = round_bf16(new[s])
    return o, new, bad


# --------------------------------------------------------------------------
# Independent numpy restatements (pins for the C oracle)
# --------------------------------------------------------------------------

def gating_scalar(A_log, a, b, dt_bias):
    """The gating formula with Python's math module, one element at a time."""
    A_log, a, b, dt_bias = map(_f64, (A_log, a, b, dt_bias))
    g = np.empty_like(a)
    beta = np.empty_like(a)
    for t in range(a.shape[0]):
        for h in range(a.shape[1]):
            x = a[t, h] + dt_bias[h]
            sp = x if x > 20.0 else math.log1p(math.exp(x))
            g[t, h] = -math.exp(A_log[h]) * sp
            beta[t, h] = 1.0 / (1.0 + math.exp(-b[t, h]))
    return g, beta


def _normalise(x, on):
    if not on:
        return x
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + L2_EPS)


def transition_product(q, k, v, g, beta, S0, scale, use_qk_l2norm=True):
    """One sequence, one head: S_t = a_t (I - beta_t k k^T) S_{t-1} + beta_t k v^T.
    q, k [T,K]; v [T,V]; g, beta [T]; S0 [K,V].  Returns (o [T,V], S_T)."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    qn, kn = _normalise(q, use_qk_l2norm), _normalise(k, use_qk_l2norm)
    K = k.shape[1]
    S = S0.copy()
    o = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        M = math.exp(g[t]) * (np.eye(K) - beta[t] * np.outer(kn[t], kn[t]))
        S = M @ S + beta[t] * np.outer(kn[t], v[t])
        o[t] = scale * (S.T @ qn[t])
    return o, S


def attention_form(q, k, v, g, beta, S0, scale, use_qk_l2norm=True):
    """One sequence as a single chunk, with a dense LU solve (numpy.linalg.solve).
    Returns (o [T,V], S_T)."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    Q, Kn = _normalise(q, use_qk_l2norm), _normalise(k, use_qk_l2norm)
    T = q.shape[0]
    gam = np.cumsum(g)
    diff = gam[:, None] - gam[None, :]
    decay = np.where(np.tril(np.ones((T, T))) > 0, np.exp(np.minimum(diff, 0.0)), 0.0)
    A = np.tril(beta[:, None] * decay * (Kn @ Kn.T), -1)
    rhs = beta[:, None] * v - (beta * np.exp(gam))[:, None] * (Kn @ S0)
    Delta = np.linalg.solve(np.eye(T) + A, rhs)
    o = scale * (np.exp(gam)[:, None] * (Q @ S0) + (decay * (Q @ Kn.T)) @ Delta)
    ST = np.exp(gam[-1]) * S0 + Kn.T @ (np.exp(gam[-1] - gam)[:, None] * Delta)
    return o, ST


def chunked_wy(q, k, v, g, beta, S0, scale, C=64, use_qk_l2norm=True):
    """The chunked WY algorithm in fp64 for one sequence and one head.

    Per chunk (rows i, j inside the chunk, L rows):
      gamma = chunk-local cumsum of g
      A_ij  = beta_i e^{gamma_i - gamma_j} k_i . k_j  for i > j, else 0
      Tm    = (I + A)^{-1}                     (dense triangular solve)
      w     = Tm diag(beta e^gamma) K,  u = Tm diag(beta) V
      v_new = u - w h
      o     = scale (diag(e^gamma) Q h + (Q K^T * causal decay) v_new)
      h     = e^{gamma_L} h + K^T diag(e^{gamma_L - gamma}) v_new
    Returns (o [T,V], h after the last chunk).
    """
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    Q, Kn = _normalise(q, use_qk_l2norm), _normalise(k, use_qk_l2norm)
    T = q.shape[0]
    h = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        L = sl.stop - sl.start
        Kc, Qc, Vc, b = Kn[sl], Q[sl], v[sl], beta[sl]
        gam = np.cumsum(g[sl])
        diff = gam[:, None] - gam[None, :]
        causal = np.tril(np.ones((L, L)))
        decay = np.where(causal > 0, np.exp(np.minimum(diff, 0.0)), 0.0)
        A = np.tril(b[:, None] * decay * (Kc @ Kc.T), -1)
        Tm = np.linalg.solve(np.eye(L) + A, np.eye(L))
        w = Tm @ ((b * np.exp(gam))[:, None] * Kc)
        u = Tm @ (b[:, None] * Vc)
        v_new = u - w @ h
        o[sl] = scale * (np.exp(gam)[:, None] * (Qc @ h) + (decay * (Qc @ Kc.T)) @ v_new)
        h = np.exp(gam[-1]) * h + Kc.T @ (np.exp(gam[-1] - gam)[:, None] * v_new)
    return o, h
