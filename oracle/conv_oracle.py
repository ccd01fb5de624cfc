"""Oracle for the causal depthwise conv1d that feeds Gated DeltaNet -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the product library never does, and this module imports
nothing from the product package.

What it computes (FastDeploy PR "support fla triton kernel for qwen3.5",
Modifications table for ``causal_conv1d.py`` and Usage sections 3 and 4; the
LightLLM "gdn.py" prefill and decode backends, which call the prefill form on
the packed q|k|v channels and a fused decode conv + split):

* The pages give the calling convention -- a per-channel (depthwise) causal
  convolution of width ``W`` over the token axis, optional bias, optional SiLU,
  a pool of per-sequence conv states addressed by slot indices and updated in
  place, ``query_start_loc`` offsets and ``has_initial_state`` flags for packed
  prefill -- but not the arithmetic.  The plain reading adopted here: for
  channel ``d`` and token position ``p`` of a sequence whose input stream is
  ``history ++ x`` (``history`` = the slot's state, or zeros),

      out[d, p] = act(bias[d] + sum_{j=0}^{W-1} weight[d, j] * stream[d, p + j])

  where ``stream`` positions are counted so that ``stream[d, p + W - 1]`` is
  ``x[d, p]`` (the last tap multiplies the current token), and the state after
  the call holds the last ``S`` entries of ``history ++ x`` (``S`` >= W - 1;
  only its last W - 1 entries reach the convolution).
* ``act`` is either the identity or SiLU, x * sigmoid(x).
* Slot index -1 (PAD) reads no state (zeros) and writes none; for the
  single-token decode form its output row is zero.

Everything is fp64 numpy with explicit loops over the taps, written for
reading, not speed.  Pinned by ``tests/test_conv_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

PAD_SLOT = -1


def silu(x):
    """x * sigmoid(x) in fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def _act(x, activation):
    if activation in (None, "none", 0):
        return x
    if activation in ("silu", 1):
        return silu(x)
    raise ValueError(f"unknown activation {activation!r}")


def conv_stream(stream, weight, bias, activation):
    """Valid causal convolution of one stream.

    stream : [dim, W - 1 + L] fp64 (history then the L inputs)
    weight : [dim, W]
    returns [dim, L]: out[:, p] = act(bias + sum_j weight[:, j] * stream[:, p + j]).
    """
    stream = np.asarray(stream, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    dim, W = weight.shape
    L = stream.shape[1] - (W - 1)
    acc = np.zeros((dim, max(L, 0)), dtype=np.float64)
    if bias is not None:
        acc += np.asarray(bias, dtype=np.float64)[:, None]
    for j in range(W):
        acc += weight[:, j:j + 1] * stream[:, j:j + L]
    return _act(acc, activation)


def causal_conv1d_varlen(x, weight, bias, conv_states, query_start_loc, cache_indices,
                         has_initial_state, activation="silu"):
    """Packed prefill (the ``causal_conv1d_fn`` form).

    x                 : [dim, total] channel-first
    weight            : [dim, W]; bias: [dim] or None
    conv_states       : [P, dim, S] pool (not modified; the new pool is returned)
    query_start_loc   : [N + 1] offsets into the token axis
    cache_indices     : [N] slot per sequence (-1: no slot)
    has_initial_state : [N] bool
    returns (out [dim, total], new_states [P, dim, S])
    """
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    states = np.array(conv_states, dtype=np.float64, copy=True)
    dim, total = x.shape
    W = weight.shape[1]
    S = states.shape[2]
    out = np.zeros((dim, total), dtype=np.float64)
    qsl = [int(v) for v in query_start_loc]
    for n in range(len(qsl) - 1):
        s0, s1 = qsl[n], qsl[n + 1]
        slot = int(cache_indices[n])
        use_state = slot != PAD_SLOT and bool(has_initial_state[n])
        full_hist = states[slot].copy() if use_state else np.zeros((dim, S))
        seq = x[:, s0:s1]
        stream = np.concatenate([full_hist[:, S - (W - 1):], seq], axis=1)
        out[:, s0:s1] = conv_stream(stream, weight, bias, activation)
        if slot != PAD_SLOT:
            whole = np.concatenate([full_hist, seq], axis=1)
            states[slot] = whole[:, whole.shape[1] - S:]
    return out, states


def causal_conv1d_update(x, conv_state, weight, bias, conv_state_indices, activation="silu"):
    """Single-token decode (the ``causal_conv1d_update`` form).

    x          : [R, dim] one token per request
    conv_state : [P, dim, S] pool (not modified; the new pool is returned)
    returns (out [R, dim], new_state [P, dim, S]); PAD rows give zeros.
    """
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    states = np.array(conv_state, dtype=np.float64, copy=True)
    R, dim = x.shape
    W = weight.shape[1]
    S = states.shape[2]
    out = np.zeros((R, dim), dtype=np.float64)
    for r in range(R):
        slot = int(conv_state_indices[r])
        if slot == PAD_SLOT:
            continue
        hist = states[slot]
        stream = np.concatenate([hist[:, S - (W - 1):], x[r][:, None]], axis=1)
        out[r] = conv_stream(stream, weight, bias, activation)[:, 0]
        states[slot] = np.concatenate([hist[:, 1:], x[r][:, None]], axis=1)
    return out, states


def conv_decode_pack(mixed_qkv, conv_state, weight, bias, conv_state_indices, H, HV, K, V,
                     activation="silu"):
    """Decode conv of the packed q | k | v channels, split into the layouts the
    recurrent decode takes: q, k [R, 1, H, K] and v [R, 1, HV, V] (the LightLLM
    "gdn.py" decode backend's conv + pack step)."""
    out, states = causal_conv1d_update(mixed_qkv, conv_state, weight, bias,
                                       conv_state_indices, activation)
    R = out.shape[0]
    q = out[:, :H * K].reshape(R, 1, H, K)
    k = out[:, H * K:2 * H * K].reshape(R, 1, H, K)
    v = out[:, 2 * H * K:2 * H * K + HV * V].reshape(R, 1, HV, V)
    return q, k, v, states
