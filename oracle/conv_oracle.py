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


def causal_conv1d_update_spec(x, conv_state, weight, bias, conv_state_indices, num_accepted_tokens,
                              query_start_loc, mtp_step, activation="silu"):
    """Multi-token (speculative / MTP) decode conv, the ``causal_conv1d_update``
    of LightLLM "gdn.py" ``_gdn_mtp_kernel`` (called with ``mtp_step``,
    ``num_accepted_tokens`` and ``query_start_loc``).

    x                   : [Ttot, dim] token-major; request n owns rows
                          [query_start_loc[n], query_start_loc[n + 1]), at most
                          mtp_step + 1 of them
    conv_state          : [P, dim, S] pool, S >= W - 1 + mtp_step (the page keeps
                          mtp_step extra entries per slot and slices them off for
                          prefill); not modified, the new pool is returned
    conv_state_indices  : [N] slot per request (-1: PAD, zero outputs, no write)
    num_accepted_tokens : [N] in [1, mtp_step + 1], or None (all 1)

    Reading (the page gives the call, not the arithmetic): a slot holds the last
    S entries of its request's input stream as of the end of the previous step,
    whose last mtp_step + 1 entries were that step's tokens; only the first A =
    num_accepted_tokens of those were accepted, so the last (mtp_step + 1 - A)
    entries are rejected drafts.  The accepted stream is slot[:S - (mtp_step + 1
    - A)]; the new tokens follow it, each output uses the W - 1 inputs before it
    (out[i] = act(bias + sum_j weight[:, j] * stream[i + j]) over the last W - 1
    accepted entries ++ x), and afterwards the slot holds the last S entries of
    accepted ++ x (zeros in front if that is shorter).  After a prefill, which
    writes slot[:W - 1] through the sliced view, A = 1 selects exactly those
    entries.  returns (out [Ttot, dim], new_states [P, dim, S]).
    """
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    states = np.array(conv_state, dtype=np.float64, copy=True)
    Ttot, dim = x.shape
    W = weight.shape[1]
    S = states.shape[2]
    m = int(mtp_step)
    if S < W - 1 + m:
        raise ValueError("state length must hold W - 1 + mtp_step entries")
    out = np.zeros((Ttot, dim), dtype=np.float64)
    qsl = [int(v) for v in query_start_loc]
    for n in range(len(qsl) - 1):
        t0, t1 = qsl[n], qsl[n + 1]
        slot = int(conv_state_indices[n])
        if slot == PAD_SLOT:
            continue
        A = 1 if num_accepted_tokens is None else int(num_accepted_tokens[n])
        accepted = states[slot][:, :S - (m + 1 - A)]
        new = x[t0:t1].T                                     # [dim, n_tokens]
        stream = np.concatenate([accepted[:, accepted.shape[1] - (W - 1):], new], axis=1)
        out[t0:t1] = conv_stream(stream, weight, bias, activation).T
        whole = np.concatenate([accepted, new], axis=1)
        if whole.shape[1] < S:
            whole = np.concatenate([np.zeros((dim, S - whole.shape[1])), whole], axis=1)
        states[slot] = whole[:, whole.shape[1] - S:]
    return out, states
