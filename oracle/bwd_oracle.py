"""Oracle for the Gated DeltaNet backward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and ``bench.py``'s CPU legs may import this module; the
product library never does, and this module imports nothing from it.

The pages name the backward as the training use case of the same operator
("NPU Training Operators - GDN": the chunked forward is paired with a backward
that returns the gradients of q, k, v, beta, g and the initial state; the
FastDeploy PR's chunk entry point takes the same inputs).  They print no
backward formulas, so the oracle is the plainest definition: reverse-mode
differentiation of the per-token recurrence

    S_t = e^{g_t} S_{t-1} + beta_t k_t (v_t - e^{g_t} S_{t-1}^T k_t)^T,
    o_t = scale * S_t^T q_t,

with the optional per-token L2 normalisation x / sqrt(sum(x^2) + 1e-6) of q
and k, written as plain fp64 PyTorch CPU ops and differentiated by
``torch.autograd``.  Given the upstream gradients do [B,T,HV,V] and (optionally)
dht [N,HV,K,V] it returns dq, dk [B,T,H,K], dv [B,T,HV,V], dg, dbeta [B,T,HV]
and dh0 [N,HV,K,V].  GVA: value head hv reads key head hv // (HV / H), so the
key-head gradients sum over the value heads of a group.

Pinned by ``tests/test_bwd_oracle_pins.py`` against central finite differences
of an independent evaluation of the forward (the C oracle).
"""
from __future__ import annotations

import numpy as np
import torch

L2_EPS = 1e-6


def _t(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def forward_torch(q, k, v, g, beta, scale, h0, cu_seqlens, use_qk_l2norm):
    """Differentiable fp64 forward (torch tensors in, (o, ht) out)."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    if use_qk_l2norm:
        q = q / torch.sqrt((q * q).sum(-1, keepdim=True) + L2_EPS)
        k = k / torch.sqrt((k * k).sum(-1, keepdim=True) + L2_EPS)
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        seqs = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    o_rows = {}
    hts = []
    for n, (b, t0, t1) in enumerate(seqs):
        heads = []
        for hv in range(HV):
            h = hv // G
            S = h0[n, hv] if h0 is not None else torch.zeros(K, V, dtype=torch.float64)
            for t in range(t0, t1):
                a = torch.exp(g[b, t, hv])
                kt = k[b, t, h]
                r = S.t() @ kt
                S = a * S + beta[b, t, hv] * torch.outer(kt, v[b, t, hv] - a * r)
                o_rows[(b, t, hv)] = scale * (S.t() @ q[b, t, h])
            heads.append(S)
        hts.append(torch.stack(heads))
    o = torch.zeros(B, T, HV, V, dtype=torch.float64)
    rows = torch.stack([o_rows[key] for key in sorted(o_rows)]) if o_rows else None
    if rows is not None:
        idx = sorted(o_rows)
        bi = torch.tensor([x[0] for x in idx])
        ti = torch.tensor([x[1] for x in idx])
        hi = torch.tensor([x[2] for x in idx])
        o = o.index_put((bi, ti, hi), rows)
    return o, torch.stack(hts)


def backward(q, k, v, g, beta, do, scale=None, initial_state=None, cu_seqlens=None, dht=None,
             use_qk_l2norm=True):
    """Gradients of sum(o * do) + sum(ht * dht) with respect to every input.

    Arrays in (numpy or torch, any float dtype), fp64 numpy arrays out:
    (dq, dk, dv, dg, dbeta, dh0) with dh0 None when initial_state is None.
    """
    q, k, v, g, beta, do = map(_t, (q, k, v, g, beta, do))
    K = q.shape[-1]
    sc = float(scale) if scale is not None and scale > 0 else 1.0 / np.sqrt(K)
    h0 = _t(initial_state) if initial_state is not None else None
    leaves = [q, k, v, g, beta] + ([h0] if h0 is not None else [])
    for x in leaves:
        x.requires_grad_(True)
    o, ht = forward_torch(q, k, v, g, beta, sc, h0, cu_seqlens, use_qk_l2norm)
    loss = (o * do).sum()
    if dht is not None:
        loss = loss + (ht * _t(dht)).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    out = [gr.detach().numpy() if gr is not None else np.zeros(x.shape) for gr, x in zip(grads, leaves)]
    dq, dk, dv, dg, db = out[:5]
    dh0 = out[5] if h0 is not None else None
    return dq, dk, dv, dg, db, dh0
