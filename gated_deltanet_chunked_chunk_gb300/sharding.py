"""Head-group sharding of the prefill across ranks (host-side bookkeeping only).

LightLLM "gdn.py", ``_init_linear_layer_metadata``, splits the key heads and
the value heads of a Gated DeltaNet layer evenly over the tensor-parallel
ranks.  With the contiguous grouping of value heads (key head h owns value
heads [h G, (h + 1) G), G = HV / H), a contiguous run of key heads owns a
contiguous run of value heads, and the recurrence of one value head reads only
its own key head: each rank runs the unchanged prefill on its slice of q, k,
v, g, beta and the initial state, with no exchange.  Concatenating the ranks'
outputs along the head axis gives the unsharded result.
"""
from __future__ import annotations

from typing import NamedTuple, Optional

import torch


class HeadShard(NamedTuple):
    h0: int    # first key head of the rank
    h1: int    # one past its last key head
    hv0: int   # first value head
    hv1: int   # one past its last value head


def head_shard(H: int, HV: int, rank: int, world: int) -> HeadShard:
    """Contiguous key-head group of ``rank`` and the value heads it owns."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if H <= 0 or HV % H != 0:
        raise ValueError(f"HV ({HV}) must be a positive multiple of H ({H})")
    if H % world != 0:
        raise ValueError(f"{H} key heads do not split evenly over {world} ranks")
    G = HV // H
    per = H // world
    h0, h1 = rank * per, (rank + 1) * per
    return HeadShard(h0, h1, h0 * G, h1 * G)


def shard_prefill_inputs(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                         beta: torch.Tensor, initial_state: Optional[torch.Tensor], rank: int, world: int):
    """The slices of one rank: q, k [B,T,H,K] -> key heads, v [B,T,HV,V], g and
    beta [B,T,HV], initial_state [N,HV,K,V] -> value heads (contiguous copies)."""
    s = head_shard(q.shape[2], v.shape[2], rank, world)
    c = lambda t: t.contiguous()
    h0 = None if initial_state is None else c(initial_state[:, s.hv0:s.hv1])
    return (c(q[:, :, s.h0:s.h1]), c(k[:, :, s.h0:s.h1]), c(v[:, :, s.hv0:s.hv1]),
            c(g[:, :, s.hv0:s.hv1]), c(beta[:, :, s.hv0:s.hv1]), h0)
