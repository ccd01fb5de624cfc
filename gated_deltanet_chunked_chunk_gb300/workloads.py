"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers; it holds none of the method's
arithmetic (no gating, no normalisation, no recurrence).  The raw gate inputs
(A_log, a, dt_bias, b) are returned as drawn; turning them into g and beta is
the job of the library's gating entry point or of the oracle.

Recipes (shapes follow the workloads of the FastDeploy PR "support fla triton
kernel for qwen3.5", Usage sections 1, 2 and 5, and the LightLLM "gdn.py"
prefill/decode paths; value distributions are this library's synthetic
stand-ins, since the pages run no public dataset for the kernel):

* q, k, v ~ N(0, 1), cast to bf16.
* A_log[h] = log U(1, 16); a ~ N(0, 1) (bf16); dt_bias[h] = log(expm1(U(1e-3, 0.1)));
  b ~ N(0, 1) (bf16).
* states ~ N(0, 0.1^2) in fp32 (0.1 read as the standard deviation).
* everything is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
  in float32 and then cast, in a fixed order, so every machine gets the same bits.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass
class PrefillCase:
    name: str
    q: torch.Tensor          # [B,T,H,K] bf16
    k: torch.Tensor          # [B,T,H,K] bf16
    v: torch.Tensor          # [B,T,HV,V] bf16
    A_log: torch.Tensor      # [HV] fp32
    a: torch.Tensor          # [B*T,HV] bf16  (token-major)
    b: torch.Tensor          # [B*T,HV] bf16
    dt_bias: torch.Tensor    # [HV] fp32
    initial_state: Optional[torch.Tensor]  # [N,HV,K,V] fp32 or None
    cu_seqlens: Optional[torch.Tensor]     # [N+1] int32 or None
    scale: Optional[float]
    use_qk_l2norm: bool = True
    output_final_state: bool = True

    @property
    def B(self): return self.q.shape[0]
    @property
    def T(self): return self.q.shape[1]
    @property
    def H(self): return self.q.shape[2]
    @property
    def K(self): return self.q.shape[3]
    @property
    def HV(self): return self.v.shape[2]
    @property
    def V(self): return self.v.shape[3]
    @property
    def N(self): return self.B if self.cu_seqlens is None else self.cu_seqlens.numel() - 1
    @property
    def tokens(self): return self.B * self.T


@dataclasses.dataclass
class DecodeCase:
    name: str
    q: torch.Tensor          # [R,1,H,K] bf16
    k: torch.Tensor          # [R,1,H,K] bf16
    v: torch.Tensor          # [R,1,HV,V] bf16
    A_log: torch.Tensor      # [HV] fp32
    a: torch.Tensor          # [R,HV] bf16
    b: torch.Tensor          # [R,HV] bf16
    dt_bias: torch.Tensor    # [HV] fp32
    ssm_pool: torch.Tensor   # [P,HV,K,V] fp32
    ssm_indices: torch.Tensor  # [R] int32, -1 = PAD
    scale: Optional[float] = None
    use_qk_l2norm: bool = True

    @property
    def R(self): return self.q.shape[0]
    @property
    def H(self): return self.q.shape[2]
    @property
    def K(self): return self.q.shape[3]
    @property
    def HV(self): return self.v.shape[2]
    @property
    def V(self): return self.v.shape[3]
    @property
    def P(self): return self.ssm_pool.shape[0]


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def gate_params(HV: int, gen: torch.Generator):
    """A_log = log U(1,16) and dt_bias = log(expm1(U(1e-3, 0.1))), per value head."""
    A_log = torch.log(torch.empty(HV).uniform_(1.0, 16.0, generator=gen))
    u = torch.empty(HV, dtype=torch.float64).uniform_(1e-3, 0.1, generator=gen)
    dt_bias = torch.log(torch.expm1(u)).to(torch.float32)
    return A_log.float(), dt_bias


def _normal(shape, gen, std=1.0, dtype=torch.bfloat16):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def prefill_case(name: str, seed: int, B: int, T: int, H: int, HV: int, K: int, V: int,
                 cu_seqlens=None, init: str = "none", scale=None,
                 use_qk_l2norm: bool = True, output_final_state: bool = True) -> PrefillCase:
    """Generic seeded prefill case.  init: 'none', 'all' or 'even' (sequences
    0, 2, 4, ... get N(0, 0.1^2) states, the others explicit zeros)."""
    gen = _gen(seed)
    A_log, dt_bias = gate_params(HV, gen)
    q = _normal((B, T, H, K), gen)
    k = _normal((B, T, H, K), gen)
    v = _normal((B, T, HV, V), gen)
    a = _normal((B * T, HV), gen)
    b = _normal((B * T, HV), gen)
    cu = None
    N = B
    if cu_seqlens is not None:
        cu = torch.as_tensor(cu_seqlens, dtype=torch.int32)
        N = cu.numel() - 1
    h0 = None
    if init in ("all", "even"):
        h0 = _normal((N, HV, K, V), gen, std=0.1, dtype=torch.float32)
        if init == "even":
            h0[1::2] = 0.0
    return PrefillCase(name, q, k, v, A_log, a, b, dt_bias, h0, cu, scale,
                       use_qk_l2norm, output_final_state)


def varlen_lengths(seed: int, n: int, lo: int, hi: int, avoid_multiple: int = 64):
    """n lengths ~ U[lo, hi] (integers), each redrawn while it is a multiple of
    ``avoid_multiple`` (so every sequence ends in a ragged chunk)."""
    gen = _gen(seed + 1000)
    out = []
    while len(out) < n:
        x = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        if avoid_multiple and x % avoid_multiple == 0:
            continue
        out.append(x)
    return out


def cu_from_lengths(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return cu


# --- the five named workloads ----------------------------------------------

def config0() -> PrefillCase:
    """Tiny chunk forward: B=1, T=256, H=HV=2, K=V=64, no initial state, seed 0."""
    return prefill_case("tiny_T256_H2_K64", 0, 1, 256, 2, 2, 64, 64, init="none")


def config1() -> PrefillCase:
    """Dense prefill: B=2, T=4096, H=16, HV=32, K=V=128, initial state, seed 1."""
    return prefill_case("dense_B2_T4096_H16_HV32_K128", 1, 2, 4096, 16, 32, 128, 128, init="all")


def config2() -> PrefillCase:
    """Varlen packed prefill: 8 sequences, lengths U[64, 8192] (never a multiple
    of 64), B=1 with cu_seqlens; states for sequences 0, 2, 4, 6; seed 2."""
    lengths = varlen_lengths(2, 8, 64, 8192)
    cu = cu_from_lengths(lengths)
    return prefill_case("varlen_8seq_H16_HV32_K128", 2, 1, cu[-1], 16, 32, 128, 128,
                        cu_seqlens=cu, init="even")


def config3() -> PrefillCase:
    """Long-context prefill: B=1, T=65536, H=16, HV=32, K=V=128, states in and out; seed 3."""
    return prefill_case("long_T65536_H16_HV32_K128", 3, 1, 65536, 16, 32, 128, 128, init="all")


def decode_case(name: str, seed: int, R: int, P: int, H: int, HV: int, K: int, V: int,
                pad_prob: float = 0.1) -> DecodeCase:
    """R one-token requests against a pool of P slots.  Slots are the first R
    entries of a random permutation of the P slots; each is replaced by -1
    (PAD) with probability ``pad_prob`` (seeded Bernoulli)."""
    gen = _gen(seed)
    A_log, dt_bias = gate_params(HV, gen)
    q = _normal((R, 1, H, K), gen)
    k = _normal((R, 1, H, K), gen)
    v = _normal((R, 1, HV, V), gen)
    a = _normal((R, HV), gen)
    b = _normal((R, HV), gen)
    perm = torch.randperm(P, generator=gen)[:R].to(torch.int32)
    pad = torch.rand(R, generator=gen) < pad_prob
    idx = torch.where(pad, torch.full_like(perm, -1), perm)
    pool = _normal((P, HV, K, V), gen, std=0.1, dtype=torch.float32)
    return DecodeCase(name, q, k, v, A_log, a, b, dt_bias, pool, idx)


def config4() -> DecodeCase:
    """Batched decode: 256 requests, pool [512,32,128,128] fp32, ~10% PAD; seed 4."""
    return decode_case("decode_R256_P512_H16_HV32_K128", 4, 256, 512, 16, 32, 128, 128)


CONFIGS = {0: config0, 1: config1, 2: config2, 3: config3, 4: config4}


# ---------------------------------------------------------------- causal conv1d
# Shapes follow the FastDeploy PR's Usage sections 3 and 4 (x channel-first
# [dim, total] for prefill, token-major [batch, dim] for decode, a conv-state
# pool [slots, dim, state_len]) with dim = 2 H K + HV V, the packed q | k | v
# channels of the LightLLM "gdn.py" backends, and width 4.  Draws: x ~ N(0, 1),
# weight ~ U(-0.5, 0.5), bias ~ N(0, 0.1^2), states ~ N(0, 1), all bf16.


@dataclasses.dataclass
class ConvPrefillCase:
    name: str
    x: torch.Tensor                # [dim, total] bf16
    weight: torch.Tensor           # [dim, W] bf16
    bias: torch.Tensor             # [dim] bf16
    conv_states: torch.Tensor      # [P, dim, S] bf16
    query_start_loc: torch.Tensor  # [N + 1] int32
    cache_indices: torch.Tensor    # [N] int32 (-1 = no slot)
    has_initial_state: torch.Tensor  # [N] bool


@dataclasses.dataclass
class ConvDecodeCase:
    name: str
    x: torch.Tensor                # [R, dim] bf16
    weight: torch.Tensor           # [dim, W] bf16
    bias: torch.Tensor             # [dim] bf16
    conv_state: torch.Tensor       # [P, dim, S] bf16
    indices: torch.Tensor          # [R] int32 (-1 = PAD)


def _uniform(shape, gen, lo, hi):
    return (torch.rand(shape, generator=gen) * (hi - lo) + lo).to(torch.bfloat16)


def conv_prefill_case(name: str, seed: int, dim: int, lengths, W: int = 4, S: int = 3, P: Optional[int] = None,
                      init_every: int = 2, pad_slot_every: int = 0) -> ConvPrefillCase:
    """Packed sequences of the given lengths.  Sequence n uses slot P - 1 - n
    (so slots are not the identity); every ``init_every``-th sequence starts
    from its slot's state; with ``pad_slot_every`` > 0 every such sequence has
    slot -1."""
    gen = _gen(seed)
    N = len(lengths)
    P = P if P is not None else N + 2
    total = int(sum(lengths))
    x = _normal((dim, total), gen)
    weight = _uniform((dim, W), gen, -0.5, 0.5)
    bias = _normal((dim,), gen, std=0.1)
    states = _normal((P, dim, S), gen)
    qsl = torch.tensor(cu_from_lengths(lengths), dtype=torch.int32)
    slots = torch.tensor([P - 1 - n for n in range(N)], dtype=torch.int32)
    if pad_slot_every:
        for n in range(0, N, pad_slot_every):
            slots[n] = -1
    init = torch.tensor([(n % init_every) == 0 for n in range(N)], dtype=torch.bool)
    return ConvPrefillCase(name, x, weight, bias, states, qsl, slots, init)


def conv_decode_case(name: str, seed: int, R: int, P: int, dim: int, W: int = 4, S: int = 3,
                     pad_prob: float = 0.1) -> ConvDecodeCase:
    """R one-token requests; slots are the first R entries of a permutation of
    the P slots, each replaced by -1 (PAD) with probability ``pad_prob``."""
    gen = _gen(seed)
    x = _normal((R, dim), gen)
    weight = _uniform((dim, W), gen, -0.5, 0.5)
    bias = _normal((dim,), gen, std=0.1)
    states = _normal((P, dim, S), gen)
    perm = torch.randperm(P, generator=gen)[:R].to(torch.int32)
    pad = torch.rand(R, generator=gen) < pad_prob
    idx = torch.where(pad, torch.full_like(perm, -1), perm)
    return ConvDecodeCase(name, x, weight, bias, states, idx)


def conv_prefill_long() -> ConvPrefillCase:
    """The long-context prefill's conv: dim = 2*16*128 + 32*128 = 8192 channels,
    one 65536-token sequence with an initial state; seed 13."""
    return conv_prefill_case("conv_prefill_T65536_dim8192", 13, 8192, [65536], init_every=1, P=4)


def conv_decode_r256() -> ConvDecodeCase:
    """The batched decode's conv: 256 requests, 512 slots, dim 8192; seed 14."""
    return conv_decode_case("conv_decode_R256_P512_dim8192", 14, 256, 512, 8192)
