"""Run one entry point on a seeded workload a few times (a target for ncu).

    python -m gated_deltanet_chunked_chunk_gb300.profile_case --case chunk_dense --reps 3

Cases:
  chunk_dense : B=2, T=4096, H=16, HV=32, K=V=128 with initial/final state
                (about 230 MB of inputs and outputs, above the 129 MB L2)
  chunk_long  : B=1, T=65536, H=16, HV=32, K=V=128 (the benchmark workload)
  decode      : 256 requests against a [512, 32, 128, 128] fp32 pool, fused gating
  decode_bf16 : the same against a bf16 pool
  gating      : 524288 x 32 gates
  bwd_dense   : gdn_chunk_bwd on the chunk_dense workload (initial state, final-state gradient)
  conv        : causal conv1d prefill, 8192 channels x 16384 tokens with an initial state
  mtp         : multi-token decode, 64 requests x 4 tokens against a [256, 32, 128, 128] fp32 pool
"""
from __future__ import annotations

import argparse

import torch

import gated_deltanet_chunked_chunk_gb300 as gdn
from gated_deltanet_chunked_chunk_gb300 import build as gbuild
from gated_deltanet_chunked_chunk_gb300 import workloads as W


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--case", default="chunk_dense",
                   choices=["chunk_dense", "chunk_long", "decode", "decode_bf16", "gating", "bwd_dense",
                            "conv", "mtp"])
    p.add_argument("--reps", type=int, default=3)
    args = p.parse_args()
    gbuild.build()
    dev = torch.device("cuda", 0)
    d = lambda t: None if t is None else t.to(dev).contiguous()
    if args.case.startswith("chunk"):
        case = W.config1() if args.case == "chunk_dense" else W.config3()
        g, beta = gdn.gdn_gating(d(case.A_log), d(case.a), d(case.b), d(case.dt_bias))
        q, k, v, h0 = d(case.q), d(case.k), d(case.v), d(case.initial_state)
        g = g.view(case.B, case.T, case.HV)
        beta = beta.view(case.B, case.T, case.HV)
        for _ in range(args.reps):
            gdn.gdn_chunk_fwd(q, k, v, g, beta, initial_state=h0)
    elif args.case == "bwd_dense":
        case = W.config1()
        g, beta = gdn.gdn_gating(d(case.A_log), d(case.a), d(case.b), d(case.dt_bias))
        g = g.view(case.B, case.T, case.HV)
        beta = beta.view(case.B, case.T, case.HV)
        gen = torch.Generator().manual_seed(31)
        do = d(torch.randn(case.B, case.T, case.HV, case.V, generator=gen).to(torch.bfloat16))
        dht = d(torch.randn(case.N, case.HV, case.K, case.V, generator=gen))
        q, k, v, h0 = d(case.q), d(case.k), d(case.v), d(case.initial_state)
        for _ in range(args.reps):
            gdn.gdn_chunk_bwd(q, k, v, g, beta, do, initial_state=h0, dht=dht)
    elif args.case in ("decode", "decode_bf16"):
        dc = W.config4()
        if args.case == "decode":
            pool = d(dc.ssm_pool)
            fn = gdn.gdn_recurrent_decode
        else:
            pool = d(dc.ssm_pool.to(torch.bfloat16))
            fn = gdn.gdn_recurrent_decode_bf16
        for _ in range(args.reps):
            fn(d(dc.q), d(dc.k), d(dc.v), pool, d(dc.ssm_indices),
               A_log=d(dc.A_log), a=d(dc.a), b=d(dc.b), dt_bias=d(dc.dt_bias))
    elif args.case == "conv":
        # dim 8192 (packed q | k | v of the long prefill) x 16384 tokens: 0.5 GB in + out
        pc = W.conv_prefill_case("conv_profile_T16384_dim8192", 13, 8192, [16384], init_every=1, P=4)
        x, w, bias, st = d(pc.x), d(pc.weight), d(pc.bias), d(pc.conv_states)
        qsl, ci, hi = d(pc.query_start_loc), d(pc.cache_indices), d(pc.has_initial_state)
        out = torch.empty_like(x)
        for _ in range(args.reps):
            gdn.gdn_causal_conv1d_fwd(x, w, bias, st, qsl, ci, hi, out=out)
    elif args.case == "mtp":
        # 64 requests x 4 tokens against a [256, 32, 128, 128] fp32 pool (0.5 GB)
        N, ld, H, HV, K, V = 64, 4, 16, 32, 128, 128
        gen = torch.Generator().manual_seed(24)
        Tt = N * ld
        qm = d(torch.randn(Tt, H, K, generator=gen).to(torch.bfloat16))
        km = d(torch.randn(Tt, H, K, generator=gen).to(torch.bfloat16))
        vm = d(torch.randn(Tt, HV, V, generator=gen).to(torch.bfloat16))
        am = d(torch.randn(Tt, HV, generator=gen).to(torch.bfloat16))
        bm = d(torch.randn(Tt, HV, generator=gen).to(torch.bfloat16))
        A_log = d(torch.zeros(HV))
        dt = d(torch.zeros(HV))
        pool = torch.randn(N * ld, HV, K, V, generator=gen).mul_(0.1).to(dev)
        slots = d(torch.arange(N, dtype=torch.int32)[:, None] * ld + torch.arange(ld, dtype=torch.int32)[None, :])
        cu = d(torch.arange(0, Tt + 1, ld, dtype=torch.int32))
        acc = d(torch.full((N,), 2, dtype=torch.int32))
        for _ in range(args.reps):
            gdn.gdn_recurrent_decode_mtp(qm, km, vm, pool, cu, slots, slots, acc, A_log=A_log, a=am, b=bm,
                                         dt_bias=dt)
    else:
        n, HV = 65536 * 8, 32
        gen = torch.Generator().manual_seed(5)
        a = d(torch.randn(n, HV, generator=gen).to(torch.bfloat16))
        b = d(torch.randn(n, HV, generator=gen).to(torch.bfloat16))
        z = torch.zeros(HV, device=dev)
        for _ in range(args.reps):
            gdn.gdn_gating(z, a, b, z)
    torch.cuda.synchronize()
    print(f"profile_case {args.case}: {args.reps} reps done")


if __name__ == "__main__":
    main()
