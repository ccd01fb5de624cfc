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
                   choices=["chunk_dense", "chunk_long", "decode", "decode_bf16", "gating", "bwd_dense"])
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
