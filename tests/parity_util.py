"""Helpers shared by the GPU parity tests: feed the same seeded inputs to the
CUDA path (through the C ABI binding) and to the fp64 oracle, and compare.

Tolerances (fp64 oracle vs the bf16-in / fp32-accumulate GPU path):
  o            : relative L2 error <= 2e-3 and max abs error <= 2e-2
  final state  : max abs error <= 1e-2
  gating g/beta: |d| <= 1e-5 |ref| + 1e-6 (fp32 exp/log1p against fp64)
  slots / PAD  : bit-exact
"""
import numpy as np
import torch

import oracle

O_REL_L2 = 2e-3
O_MAX_ABS = 2e-2
STATE_MAX_ABS = 1e-2
GATE_RTOL = 1e-5
GATE_ATOL = 1e-6


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def assert_o_close(o_gpu, o_ref, what="o"):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite values"
    r = rel_l2(o_gpu, o_ref)
    m = float(np.abs(o_gpu - o_ref).max()) if o_gpu.size else 0.0
    assert r <= O_REL_L2, f"{what}: rel-L2 {r:.3e} > {O_REL_L2}"
    assert m <= O_MAX_ABS, f"{what}: max-abs {m:.3e} > {O_MAX_ABS}"
    return r, m


def assert_state_close(s_gpu, s_ref, what="final_state"):
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    assert np.isfinite(s_gpu).all(), f"{what}: non-finite values"
    m = float(np.abs(s_gpu - s_ref).max()) if s_gpu.size else 0.0
    assert m <= STATE_MAX_ABS, f"{what}: max-abs {m:.3e} > {STATE_MAX_ABS}"
    return m


def oracle_gates(case):
    """g, beta for a prefill case from the oracle's fp64 gating, rounded to fp32
    (the dtype the chunk entry point takes).  Both sides get these same values."""
    g, beta = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    shp = (case.B, case.T, case.HV)
    return (torch.from_numpy(g.astype(np.float32)).reshape(shp),
            torch.from_numpy(beta.astype(np.float32)).reshape(shp))


def to_dev(t, dev="cuda"):
    return None if t is None else t.to(dev).contiguous()


def run_chunk_gpu(case, g, beta, dev="cuda", **kw):
    import gated_deltanet_chunked_chunk_gb300 as gdn
    o, ht = gdn.gdn_chunk_fwd(to_dev(case.q, dev), to_dev(case.k, dev), to_dev(case.v, dev),
                              to_dev(g, dev), to_dev(beta, dev), scale=case.scale,
                              initial_state=to_dev(case.initial_state, dev),
                              output_final_state=case.output_final_state,
                              cu_seqlens=to_dev(case.cu_seqlens, dev),
                              use_qk_l2norm=case.use_qk_l2norm, **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), (None if ht is None else ht.cpu().numpy())


def run_chunk_oracle(case, g, beta, items=None):
    cu = None if case.cu_seqlens is None else case.cu_seqlens.numpy()
    return oracle.recurrent(case.q, case.k, case.v, g, beta, scale=case.scale,
                            initial_state=case.initial_state, cu_seqlens=cu,
                            use_qk_l2norm=case.use_qk_l2norm,
                            output_final_state=case.output_final_state, items=items)


def oracle_single_head(case, g, beta, n, hv):
    """Oracle for one (sequence, value head) of a dense or varlen case, on
    sliced inputs so that only that head is widened to fp64."""
    G = case.HV // case.H
    h = hv // G
    if case.cu_seqlens is None:
        b0, t0, t1 = n, 0, case.T
    else:
        cu = case.cu_seqlens.tolist()
        b0, t0, t1 = 0, cu[n], cu[n + 1]
    sl = slice(t0, t1)
    q = case.q[b0:b0 + 1, sl, h:h + 1]
    k = case.k[b0:b0 + 1, sl, h:h + 1]
    v = case.v[b0:b0 + 1, sl, hv:hv + 1]
    gg = g[b0:b0 + 1, sl, hv:hv + 1]
    bb = beta[b0:b0 + 1, sl, hv:hv + 1]
    h0 = None if case.initial_state is None else case.initial_state[n:n + 1, hv:hv + 1]
    scale = case.scale if case.scale is not None else 1.0 / np.sqrt(case.K)
    o, ht = oracle.recurrent(q, k, v, gg, bb, scale=scale, initial_state=h0,
                             use_qk_l2norm=case.use_qk_l2norm, output_final_state=True)
    return o[0, :, 0], ht[0, 0], (b0, sl)
