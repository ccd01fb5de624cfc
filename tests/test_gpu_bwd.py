"""GPU parity of gdn_chunk_bwd against the fp64 autograd oracle.

The GPU recomputes the forward from the same bf16 inputs and runs the
backward in fp32; the one bf16 factor it reuses from the forward is W (in the
state-gradient walk), so each gradient tensor must agree with the fp64
reference to rel-L2 <= 5e-3 (five times the bf16 rounding of W), and dh0
likewise."""
import numpy as np
import pytest
import torch

from gated_deltanet_chunked_chunk_gb300 import workloads as W
from oracle import bwd_oracle as BO
import parity_util as P

pytestmark = pytest.mark.gpu
DEV = "cuda"
BWD_REL_L2 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_chunked_chunk_gb300 import build
    build.build()


def _run(case, l2=True, with_dht=True, seed=0):
    import gated_deltanet_chunked_chunk_gb300 as gdn
    g, beta = P.oracle_gates(case)
    gen = torch.Generator().manual_seed(1000 + seed)
    do = torch.randn(case.B, case.T, case.HV, case.V, generator=gen).to(torch.bfloat16)
    dht = torch.randn(case.N, case.HV, case.K, case.V, generator=gen) if with_dht else None
    d = lambda t: None if t is None else t.to(DEV).contiguous()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_chunk_bwd(d(case.q), d(case.k), d(case.v), d(g), d(beta), d(do), initial_state=d(case.initial_state),
                            cu_seqlens=d(case.cu_seqlens), dht=d(dht), use_qk_l2norm=l2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cu = case.cu_seqlens.numpy() if case.cu_seqlens is not None else None
    ref = BO.backward(case.q.float().numpy(), case.k.float().numpy(), case.v.float().numpy(), g.numpy(),
                      beta.numpy(), do.float().numpy(), initial_state=None if case.initial_state is None
                      else case.initial_state.numpy(), cu_seqlens=cu,
                      dht=None if dht is None else dht.numpy(), use_qk_l2norm=l2)
    names = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]
    for name, gpu, r in zip(names, out, ref):
        if r is None:
            assert gpu is None
            continue
        x = gpu.cpu().numpy().astype(np.float64)
        assert np.isfinite(x).all(), name
        err = P.rel_l2(x, r)
        assert err <= BWD_REL_L2, f"{name}: rel-L2 {err:.3e}"


def test_bwd_small_gva_ragged():
    case = W.prefill_case("bwd_small", 41, 1, 200, 2, 4, 64, 64, init="all")
    _run(case, seed=1)


def test_bwd_k128_two_sequences():
    case = W.prefill_case("bwd_k128", 42, 2, 130, 2, 4, 128, 128, init="all")
    _run(case, seed=2)


def test_bwd_without_l2norm_or_state_gradients():
    # Without the norm, N(0, 1) keys of dimension 64 (|k|^2 ~ 64) make the
    # recurrence explosive; keys and queries scaled by 1/8 (exact in bf16) keep
    # |k| near 1, as normalised inputs would be.
    case = W.prefill_case("bwd_nol2", 43, 1, 96, 1, 2, 64, 128, init="none")
    case.q = case.q * 0.125
    case.k = case.k * 0.125
    _run(case, l2=False, with_dht=False, seed=3)


def test_bwd_varlen_with_empty_sequence():
    lengths = [70, 0, 5, 64]
    case = W.prefill_case("bwd_var", 44, 1, sum(lengths), 2, 4, 128, 64, init="all",
                          cu_seqlens=W.cu_from_lengths(lengths))
    _run(case, seed=4)


def test_bwd_qwen_heads_sampled_group():
    # H=16, HV=32, K=V=128, T=1024 with initial and final-state gradients; the
    # oracle runs on one key-head group (key head 5, value heads 10 and 11),
    # whose gradients do not depend on the other heads.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    case = W.prefill_case("bwd_qwen", 45, 1, 1024, 16, 32, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    gen = torch.Generator().manual_seed(1045)
    do = torch.randn(1, 1024, 32, 128, generator=gen).to(torch.bfloat16)
    dht = torch.randn(1, 32, 128, 128, generator=gen)
    d = lambda t: t.to(DEV).contiguous()
    out = gdn.gdn_chunk_bwd(d(case.q), d(case.k), d(case.v), d(g), d(beta), d(do), initial_state=d(case.initial_state),
                            dht=d(dht))
    torch.cuda.synchronize()
    h, hv = 5, slice(10, 12)
    ref = BO.backward(case.q[:, :, h:h + 1].float().numpy(), case.k[:, :, h:h + 1].float().numpy(),
                      case.v[:, :, hv].float().numpy(), g[:, :, hv].numpy(), beta[:, :, hv].numpy(),
                      do[:, :, hv].float().numpy(), initial_state=case.initial_state[:, hv].numpy(),
                      dht=dht[:, hv].numpy(), use_qk_l2norm=True, scale=1.0 / np.sqrt(128))
    gpu = [out[0][:, :, h:h + 1], out[1][:, :, h:h + 1], out[2][:, :, hv], out[3][:, :, hv], out[4][:, :, hv],
           out[5][:, hv]]
    for name, x, r in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], gpu, ref):
        err = P.rel_l2(x.cpu().numpy().astype(np.float64), r)
        assert err <= BWD_REL_L2, f"{name}: rel-L2 {err:.3e}"


def test_bwd_varlen_many_sequences():
    # 120 sequences of 0..80 tokens: the chunk-start table in the backward kernels.
    rng = np.random.default_rng(46)
    lens = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(1, 81, 120)]
    case = W.prefill_case("bwd_many", 46, 1, sum(lens), 1, 2, 64, 64, init="all",
                          cu_seqlens=W.cu_from_lengths(lens))
    _run(case, seed=6)


def test_bwd_k128_varlen_short_sequences():
    # K = 128 takes the tcgen05 state-gradient walk: 40 packed sequences of
    # 0..150 tokens, so most chunks are partial and the rows past a sequence's
    # end that the walk's tile loads bring in belong to the next sequence.
    rng = np.random.default_rng(47)
    lens = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 151, 40)]
    case = W.prefill_case("bwd_k128_var", 47, 1, sum(lens), 2, 4, 128, 128, init="even",
                          cu_seqlens=W.cu_from_lengths(lens))
    _run(case, seed=7)


def test_bwd_k128_without_l2norm_or_state_gradients():
    # The tcgen05 state-gradient walk with raw keys and queries (no norm, no
    # initial state, no final-state gradient); dimension 128 keys scaled by
    # 1/16 (exact in bf16) keep |k| near 0.7.
    case = W.prefill_case("bwd_nol2_k128", 48, 1, 200, 2, 4, 128, 128, init="none")
    case.q = case.q * 0.0625
    case.k = case.k * 0.0625
    _run(case, l2=False, with_dht=False, seed=8)


@pytest.mark.parametrize("K,varlen", [(64, True), (128, True), (128, False)])
def test_bwd_four_value_heads_per_key_head_and_repeatable(K, varlen):
    # Each value head's dq, dk share is stored on its own and the three later
    # ones are added in head order: parity with the oracle, and a second call
    # on the same inputs returns the same bits in every output.  Dense input
    # takes no memsets: every row of dq, dk and of the shares is written.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    lengths = [70, 1, 130, 64]
    if varlen:
        case = W.prefill_case("bwd_g4", 49, 1, sum(lengths), 1, 4, K, 128, init="all",
                              cu_seqlens=W.cu_from_lengths(lengths))
    else:
        case = W.prefill_case("bwd_g4_dense", 50, 2, 133, 1, 4, K, 128, init="all")
    _run(case, seed=9)
    g, beta = P.oracle_gates(case)
    gen = torch.Generator().manual_seed(1009)
    do = torch.randn(case.B, case.T, case.HV, case.V, generator=gen).to(torch.bfloat16).to(DEV)
    dht = torch.randn(case.N, case.HV, case.K, case.V, generator=gen).to(DEV)
    d = lambda t: t.to(DEV).contiguous()
    args = (d(case.q), d(case.k), d(case.v), d(g), d(beta), do)
    kw = dict(initial_state=d(case.initial_state), dht=dht,
              cu_seqlens=None if case.cu_seqlens is None else d(case.cu_seqlens))
    first = gdn.gdn_chunk_bwd(*args, **kw)
    second = gdn.gdn_chunk_bwd(*args, **kw)
    for a, b in zip(first, second):
        assert torch.equal(a, b)


def test_bwd_long_single_sequence_matches_batched_bitwise():
    # One sequence of 71 chunks: the recomputed forward takes the chunk ranges
    # (each range's walk saving its own chunks' states).  The same sequence as
    # the first of a batch of two recomputes in one range: the same gradients,
    # bit for bit (the one-range path is the one the oracle tests above pin).
    import gated_deltanet_chunked_chunk_gb300 as gdn
    T = 64 * 70 + 20
    case = W.prefill_case("bwd_long", 51, 1, T, 2, 4, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    gen = torch.Generator().manual_seed(1051)
    do = torch.randn(1, T, 4, 128, generator=gen).to(torch.bfloat16)
    dht = torch.randn(1, 4, 128, 128, generator=gen)
    d = lambda t: t.to(DEV).contiguous()
    two = lambda t: torch.cat([t, t.flip(1)], 0)
    one = gdn.gdn_chunk_bwd(d(case.q), d(case.k), d(case.v), d(g), d(beta), d(do),
                            initial_state=d(case.initial_state), dht=d(dht))
    both = gdn.gdn_chunk_bwd(d(two(case.q)), d(two(case.k)), d(two(case.v)), d(two(g)), d(two(beta)), d(two(do)),
                             initial_state=d(torch.cat([case.initial_state] * 2, 0)), dht=d(torch.cat([dht] * 2, 0)))
    torch.cuda.synchronize()
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], one, both):
        assert torch.equal(a, b[:1]), name
    assert gdn.chunk_fwd_kernel_launches(1, T, 2, 4, 128, 128, 1, False) == 4


def test_bwd_maximum_sequence_count_sampled():
    # 65535 packed sequences of 0 to 3 tokens (the largest count the grids
    # take), each with its own initial state and final-state gradient: sampled
    # sequences against the oracle run on that sequence alone.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    N = 65535
    rng = np.random.default_rng(62)
    lens = [int(x) for x in rng.integers(0, 4, N)]
    cu = W.cu_from_lengths(lens)
    case = W.prefill_case("bwd_max_n", 62, 1, cu[-1], 1, 1, 64, 64, cu_seqlens=cu, init="all")
    g, beta = P.oracle_gates(case)
    gen = torch.Generator().manual_seed(1062)
    do = torch.randn(1, case.T, 1, 64, generator=gen).to(torch.bfloat16)
    dht = torch.randn(N, 1, 64, 64, generator=gen)
    d = lambda t: t.to(DEV).contiguous()
    out = gdn.gdn_chunk_bwd(d(case.q), d(case.k), d(case.v), d(g), d(beta), d(do),
                            initial_state=d(case.initial_state), cu_seqlens=d(case.cu_seqlens), dht=d(dht))
    torch.cuda.synchronize()
    dq, dk, dv, dg, db, dh0 = [x.cpu().numpy().astype(np.float64) for x in out]
    picks = [0, 1, 2, 3, 77, 32767, N - 2, N - 1] + [int(x) for x in rng.integers(0, N, 24)]
    checked = 0
    for n in picks:
        t0, t1 = cu[n], cu[n + 1]
        if t1 == t0:
            continue
        sl = slice(t0, t1)
        ref = BO.backward(case.q[:, sl].float().numpy(), case.k[:, sl].float().numpy(), case.v[:, sl].float().numpy(),
                          g[:, sl].numpy(), beta[:, sl].numpy(), do[:, sl].float().numpy(),
                          initial_state=case.initial_state[n:n + 1].numpy(), dht=dht[n:n + 1].numpy(),
                          use_qk_l2norm=True)
        got = [dq[:, sl], dk[:, sl], dv[:, sl], dg[:, sl], db[:, sl], dh0[n:n + 1]]
        for name, x, r in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], got, ref):
            err = P.rel_l2(x, r)
            assert err <= BWD_REL_L2, f"seq {n} {name}: rel-L2 {err:.3e}"
        checked += 1
    assert checked >= 20
