"""GPU parity of the multi-token (MTP) decode and the bf16-pool decode
against the fp64 oracle (same tolerances as the single-token decode; slots a
call must not touch are compared bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_chunk_gb300 import workloads as W
import parity_util as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_chunked_chunk_gb300 import build
    build.build()


def _gdn():
    import gated_deltanet_chunked_chunk_gb300 as gdn
    return gdn


def _mtp_inputs(seed, N, ld, H, HV, K, V, short_every=3, pad_request=None):
    """Requests of ld tokens (every short_every-th one shorter), each owning
    slots n*ld .. n*ld + ld - 1 of the pool (the LightLLM layout), a random
    number of accepted tokens in [1, ld]; fused raw gates."""
    gen = torch.Generator().manual_seed(seed)
    lens = [ld if (n % short_every) else max(1, ld - 1 - (n % ld)) for n in range(N)]
    cu = W.cu_from_lengths(lens)
    Tt = cu[-1]
    A_log, dt = W.gate_params(HV, gen)
    q = (torch.randn(Tt, H, K, generator=gen)).to(torch.bfloat16)
    k = (torch.randn(Tt, H, K, generator=gen)).to(torch.bfloat16)
    v = (torch.randn(Tt, HV, V, generator=gen)).to(torch.bfloat16)
    a = torch.randn(Tt, HV, generator=gen).to(torch.bfloat16)
    b = torch.randn(Tt, HV, generator=gen).to(torch.bfloat16)
    P_ = N * ld + 3
    pool = torch.randn(P_, HV, K, V, generator=gen) * 0.1
    slots = (torch.arange(N, dtype=torch.int32)[:, None] * ld + torch.arange(ld, dtype=torch.int32)[None, :])
    acc = torch.randint(1, ld + 1, (N,), generator=gen, dtype=torch.int32)
    read = slots.clone()
    if pad_request is not None:
        read[pad_request] = -1
    return dict(cu=torch.tensor(cu, dtype=torch.int32), q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt=dt, pool=pool,
                read=read, write=slots, acc=acc, Tt=Tt)


@pytest.mark.parametrize("N,ld,H,HV,K,V", [(16, 4, 16, 32, 128, 128), (9, 2, 2, 4, 64, 64), (5, 8, 4, 8, 128, 64)])
def test_mtp_decode_matches_oracle(N, ld, H, HV, K, V):
    x = _mtp_inputs(100 + N, N, ld, H, HV, K, V, pad_request=1)
    gdn = _gdn()
    pool = x["pool"].to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gdn.gdn_recurrent_decode_mtp(
        x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), pool, x["cu"].to(DEV), x["read"].to(DEV),
        x["write"].to(DEV), x["acc"].to(DEV), A_log=x["A_log"].to(DEV), a=x["a"].to(DEV), b=x["b"].to(DEV),
        dt_bias=x["dt"].to(DEV), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g_ref, b_ref = oracle.gating(x["A_log"], x["a"], x["b"], x["dt"])
    o_ref, pool_ref, bad = oracle.decode_mtp(x["q"], x["k"], x["v"], g_ref, b_ref, x["pool"], x["cu"].numpy(),
                                             x["read"].numpy(), x["write"].numpy(), x["acc"].numpy())
    assert bad == 0
    P.assert_o_close(o.float().cpu().numpy(), o_ref, "o (mtp)")
    pool_np = pool.cpu().numpy()
    written = set()
    for n in range(N):
        if int(x["read"][n, 0]) < 0:
            continue
        for i in range(int(x["cu"][n + 1] - x["cu"][n])):
            written.add(int(x["write"][n, i]))
    w = sorted(written)
    P.assert_state_close(pool_np[w], pool_ref[w], "written states (mtp)")
    rest = sorted(set(range(pool_np.shape[0])) - written)
    np.testing.assert_array_equal(pool_np[rest], x["pool"].numpy()[rest])   # bit-exact
    c = x["cu"]
    assert (o[c[1]:c[2]] == 0).all()                                        # the PAD request


def test_mtp_one_token_per_request_equals_single_token_decode():
    # cu = arange, ld = 1, read = write = idx: the MTP entry point must give the
    # single-token decode's results bit for bit.
    case = W.config4()
    gdn = _gdn()
    R = case.q.shape[0]
    p1 = case.ssm_pool.to(DEV)
    p2 = p1.clone()
    kw = dict(A_log=case.A_log.to(DEV), a=case.a.to(DEV), b=case.b.to(DEV), dt_bias=case.dt_bias.to(DEV))
    o1 = gdn.gdn_recurrent_decode(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV), p1, case.ssm_indices.to(DEV), **kw)
    idx2 = case.ssm_indices.to(DEV).view(R, 1).contiguous()
    o2 = gdn.gdn_recurrent_decode_mtp(case.q.to(DEV)[:, 0].contiguous(), case.k.to(DEV)[:, 0].contiguous(),
                                      case.v.to(DEV)[:, 0].contiguous(), p2,
                                      torch.arange(R + 1, dtype=torch.int32, device=DEV), idx2, idx2, None, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1[:, 0], o2)
    assert torch.equal(p1, p2)


def test_mtp_bad_counts_and_offsets_set_status():
    x = _mtp_inputs(7, 4, 3, 2, 4, 64, 64)
    gdn = _gdn()
    acc = x["acc"].clone()
    acc[2] = 0                                                              # outside [1, ld]
    cu = x["cu"].clone()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gdn.gdn_recurrent_decode_mtp(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["pool"].to(DEV), cu.to(DEV),
                                 x["read"].to(DEV), x["write"].to(DEV), acc.to(DEV), A_log=x["A_log"].to(DEV),
                                 a=x["a"].to(DEV), b=x["b"].to(DEV), dt_bias=x["dt"].to(DEV), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _gdn().DEV_BAD_SLOT
    cu[2] = cu[1] + 5                                                       # 5 tokens > ld = 3
    st.zero_()
    gdn.gdn_recurrent_decode_mtp(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["pool"].to(DEV), cu.to(DEV),
                                 x["read"].to(DEV), x["write"].to(DEV), None, A_log=x["A_log"].to(DEV),
                                 a=x["a"].to(DEV), b=x["b"].to(DEV), dt_bias=x["dt"].to(DEV), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _gdn().DEV_BAD_CU_SEQLENS


@pytest.mark.parametrize("fused", [True, False])
def test_bf16_pool_decode_matches_oracle(fused):
    case = W.config4()
    gdn = _gdn()
    pool16 = case.ssm_pool.to(torch.bfloat16)
    pool = pool16.to(DEV)
    before = pool.clone()
    g_ref, b_ref = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    if fused:
        kw = dict(A_log=case.A_log.to(DEV), a=case.a.to(DEV), b=case.b.to(DEV), dt_bias=case.dt_bias.to(DEV))
    else:
        kw = dict(g=torch.from_numpy(g_ref.astype(np.float32)).to(DEV),
                  beta=torch.from_numpy(b_ref.astype(np.float32)).to(DEV))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gdn.gdn_recurrent_decode_bf16(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV), pool,
                                      case.ssm_indices.to(DEV), dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx = case.ssm_indices.numpy()
    sample = [r for r in range(len(idx)) if idx[r] >= 0][:40] + [r for r in range(len(idx)) if idx[r] < 0][:4]
    sub_idx = np.full(len(idx), -1, np.int32)
    sub_idx[sample] = idx[sample]
    o_ref, pool_ref, _ = oracle.decode_bf16_pool(case.q, case.k, case.v, g_ref, b_ref, pool16.float().numpy(),
                                                 sub_idx)
    P.assert_o_close(o.float().cpu().numpy()[sample, 0], o_ref[sample], "o (bf16 pool)")
    slots = [int(idx[r]) for r in sample if idx[r] >= 0]
    P.assert_state_close(pool.float().cpu().numpy()[slots], pool_ref[slots], "stored bf16 states")
    untouched = sorted(set(range(case.ssm_pool.shape[0])) - {int(s) for s in idx if s >= 0})
    ut = torch.tensor(untouched, device=DEV)
    assert torch.equal(pool.index_select(0, ut), before.index_select(0, ut))
    for r in range(len(idx)):
        if idx[r] < 0:
            assert (o[r] == 0).all()


def test_mtp_skipped_and_repeated_write_slots():
    """A write slot of -1 in the middle of a request stores nothing for that
    token, and a slot written twice by one request keeps the later state (the
    kernel orders its per-token stores); every other slot stays bit-exact."""
    N, ld, H, HV, K, V = 6, 4, 2, 4, 128, 128
    x = _mtp_inputs(311, N, ld, H, HV, K, V, short_every=100)
    write = x["write"].clone()
    write[:, 1] = -1                   # token 1 of every request is not kept
    write[:, 2] = write[:, 0]          # token 2 overwrites token 0's slot
    gdn = _gdn()
    pool = x["pool"].to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gdn.gdn_recurrent_decode_mtp(
        x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), pool, x["cu"].to(DEV), x["read"].to(DEV),
        write.to(DEV), x["acc"].to(DEV), A_log=x["A_log"].to(DEV), a=x["a"].to(DEV), b=x["b"].to(DEV),
        dt_bias=x["dt"].to(DEV), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g_ref, b_ref = oracle.gating(x["A_log"], x["a"], x["b"], x["dt"])
    o_ref, pool_ref, bad = oracle.decode_mtp(x["q"], x["k"], x["v"], g_ref, b_ref, x["pool"], x["cu"].numpy(),
                                             x["read"].numpy(), write.numpy(), x["acc"].numpy())
    assert bad == 0
    P.assert_o_close(o.float().cpu().numpy(), o_ref, "o (mtp, skipped / repeated slots)")
    pool_np = pool.cpu().numpy()
    written = sorted({int(s) for s in write.flatten().tolist() if s >= 0 and
                      any(int(write[n, i]) == s for n in range(N) for i in range(int(x["cu"][n + 1] - x["cu"][n])))})
    P.assert_state_close(pool_np[written], pool_ref[written], "written states")
    for s in written:   # the kept state is the later token's, not token 0's
        n = s // ld
        if int(x["cu"][n + 1] - x["cu"][n]) >= 3:
            assert not np.allclose(pool_ref[s], x["pool"].numpy()[s])
    rest = sorted(set(range(pool_np.shape[0])) - set(written))
    np.testing.assert_array_equal(pool_np[rest], x["pool"].numpy()[rest])
