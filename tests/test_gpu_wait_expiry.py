"""The failure path of the bounded waits, driven on the GPU without a fault.

The testing hook gdn_testing_force_wait_expiry makes the first bounded wait of
every block wait on a barrier that nothing completes, with a limit of a few
thousand cycles, so it runs out every time.  The block must then wait (with
the normal limit) for its own copies in flight, write nothing to the state
pool, report GDN_DEV_WAIT_TIMEOUT through dev_status, and leave the context
usable: the next normal call passes parity.  Nothing here traps or hangs."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_chunk_gb300 import workloads as W
import parity_util as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_chunked_chunk_gb300 import build
    build.build()


def _gdn():
    import gated_deltanet_chunked_chunk_gb300 as gdn
    return gdn


def _decode(case, pool, st):
    kw = dict(A_log=case.A_log.cuda(), a=case.a.cuda(), b=case.b.cuda(), dt_bias=case.dt_bias.cuda())
    return _gdn().gdn_recurrent_decode(case.q.cuda(), case.k.cuda(), case.v.cuda(), pool,
                                       case.ssm_indices.cuda(), dev_status=st, **kw)


def test_decode_wait_expiry_reports_and_writes_nothing():
    gdn = _gdn()
    case = W.decode_case("expire", 91, 24, 40, 2, 4, 128, 128, pad_prob=0.2)
    pool = case.ssm_pool.cuda()
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = gdn.testing_force_wait_expiry(True)
    try:
        _decode(case, pool, st)
        torch.cuda.synchronize()
    finally:
        gdn.testing_force_wait_expiry(prev)
    status = int(st.item())
    assert status & gdn.DEV_WAIT_TIMEOUT
    assert not status & gdn.DEV_DRAIN_TIMEOUT      # every copy in flight drained
    assert torch.equal(pool, before)               # no block wrote its state
    # the context is still usable and a normal call right after passes parity
    st.zero_()
    o = _decode(case, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g_ref, b_ref = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    o_ref, pool_ref, bad = oracle.decode(case.q, case.k, case.v, g_ref, b_ref, case.ssm_pool,
                                         case.ssm_indices.numpy())
    assert bad == 0
    P.assert_o_close(o.float().cpu().numpy()[:, 0], o_ref)
    P.assert_state_close(pool.cpu().numpy(), pool_ref, what="pool")


def test_mtp_decode_wait_expiry_reports_and_writes_nothing():
    gdn = _gdn()
    N, ld, H, HV, K, V = 5, 3, 2, 4, 64, 64
    gen = torch.Generator().manual_seed(92)
    cu = torch.tensor(W.cu_from_lengths([ld] * N), dtype=torch.int32)
    Tt = int(cu[-1])
    q = torch.randn(Tt, H, K, generator=gen).to(torch.bfloat16)
    k = torch.randn(Tt, H, K, generator=gen).to(torch.bfloat16)
    v = torch.randn(Tt, HV, V, generator=gen).to(torch.bfloat16)
    g = -torch.rand(Tt, HV, generator=gen)
    b = torch.rand(Tt, HV, generator=gen)
    slots = (torch.arange(N, dtype=torch.int32)[:, None] * ld + torch.arange(ld, dtype=torch.int32)[None])
    pool = (torch.randn(N * ld, HV, K, V, generator=gen) * 0.1).cuda()
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = gdn.testing_force_wait_expiry(True)
    try:
        gdn.gdn_recurrent_decode_mtp(q.cuda(), k.cuda(), v.cuda(), pool, cu.cuda(), slots.cuda(), slots.cuda(),
                                     None, g=g.cuda(), beta=b.cuda(), dev_status=st)
        torch.cuda.synchronize()
    finally:
        gdn.testing_force_wait_expiry(prev)
    assert int(st.item()) & gdn.DEV_WAIT_TIMEOUT
    assert not int(st.item()) & gdn.DEV_DRAIN_TIMEOUT
    assert torch.equal(pool, before)


def test_chunk_fwd_wait_expiry_reports_and_writes_no_state():
    """The state walk of the prefill with its first wait forced to run out: the
    walk drains its loads and products, writes no final state, reports the
    expiry, and the next normal call is correct."""
    gdn = _gdn()
    case = W.prefill_case("expire_chunk", 93, 1, 300, 2, 4, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    d = lambda t: t.cuda().contiguous()
    q, k, v, gg, bb, h0 = map(d, (case.q, case.k, case.v, g, beta, case.initial_state))
    ht = torch.full_like(h0, 12345.0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = gdn.testing_force_wait_expiry(True)
    try:
        gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, final_state=ht, dev_status=st)
        torch.cuda.synchronize()
    finally:
        gdn.testing_force_wait_expiry(prev)
    assert int(st.item()) & gdn.DEV_WAIT_TIMEOUT
    assert not int(st.item()) & gdn.DEV_DRAIN_TIMEOUT
    assert bool((ht == 12345.0).all())
    st.zero_()
    o, ht2 = gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, ht_ref = P.run_chunk_oracle(case, g, beta)
    P.assert_o_close(o.float().cpu().numpy(), o_ref)
    P.assert_state_close(ht2.cpu().numpy(), ht_ref)
