"""GPU parity of gdn_recurrent_decode and gdn_gating against the fp64 oracle."""
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


# ----------------------------------------------------------------- gating ---

@pytest.mark.parametrize("Ttok,HV", [(1, 32), (7, 3), (256, 32), (1001, 6), (65536, 32)])
def test_gating_matches_oracle(Ttok, HV):
    gen = torch.Generator().manual_seed(Ttok * 31 + HV)
    A_log, dt = W.gate_params(HV, gen)
    a = (torch.randn(Ttok, HV, generator=gen) * 4).to(torch.bfloat16)
    b = (torch.randn(Ttok, HV, generator=gen) * 4).to(torch.bfloat16)
    g, beta = _gdn().gdn_gating(A_log.cuda(), a.cuda(), b.cuda(), dt.cuda())
    torch.cuda.synchronize()
    g_ref, b_ref = oracle.gating(A_log, a, b, dt)
    np.testing.assert_allclose(g.cpu().numpy(), g_ref, rtol=P.GATE_RTOL, atol=P.GATE_ATOL)
    np.testing.assert_allclose(beta.cpu().numpy(), b_ref, rtol=P.GATE_RTOL, atol=P.GATE_ATOL)


def test_gating_closed_forms_on_gpu():
    A_log = torch.tensor([0.0, np.log(2.0)], dtype=torch.float32)
    dt = torch.tensor([0.0, -0.25], dtype=torch.float32)
    a = torch.tensor([[0.0, 0.25], [20.5, 0.25]], dtype=torch.bfloat16)
    b = torch.tensor([[0.0, 0.0], [0.0, 0.0]], dtype=torch.bfloat16)
    g, beta = _gdn().gdn_gating(A_log.cuda(), a.cuda(), b.cuda(), dt.cuda())
    g = g.cpu().numpy()
    np.testing.assert_allclose(g[0], [-np.log(2.0), -2 * np.log(2.0)], rtol=1e-6)
    assert g[1, 0] == np.float32(-20.5)
    assert (beta.cpu().numpy() == 0.5).all()


# ----------------------------------------------------------------- decode ---

def _decode_check(case, fused, sample=None):
    gdn = _gdn()
    dev = "cuda"
    pool = case.ssm_pool.to(dev)
    pool_before = pool.clone()
    idx = case.ssm_indices.to(dev)
    g_ref, b_ref = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    kw = {}
    if fused:
        kw = dict(A_log=case.A_log.to(dev), a=case.a.to(dev), b=case.b.to(dev), dt_bias=case.dt_bias.to(dev))
    else:
        kw = dict(g=torch.from_numpy(g_ref.astype(np.float32)).to(dev),
                  beta=torch.from_numpy(b_ref.astype(np.float32)).to(dev))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o = gdn.gdn_recurrent_decode(case.q.to(dev), case.k.to(dev), case.v.to(dev), pool, idx,
                                 dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx_l = case.ssm_indices.tolist()
    valid = [s for s in idx_l if s >= 0]
    # untouched slots (never referenced) are bit-exact
    untouched = sorted(set(range(case.P)) - set(valid))
    ut = torch.tensor(untouched, device=dev, dtype=torch.long)
    assert torch.equal(pool.index_select(0, ut), pool_before.index_select(0, ut))
    o_np = o.float().cpu().numpy()[:, 0]
    for r, s in enumerate(idx_l):
        if s < 0:
            assert (o_np[r] == 0).all()
    rows = [r for r, s in enumerate(idx_l) if s >= 0]
    if sample is not None:
        rows = rows[:: max(1, len(rows) // sample)][:sample]
    sl = torch.tensor([idx_l[r] for r in rows], dtype=torch.long)
    sub_pool = case.ssm_pool.index_select(0, sl)
    gsel = torch.from_numpy(g_ref.astype(np.float32))[rows]
    bsel = torch.from_numpy(b_ref.astype(np.float32))[rows]
    o_ref, pool_ref, bad = oracle.decode(case.q[rows], case.k[rows], case.v[rows], gsel, bsel,
                                         sub_pool, np.arange(len(rows), dtype=np.int32),
                                         scale=case.scale, use_qk_l2norm=case.use_qk_l2norm)
    assert bad == 0
    P.assert_o_close(o_np[rows], o_ref)
    P.assert_state_close(pool.index_select(0, sl.to(dev)).cpu().numpy(), pool_ref, what="pool")


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_small(K, V, fused):
    case = W.decode_case("dec", 40 + K + V, 37, 50, 2, 4, K, V, pad_prob=0.2)
    _decode_check(case, fused)


def test_decode_config4_fused_gating():
    """256 requests against the [512, 32, 128, 128] pool: every valid request and
    every slot it touches against the oracle, untouched slots bit-exact."""
    _decode_check(W.config4(), fused=True)


def test_decode_maximum_request_count():
    """65535 requests (the largest count its grid takes; one more is refused on
    the host) against a pool of 70000 slots, about 10 % PAD: sampled requests
    against the oracle, PAD outputs zero, untouched slots bit-exact."""
    _decode_check(W.decode_case("dec_max_r", 61, 65535, 70000, 1, 1, 64, 64, pad_prob=0.1), fused=True, sample=200)


def test_decode_bad_slot_flagged_and_skipped():
    gdn = _gdn()
    case = W.decode_case("bad", 77, 4, 6, 2, 2, 64, 64, pad_prob=0.0)
    idx = torch.tensor([0, 6, -7, -1], dtype=torch.int32)
    pool = case.ssm_pool.cuda()
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_recurrent_decode(case.q.cuda(), case.k.cuda(), case.v.cuda(), pool, idx.cuda(),
                                 A_log=case.A_log.cuda(), a=case.a.cuda(), b=case.b.cuda(),
                                 dt_bias=case.dt_bias.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gdn.DEV_BAD_SLOT
    assert (o[1:].float() == 0).all()
    assert torch.equal(pool[1:], before[1:])
    assert not torch.equal(pool[0], before[0])


def test_gating_accuracy_sweep():
    """g and beta over a dense sweep of a + dt_bias in [-40, 40] (both softplus
    branches, the far tails where softplus(x) ~ e^x and ~ x) against fp64."""
    x = torch.linspace(-40.0, 40.0, 8 * 65536).to(torch.bfloat16).reshape(-1, 8)
    A_log = torch.log(torch.linspace(1.0, 16.0, 8))
    dt = torch.zeros(8)
    g, beta = _gdn().gdn_gating(A_log.cuda(), x.cuda(), x.cuda(), dt.cuda())
    torch.cuda.synchronize()
    g_ref, b_ref = oracle.gating(A_log, x, x, dt)
    np.testing.assert_allclose(g.cpu().numpy(), g_ref, rtol=P.GATE_RTOL, atol=P.GATE_ATOL)
    np.testing.assert_allclose(beta.cpu().numpy(), b_ref, rtol=P.GATE_RTOL, atol=P.GATE_ATOL)
