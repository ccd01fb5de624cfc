"""chunk_gated_delta_rule (torch.autograd over gdn_chunk_fwd / gdn_chunk_bwd):
the gradients autograd returns are the ones gdn_chunk_bwd computes for the
same upstream gradients, bit for bit (every sum in the backward has a fixed
order), and they match the fp64 autograd oracle."""
import numpy as np
import pytest
import torch

from gated_deltanet_chunked_chunk_gb300 import workloads as W
from oracle import bwd_oracle as BO
import parity_util as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_chunked_chunk_gb300 import build
    build.build()


@pytest.mark.parametrize("with_state", [True, False])
def test_autograd_matches_gdn_chunk_bwd(with_state):
    import gated_deltanet_chunked_chunk_gb300 as gdn
    case = W.prefill_case("autograd", 61, 1, 150, 2, 4, 64, 128, init="all" if with_state else "none")
    g, beta = P.oracle_gates(case)
    leaves = [t.to(DEV).contiguous() for t in (case.q, case.k, case.v, g, beta)]
    h0 = case.initial_state.to(DEV).contiguous() if with_state else None
    if h0 is not None:
        leaves.append(h0)
    for t in leaves:
        t.requires_grad_(True)
    q, k, v, gg, bb = leaves[:5]
    o, ht = gdn.chunk_gated_delta_rule(q, k, v, gg, bb, initial_state=h0, output_final_state=True)
    gen = torch.Generator().manual_seed(62)
    do = torch.randn(o.shape, generator=gen).to(torch.bfloat16).to(DEV)
    dht = torch.randn(ht.shape, generator=gen).to(DEV)
    grads = torch.autograd.grad([o, ht], leaves, [do, dht])
    direct = gdn.gdn_chunk_bwd(q.detach(), k.detach(), v.detach(), gg.detach(), bb.detach(), do,
                               initial_state=None if h0 is None else h0.detach(), dht=dht)
    for x, y, leaf in zip(grads, direct, leaves):
        assert x.dtype == leaf.dtype and x.shape == leaf.shape
        assert torch.equal(x, y.to(leaf.dtype))
    ref = BO.backward(case.q.float().numpy(), case.k.float().numpy(), case.v.float().numpy(), g.numpy(),
                      beta.numpy(), do.float().cpu().numpy(),
                      initial_state=None if h0 is None else case.initial_state.numpy(),
                      dht=dht.cpu().numpy())
    for name, x, r in zip(("dg", "dbeta"), direct[3:5], ref[3:5]):
        assert P.rel_l2(x.cpu().numpy().astype(np.float64), r) <= 5e-3, name


def test_autograd_without_final_state():
    import gated_deltanet_chunked_chunk_gb300 as gdn
    case = W.prefill_case("autograd_nofinal", 63, 1, 70, 1, 1, 64, 64)
    g, beta = P.oracle_gates(case)
    q = case.q.to(DEV).requires_grad_(True)
    o, ht = gdn.chunk_gated_delta_rule(q, case.k.to(DEV), case.v.to(DEV), g.to(DEV), beta.to(DEV),
                                       output_final_state=False)
    assert ht is None
    (dq,) = torch.autograd.grad(o.float().sum(), [q])
    assert dq.shape == q.shape and torch.isfinite(dq.float()).all()
