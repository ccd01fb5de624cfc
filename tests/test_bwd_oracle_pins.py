"""Pins for the backward oracle (CPU only): its gradients must match central
finite differences of an independent forward, the C per-token oracle
(``oracle.recurrent``), on tiny inputs.  A sign error, a missing GVA sum or a
dropped normalisation term in the backward each fail these."""
import numpy as np
import pytest

import oracle
from oracle import bwd_oracle as BO

RNG = np.random.default_rng


def _loss(q, k, v, g, beta, do, h0, dht, cu, l2, scale):
    o, ht = oracle.recurrent(q, k, v, g, beta, scale=scale, initial_state=h0, cu_seqlens=cu,
                             use_qk_l2norm=l2)
    val = float((o * do).sum())
    if dht is not None:
        val += float((ht * dht).sum())
    return val


def _fd_check(case, l2, cu=None, eps=1e-6, tol=2e-7):
    q, k, v, g, beta, do, h0, dht, scale = case
    dq, dk, dv, dg, db, dh0 = BO.backward(q, k, v, g, beta, do, scale=scale, initial_state=h0, cu_seqlens=cu,
                                          dht=dht, use_qk_l2norm=l2)
    named = [("q", q, dq), ("k", k, dk), ("v", v, dv), ("g", g, dg), ("beta", beta, db)]
    if h0 is not None:
        named.append(("h0", h0, dh0))
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    for name, x, grad in named:
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = x[i]
            x[i] = old + eps
            lp = _loss(args["q"], args["k"], args["v"], args["g"], args["beta"], do, args["h0"], dht, cu, l2, scale)
            x[i] = old - eps
            lm = _loss(args["q"], args["k"], args["v"], args["g"], args["beta"], do, args["h0"], dht, cu, l2, scale)
            x[i] = old
            num[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=0, atol=tol * max(1.0, np.abs(num).max()), err_msg=name)


def _case(seed, B=1, T=5, H=1, HV=2, K=3, V=2, N=None, init=True, final=True):
    r = RNG(seed)
    N = B if N is None else N
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, HV, V))
    g = -r.uniform(0.05, 1.0, (B, T, HV))
    beta = r.uniform(0.1, 0.9, (B, T, HV))
    do = r.standard_normal((B, T, HV, V))
    h0 = r.standard_normal((N, HV, K, V)) * 0.5 if init else None
    dht = r.standard_normal((N, HV, K, V)) if final else None
    return [q, k, v, g, beta, do, h0, dht, 0.7]


@pytest.mark.parametrize("l2", [True, False])
def test_backward_matches_finite_differences(l2):
    _fd_check(_case(0), l2)


def test_backward_gva_and_no_state_inputs():
    # G = 3 value heads per key head: dq, dk must sum over the group.
    _fd_check(_case(1, H=1, HV=3, T=4, init=False, final=False), True)


def test_backward_varlen():
    # Two packed sequences: gradients must not flow across the boundary.
    c = _case(2, B=1, T=6, N=2)
    _fd_check(c, True, cu=[0, 2, 6])


def test_backward_of_a_linear_output_is_the_transpose():
    # With beta = 0 and g = 0 the state never changes: o_t = scale S0^T q_t, so
    # dh0 = scale * sum_t q_t do_t^T and dv = 0 (a closed form, no autograd logic
    # involved in the reference).
    q, k, v, g, beta, do, h0, _, scale = _case(3, T=4, HV=1)
    g[:] = 0.0
    beta[:] = 0.0
    dq, dk, dv, dg, db, dh0 = BO.backward(q, k, v, g, beta, do, scale=scale, initial_state=h0, use_qk_l2norm=False)
    ref = scale * np.einsum("tk,tv->kv", q[0, :, 0], do[0, :, 0])
    np.testing.assert_allclose(dh0[0, 0], ref, rtol=0, atol=1e-13)
    assert np.all(dv == 0.0)
    np.testing.assert_allclose(dq[0, :, 0], scale * np.einsum("kv,tv->tk", h0[0, 0], do[0, :, 0]), atol=1e-13)
