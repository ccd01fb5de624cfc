"""Pins for the fp64 oracle (CPU only).

The pages print no worked numbers for the kernel, so the oracle is pinned to
things other than itself: hand-worked fixtures (tests/golden/), closed forms,
invariants of the recurrence, brute-force restatements in a different
factorisation, and the chunked algorithm's exact equivalence with the
recurrence.  Each test names the mistake it is there to catch.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng


def _rand_case(seed, T=23, H=1, HV=1, K=8, V=6, B=1, decay=(0.05, 1.0)):
    r = RNG(seed)
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K))
    v = r.standard_normal((B, T, HV, V))
    g = -r.uniform(*decay, (B, T, HV))
    beta = r.uniform(0.0, 1.0, (B, T, HV))
    return q, k, v, g, beta


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- golden ----

def test_golden_k1_hand_worked():
    """Scalar case worked by hand: catches a wrong sign in the delta term or the
    decay applied after instead of before the read."""
    rows = _read_rows("recurrence_k1_worked.txt")
    S0 = float(rows[0][1])
    data = np.array([[float(x) for x in r] for r in rows[1:-1]])
    final = float(rows[-1][1])
    T = len(data)
    a, beta, k, q, v, o_exp = data.T
    o, ht = oracle.recurrent(q.reshape(1, T, 1, 1), k.reshape(1, T, 1, 1), v.reshape(1, T, 1, 1),
                             np.log(a).reshape(1, T, 1), beta.reshape(1, T, 1), scale=1.0,
                             initial_state=np.array([[[[S0]]]]), use_qk_l2norm=False)
    np.testing.assert_allclose(o.reshape(-1), o_exp, rtol=0, atol=1e-15)
    assert abs(ht.item() - final) < 1e-15


def test_golden_k2_hand_worked():
    """2x2 case worked by hand: catches a transposed state (S vs S^T) and a
    transposed outer product (k delta^T vs delta k^T)."""
    rows = _read_rows("recurrence_k2_worked.txt")
    S0 = np.array([float(x) for x in rows[0][1:]]).reshape(1, 1, 2, 2)
    data = np.array([[float(x) for x in r] for r in rows[1:-1]])
    final = np.array([float(x) for x in rows[-1][1:]]).reshape(2, 2)
    T = len(data)
    a, beta = data[:, 0], data[:, 1]
    k, q, v, o_exp = data[:, 2:4], data[:, 4:6], data[:, 6:8], data[:, 8:10]
    o, ht = oracle.recurrent(q.reshape(1, T, 1, 2), k.reshape(1, T, 1, 2), v.reshape(1, T, 1, 2),
                             np.log(a).reshape(1, T, 1), beta.reshape(1, T, 1), scale=1.0,
                             initial_state=S0, use_qk_l2norm=False)
    np.testing.assert_allclose(o.reshape(T, 2), o_exp, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht[0, 0], final, rtol=0, atol=1e-14)


def test_golden_gating_closed_forms():
    """softplus(0) = ln 2, the x > 20 branch, sigmoid(+-ln 3): catches a missing
    exp on A_log, a missing dt_bias, or sigmoid(-b)."""
    rows = np.array([[float(x) for x in r] for r in _read_rows("gating_closed_forms.txt")])
    for A_log, a, dt, b, g_exp, beta_exp in rows:
        g, beta = oracle.gating(np.array([A_log]), np.array([[a]]), np.array([[b]]), np.array([dt]))
        assert abs(g.item() - g_exp) <= 1e-14 * max(1.0, abs(g_exp))
        assert abs(beta.item() - beta_exp) <= 1e-15


# ---------------------------------------------------------------- gating ----

def test_gating_matches_python_math_and_bounds():
    r = RNG(1)
    HV, Tt = 5, 40
    A_log = np.log(r.uniform(1, 16, HV))
    dt = np.log(np.expm1(r.uniform(1e-3, 0.1, HV)))
    a = r.standard_normal((Tt, HV)) * 8
    b = r.standard_normal((Tt, HV)) * 8
    g, beta = oracle.gating(A_log, a, b, dt)
    g2, beta2 = oracle.gating_scalar(A_log, a, b, dt)
    np.testing.assert_allclose(g, g2, rtol=1e-15, atol=0)
    np.testing.assert_allclose(beta, beta2, rtol=1e-15, atol=0)
    assert (g <= 0).all() and (beta > 0).all() and (beta < 1).all()
    # softplus(dt_bias) returns the drawn U(1e-3, 0.1) value by construction
    u = r.uniform(1e-3, 0.1, HV)
    g0, _ = oracle.gating(np.zeros(HV), np.zeros((1, HV)), np.zeros((1, HV)), np.log(np.expm1(u)))
    np.testing.assert_allclose(-g0[0], u, rtol=1e-13)


# ------------------------------------------------------ brute-force forms ----

@pytest.mark.parametrize("l2", [True, False])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_recurrence_vs_transition_product_and_attention_form(seed, l2):
    """Three formulations -- the C loop, the transition-matrix product and the
    one-chunk attention form with a dense LU -- must agree to rounding."""
    T, K, V = 16, 5, 4
    q, k, v, g, beta = _rand_case(seed, T=T, K=K, V=V)
    S0 = RNG(seed + 50).standard_normal((1, 1, K, V))
    sc = 0.37
    o, ht = oracle.recurrent(q, k, v, g, beta, scale=sc, initial_state=S0, use_qk_l2norm=l2)
    o2, S2 = oracle.transition_product(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0],
                                       beta[0, :, 0], S0[0, 0], sc, use_qk_l2norm=l2)
    o3, S3 = oracle.attention_form(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0],
                                   beta[0, :, 0], S0[0, 0], sc, use_qk_l2norm=l2)
    np.testing.assert_allclose(o[0, :, 0], o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], S2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[0, :, 0], o3, rtol=0, atol=1e-11)
    np.testing.assert_allclose(ht[0, 0], S3, rtol=0, atol=1e-11)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunked_wy_equals_recurrence(C):
    """The chunked WY derivation (cumsum, KK^T, solve, w/u, state walk, output)
    reaches the per-token result; C = 1 degenerates to the recurrence."""
    T, K, V = 150, 16, 12
    q, k, v, g, beta = _rand_case(7, T=T, K=K, V=V)
    S0 = RNG(8).standard_normal((1, 1, K, V)) * 0.1
    o, ht = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    o2, h2 = oracle.chunked_wy(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                               S0[0, 0], 1 / math.sqrt(K), C=C)
    np.testing.assert_allclose(o[0, :, 0], o2, rtol=0, atol=1e-10)
    np.testing.assert_allclose(ht[0, 0], h2, rtol=0, atol=1e-10)


# ------------------------------------------------------------- invariants ---

def test_beta0_g0_leaves_state_and_reads_it():
    T, K, V = 12, 6, 5
    q, k, v, _, _ = _rand_case(3, T=T, K=K, V=V)
    S0 = RNG(4).standard_normal((1, 1, K, V))
    o, ht = oracle.recurrent(q, k, v, np.zeros((1, T, 1)), np.zeros((1, T, 1)), scale=0.5,
                             initial_state=S0)
    np.testing.assert_array_equal(ht, S0)
    qn = q[0, :, 0] / np.sqrt((q[0, :, 0] ** 2).sum(-1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(o[0, :, 0], 0.5 * qn @ S0[0, 0], rtol=0, atol=1e-14)


def test_beta0_is_pure_decay():
    """beta = 0: S_t = exp(gamma_t) S0 (catches a decay applied to the update only)."""
    T, K, V = 9, 4, 3
    q, k, v, g, _ = _rand_case(5, T=T, K=K, V=V)
    S0 = RNG(6).standard_normal((1, 1, K, V))
    _, ht = oracle.recurrent(q, k, v, g, np.zeros((1, T, 1)), initial_state=S0)
    np.testing.assert_allclose(ht[0, 0], math.exp(g.sum()) * S0[0, 0], rtol=1e-13, atol=0)


def test_large_negative_gate_forgets_state():
    """g = -1e3 at token t: exp underflows to 0, so the result equals a fresh
    start at t with a zero state."""
    T, K, V, t0 = 20, 6, 5, 8
    q, k, v, g, beta = _rand_case(9, T=T, K=K, V=V)
    g[0, t0, 0] = -1e3
    S0 = RNG(10).standard_normal((1, 1, K, V))
    o, ht = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    sl = slice(t0, T)
    o2, h2 = oracle.recurrent(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], initial_state=None)
    np.testing.assert_allclose(o[:, sl], o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht, h2, rtol=0, atol=1e-14)


def test_beta1_unit_key_recalls_value_for_any_gate():
    """beta = 1 with a unit key: S_t^T k_t = v_t exactly, whatever g is."""
    T, K, V = 15, 8, 6
    q, k, v, g, _ = _rand_case(11, T=T, K=K, V=V, decay=(0.0, 3.0))
    S0 = RNG(12).standard_normal((1, 1, K, V))
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    for t in range(1, T + 1):
        _, ht = oracle.recurrent(q[:, :t], kn[:, :t], v[:, :t], g[:, :t], np.ones((1, t, 1)),
                                 initial_state=S0, use_qk_l2norm=False)
        np.testing.assert_allclose(ht[0, 0].T @ kn[0, t - 1, 0], v[0, t - 1, 0], rtol=0, atol=1e-13)


def test_orthonormal_keys_recall_every_pair():
    """Orthonormal keys (T <= K), g = 0, beta = 1: every stored pair is recalled."""
    K, V = 8, 5
    T = K
    r = RNG(13)
    Qm, _ = np.linalg.qr(r.standard_normal((K, K)))
    k = Qm.T.reshape(1, T, 1, K)
    v = r.standard_normal((1, T, 1, V))
    q = r.standard_normal((1, T, 1, K))
    _, ht = oracle.recurrent(q, k, v, np.zeros((1, T, 1)), np.ones((1, T, 1)),
                             initial_state=r.standard_normal((1, 1, K, V)), use_qk_l2norm=False)
    np.testing.assert_allclose(k[0, :, 0] @ ht[0, 0], v[0, :, 0], rtol=0, atol=1e-13)


def test_linearity_in_values_and_state():
    """(V, S0) -> (o, S_T) is linear for fixed q, k, g, beta."""
    T, K, V = 17, 6, 4
    q, k, v1, g, beta = _rand_case(14, T=T, K=K, V=V)
    r = RNG(15)
    v2 = r.standard_normal(v1.shape)
    s1, s2 = r.standard_normal((1, 1, K, V)), r.standard_normal((1, 1, K, V))
    o1, h1 = oracle.recurrent(q, k, v1, g, beta, initial_state=s1)
    o2, h2 = oracle.recurrent(q, k, v2, g, beta, initial_state=s2)
    o3, h3 = oracle.recurrent(q, k, 2.0 * v1 - 3.0 * v2, g, beta, initial_state=2.0 * s1 - 3.0 * s2)
    np.testing.assert_allclose(o3, 2 * o1 - 3 * o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h3, 2 * h1 - 3 * h2, rtol=0, atol=1e-12)


def test_varlen_equals_separate_calls_and_gva_mapping():
    """Packed varlen = one call per sequence; value head hv reads key head hv // G."""
    lens = [5, 1, 0, 13, 7]
    cu = np.cumsum([0] + lens)
    Tt, H, HV, K, V = cu[-1], 2, 6, 5, 3
    r = RNG(16)
    q = r.standard_normal((1, Tt, H, K))
    k = r.standard_normal((1, Tt, H, K))
    v = r.standard_normal((1, Tt, HV, V))
    g = -r.uniform(0.05, 1, (1, Tt, HV))
    beta = r.uniform(0, 1, (1, Tt, HV))
    S0 = r.standard_normal((len(lens), HV, K, V))
    o, ht = oracle.recurrent(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        for hv in range(HV):
            h = hv // (HV // H)
            # one-head dense call with the key head expanded explicitly
            o1, h1 = oracle.recurrent(q[:, sl, h:h + 1], k[:, sl, h:h + 1], v[:, sl, hv:hv + 1],
                                      g[:, sl, hv:hv + 1], beta[:, sl, hv:hv + 1],
                                      initial_state=S0[n:n + 1, hv:hv + 1], scale=1 / math.sqrt(K))
            np.testing.assert_array_equal(o[:, sl, hv], o1[:, :, 0])
            np.testing.assert_array_equal(ht[n, hv], h1[0, 0])
    # empty sequence: final state equals the initial state
    np.testing.assert_array_equal(ht[2], S0[2])


def test_split_with_state_carry_equals_one_shot():
    T, K, V = 40, 6, 5
    q, k, v, g, beta = _rand_case(17, T=T, K=K, V=V)
    S0 = RNG(18).standard_normal((1, 1, K, V))
    o, ht = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    for cut in (1, 13, 32):
        oa, ha = oracle.recurrent(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut], beta[:, :cut],
                                  initial_state=S0)
        ob, hb = oracle.recurrent(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], beta[:, cut:],
                                  initial_state=ha)
        np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(hb, ht, rtol=0, atol=1e-13)


def test_l2norm_zero_vector_gives_zero_not_nan():
    T, K, V = 3, 4, 2
    q = np.zeros((1, T, 1, K))
    k = np.zeros((1, T, 1, K))
    v = np.ones((1, T, 1, V))
    o, ht = oracle.recurrent(q, k, v, -np.ones((1, T, 1)) * 0.1, np.ones((1, T, 1)) * 0.5)
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    np.testing.assert_array_equal(o, 0.0)


def test_scale_default_is_inverse_sqrt_k():
    q, k, v, g, beta = _rand_case(19, T=6, K=9, V=3)
    o1, _ = oracle.recurrent(q, k, v, g, beta, scale=None)
    o2, _ = oracle.recurrent(q, k, v, g, beta, scale=1 / 3)
    np.testing.assert_array_equal(o1, o2)


def test_items_subset_matches_full():
    q, k, v, g, beta = _rand_case(20, T=11, H=2, HV=4, K=5, V=3, B=3)
    S0 = RNG(21).standard_normal((3, 4, 5, 3))
    o, ht = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    o2, h2 = oracle.recurrent(q, k, v, g, beta, initial_state=S0, items=[(2, 1), (0, 3)])
    np.testing.assert_array_equal(o2[2, :, 1], o[2, :, 1])
    np.testing.assert_array_equal(h2[0, 3], ht[0, 3])
    assert np.isnan(o2[1]).all()


def test_thread_count_does_not_change_result():
    q, k, v, g, beta = _rand_case(22, T=30, H=2, HV=4, K=6, V=4, B=2)
    a = oracle.recurrent(q, k, v, g, beta, nthreads=1)
    b = oracle.recurrent(q, k, v, g, beta, nthreads=5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ----------------------------------------------------------------- decode ---

def test_decode_equals_one_token_prefill_and_skips_pad():
    r = RNG(23)
    R, P, H, HV, K, V = 6, 9, 2, 4, 5, 3
    q = r.standard_normal((R, H, K))
    k = r.standard_normal((R, H, K))
    v = r.standard_normal((R, HV, V))
    g = -r.uniform(0.05, 1, (R, HV))
    beta = r.uniform(0, 1, (R, HV))
    pool = r.standard_normal((P, HV, K, V))
    idx = np.array([3, -1, 0, 8, -1, 5], dtype=np.int32)
    o, newpool, bad = oracle.decode(q, k, v, g, beta, pool, idx)
    assert bad == 0
    touched = set(int(i) for i in idx if i >= 0)
    for s in range(P):
        if s not in touched:
            np.testing.assert_array_equal(newpool[s], pool[s])
    for rq in range(R):
        if idx[rq] < 0:
            np.testing.assert_array_equal(o[rq], 0.0)
            continue
        o1, h1 = oracle.recurrent(q[rq][None, None], k[rq][None, None], v[rq][None, None],
                                  g[rq][None, None], beta[rq][None, None],
                                  initial_state=pool[idx[rq]][None])
        np.testing.assert_array_equal(o[rq], o1[0, 0])
        np.testing.assert_array_equal(newpool[idx[rq]], h1[0])
    # an out-of-range slot is flagged and handled like PAD
    o2, p2, bad2 = oracle.decode(q[:1], k[:1], v[:1], g[:1], beta[:1], pool, np.array([P], np.int32))
    assert bad2 == 1 and (o2 == 0).all()
    np.testing.assert_array_equal(p2, pool)
