"""Pins for the multi-token (MTP) decode and the bf16-pool decode of the
oracle (CPU only).  The MTP bookkeeping (which slot a request starts from,
which slot each token's state goes to) is pinned against the sequence form of
the recurrence, ``oracle.recurrent``, which the other pins tie to the
definition; the bf16 storage rounding against numpy's own float32 rounding and
hand-picked ties."""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng


def _mtp_case(seed, N=3, ld=4, H=1, HV=2, K=6, V=5, P=14):
    r = RNG(seed)
    lens = [ld, ld - 1, ld]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Tt = int(cu[-1])
    q = r.standard_normal((Tt, H, K))
    k = r.standard_normal((Tt, H, K))
    v = r.standard_normal((Tt, HV, V))
    g = -r.uniform(0.05, 1.0, (Tt, HV))
    beta = r.uniform(0.0, 1.0, (Tt, HV))
    pool = r.standard_normal((P, HV, K, V)) * 0.3
    slots = np.arange(N * ld, dtype=np.int32).reshape(N, ld)    # request n owns slots n*ld .. n*ld+ld-1
    acc = np.array([1, 3, ld], dtype=np.int32)
    return q, k, v, g, beta, pool, cu, slots, acc


def test_mtp_equals_recurrence_from_the_accepted_slot():
    # o of every token and every stored intermediate state must equal the
    # sequence recurrence started from pool[slot[n][acc[n]-1]] over the
    # request's first i+1 tokens.  Catches an off-by-one in num_accepted,
    # storing the state before instead of after a token, or a wrong column.
    q, k, v, g, beta, pool, cu, slots, acc = _mtp_case(0)
    o, new, bad = oracle.decode_mtp(q, k, v, g, beta, pool, cu, slots, slots, acc)
    assert bad == 0
    for n in range(3):
        t0, t1 = cu[n], cu[n + 1]
        s0 = pool[slots[n, acc[n] - 1]]
        for i in range(t1 - t0):
            oi, hi = oracle.recurrent(q[None, t0:t0 + i + 1], k[None, t0:t0 + i + 1], v[None, t0:t0 + i + 1],
                                      g[None, t0:t0 + i + 1], beta[None, t0:t0 + i + 1],
                                      initial_state=s0[None])
            np.testing.assert_allclose(o[t0 + i], oi[0, -1], rtol=0, atol=1e-12)
            np.testing.assert_allclose(new[slots[n, i]], hi[0], rtol=0, atol=1e-12)
    # slots past a short request's tokens keep their old contents
    np.testing.assert_array_equal(new[slots[1, 3]], pool[slots[1, 3]])
    np.testing.assert_array_equal(new[12:], pool[12:])


def test_mtp_with_one_token_equals_single_token_decode():
    r = RNG(1)
    R, H, HV, K, V, P = 5, 2, 4, 8, 4, 9
    q, k = r.standard_normal((R, H, K)), r.standard_normal((R, H, K))
    v = r.standard_normal((R, HV, V))
    g, beta = -r.uniform(0.05, 1, (R, HV)), r.uniform(0, 1, (R, HV))
    pool = r.standard_normal((P, HV, K, V))
    idx = np.array([3, -1, 0, 8, 5], dtype=np.int32)
    o1, p1, b1 = oracle.decode(q, k, v, g, beta, pool, idx)
    o2, p2, b2 = oracle.decode_mtp(q, k, v, g, beta, pool, np.arange(R + 1), idx[:, None], idx[:, None])
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(p1, p2)
    assert b1 == b2 == 0


def test_mtp_pad_request_and_bad_counts():
    q, k, v, g, beta, pool, cu, slots, acc = _mtp_case(2)
    rd = slots.copy()
    rd[1, :] = -1                                  # request 1 is PAD
    o, new, bad = oracle.decode_mtp(q, k, v, g, beta, pool, cu, rd, slots, acc)
    assert bad == 0
    assert np.all(o[cu[1]:cu[2]] == 0.0)
    np.testing.assert_array_equal(new[slots[1]], pool[slots[1]])
    _, _, bad = oracle.decode_mtp(q, k, v, g, beta, pool, cu, slots, slots, np.array([0, 1, 1], np.int32))
    assert bad == 1                                # num_accepted 0 is outside [1, ld]


def test_round_bf16_matches_float32_path_and_ties():
    # On values that are exact in fp32, rounding to bf16 must agree with the
    # classic fp32 bit trick (add 0x7fff + lsb, truncate); ties go to even.
    r = RNG(3)
    x = r.standard_normal(20000).astype(np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    trick = (((bits + 0x7FFF + lsb) >> 16) << 16).astype(np.uint32).view(np.float32)
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), trick.astype(np.float64))
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even mantissa -> 1;
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even -> 1 + 2^-6
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8)) == -1.0


def test_bf16_pool_decode_rounds_only_the_touched_states():
    r = RNG(4)
    R, H, HV, K, V, P = 4, 1, 2, 8, 8, 6
    q, k = r.standard_normal((R, H, K)), r.standard_normal((R, H, K))
    v = r.standard_normal((R, HV, V))
    g, beta = -r.uniform(0.05, 1, (R, HV)), r.uniform(0, 1, (R, HV))
    pool = oracle.round_bf16(r.standard_normal((P, HV, K, V)))
    idx = np.array([4, -1, 1, 2], dtype=np.int32)
    o, new, _ = oracle.decode_bf16_pool(q, k, v, g, beta, pool, idx)
    o32, new32, _ = oracle.decode(q, k, v, g, beta, pool, idx)
    np.testing.assert_array_equal(o, o32)                      # output from the unrounded new state
    for s in (4, 1, 2):
        np.testing.assert_array_equal(new[s], oracle.round_bf16(new32[s]))
        assert np.any(new[s] != new32[s])
    for s in (0, 3, 5):
        np.testing.assert_array_equal(new[s], pool[s])
