"""Pins for the conv1d oracle (CPU only).

The pages print no worked values for the causal conv either, so the oracle
(``oracle/conv_oracle.py``) is pinned to closed forms, a library routine
(``numpy.convolve``) on the special case of one stream, and invariants of the
stream definition.  Each test names the mistake it is there to catch.
"""
import math

import numpy as np
import pytest

from oracle import conv_oracle as CO

RNG = np.random.default_rng


def _rand(seed, dim=5, total=17, W=4, S=3, P=4):
    r = RNG(seed)
    x = r.standard_normal((dim, total))
    w = r.uniform(-0.5, 0.5, (dim, W))
    b = r.standard_normal(dim) * 0.1
    st = r.standard_normal((P, dim, S))
    return x, w, b, st


def test_silu_closed_forms():
    # silu(0) = 0; silu(ln 3) = ln 3 * 3/4; silu(-ln 3) = -ln 3 / 4 (a sign error fails)
    assert CO.silu(0.0) == 0.0
    assert abs(CO.silu(math.log(3.0)) - math.log(3.0) * 0.75) < 1e-15
    assert abs(CO.silu(-math.log(3.0)) + math.log(3.0) * 0.25) < 1e-15


def test_single_stream_equals_numpy_convolve():
    # One sequence, no history, no activation: out[d] is the 'valid' convolution
    # of the zero-padded row with the reversed taps (numpy.convolve flips its
    # second argument, so reversed taps give the correlation the conv computes).
    # Catches reversed taps or an off-by-one in the window.
    x, w, b, st = _rand(0, dim=3, total=20, W=4, S=3)
    out, _ = CO.causal_conv1d_varlen(x, w, None, st, [0, 20], [0], [False], activation=None)
    for d in range(3):
        padded = np.concatenate([np.zeros(3), x[d]])
        ref = np.convolve(padded, w[d][::-1], mode="valid")
        np.testing.assert_allclose(out[d], ref, rtol=0, atol=1e-13)


def test_identity_tap_and_shift_taps():
    # weight = e_{W-1}: out = act(x + b); weight = e_{W-1-s}: out[t] = x[t - s]
    # (zeros before the sequence start without history).  Catches a tap-order
    # mix-up and the activation being applied before the bias.
    x, _, b, st = _rand(1, dim=2, total=9, W=4, S=3)
    for s in range(4):
        w = np.zeros((2, 4))
        w[:, 3 - s] = 1.0
        out, _ = CO.causal_conv1d_varlen(x, w, None, st, [0, 9], [0], [False], activation=None)
        ref = np.concatenate([np.zeros((2, s)), x[:, :9 - s]], axis=1)
        np.testing.assert_array_equal(out, ref)
    w = np.zeros((2, 4))
    w[:, 3] = 1.0
    out, _ = CO.causal_conv1d_varlen(x, w, b, st, [0, 9], [0], [False], activation="silu")
    np.testing.assert_allclose(out, CO.silu(x + b[:, None]), rtol=0, atol=1e-15)


def test_history_enters_the_first_taps():
    # With has_initial_state the first W-1 outputs see the last W-1 state
    # entries: a shift by s at position p < s reads state[:, S - s + p].
    x, _, _, st = _rand(2, dim=2, total=6, W=4, S=5)
    for s in range(1, 4):
        w = np.zeros((2, 4))
        w[:, 3 - s] = 1.0
        out, _ = CO.causal_conv1d_varlen(x, w, None, st, [0, 6], [2], [True], activation=None)
        for p in range(6):
            ref = st[2][:, 5 - s + p] if p < s else x[:, p - s]
            np.testing.assert_array_equal(out[:, p], ref)


def test_state_is_the_last_S_inputs():
    # New state = last S entries of history ++ x, also for sequences shorter
    # than S (part old state, part input); without initial state the history
    # is zeros.  Catches keeping W-1 instead of S entries or dropping history.
    x, w, b, st = _rand(3, dim=3, total=10, W=4, S=5, P=3)
    qsl = [0, 2, 2, 10]
    _, new = CO.causal_conv1d_varlen(x, w, b, st, qsl, [0, 1, 2], [True, True, False], activation="silu")
    np.testing.assert_array_equal(new[0], np.concatenate([st[0][:, 2:], x[:, 0:2]], axis=1))
    np.testing.assert_array_equal(new[1], st[1])              # empty sequence keeps its state
    np.testing.assert_array_equal(new[2], x[:, 10 - 5:10])    # 8 tokens >= S
    _, new2 = CO.causal_conv1d_varlen(x[:, :2], w, b, st, [0, 2], [0], [False], activation=None)
    np.testing.assert_array_equal(new2[0], np.concatenate([np.zeros((3, 3)), x[:, :2]], axis=1))


def test_varlen_equals_separate_calls_and_pad_slot():
    # Packing sequences must not leak tokens across a boundary; a PAD slot
    # (-1) reads zeros and leaves the pool alone.
    x, w, b, st = _rand(4, dim=4, total=15, W=4, S=3, P=4)
    qsl = [0, 5, 6, 15]
    slots = [3, -1, 1]
    init = [True, True, False]
    out, new = CO.causal_conv1d_varlen(x, w, b, st, qsl, slots, init)
    for n in range(3):
        s0, s1 = qsl[n], qsl[n + 1]
        o1, n1 = CO.causal_conv1d_varlen(x[:, s0:s1], w, b, st, [0, s1 - s0], [slots[n]], [init[n]])
        np.testing.assert_array_equal(out[:, s0:s1], o1)
        if slots[n] >= 0:
            np.testing.assert_array_equal(new[slots[n]], n1[slots[n]])
    np.testing.assert_array_equal(new[0], st[0])
    np.testing.assert_array_equal(new[2], st[2])


def test_split_with_state_carry_equals_one_shot():
    # conv(x[:a]) then conv(x[a:]) from the updated state == conv(x): the state
    # is exactly what the stream needs to continue.
    x, w, b, st = _rand(5, dim=3, total=13, W=4, S=3, P=1)
    full, fstate = CO.causal_conv1d_varlen(x, w, b, st, [0, 13], [0], [True])
    for a in (1, 2, 3, 7):
        o1, s1 = CO.causal_conv1d_varlen(x[:, :a], w, b, st, [0, a], [0], [True])
        o2, s2 = CO.causal_conv1d_varlen(x[:, a:], w, b, s1, [0, 13 - a], [0], [True])
        np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), full, rtol=0, atol=1e-14)
        np.testing.assert_array_equal(s2, fstate)


def test_decode_step_equals_length_one_prefill():
    # The decode update is the prefill of a one-token sequence with history;
    # PAD rows give zeros and leave the pool untouched.
    r = RNG(6)
    R, dim, W, S, P = 5, 6, 4, 4, 7
    x = r.standard_normal((R, dim))
    w = r.uniform(-0.5, 0.5, (dim, W))
    b = r.standard_normal(dim)
    st = r.standard_normal((P, dim, S))
    idx = [4, -1, 0, 6, 2]
    out, new = CO.causal_conv1d_update(x, st, w, b, idx)
    for i, s in enumerate(idx):
        if s < 0:
            np.testing.assert_array_equal(out[i], 0.0)
            continue
        o1, n1 = CO.causal_conv1d_varlen(x[i][:, None], w, b, st, [0, 1], [s], [True])
        np.testing.assert_allclose(out[i], o1[:, 0], rtol=0, atol=1e-15)
        np.testing.assert_array_equal(new[s], n1[s])
    for s in (1, 3, 5):
        np.testing.assert_array_equal(new[s], st[s])


def test_linearity_without_activation():
    # Without bias and activation the conv is linear in (x, history).
    x, w, _, st = _rand(7, dim=3, total=11, W=3, S=2, P=1)
    y = RNG(8).standard_normal(x.shape)
    st2 = RNG(9).standard_normal(st.shape)
    a, c = 0.7, -1.3
    o1, _ = CO.causal_conv1d_varlen(x, w, None, st, [0, 11], [0], [True], activation=None)
    o2, _ = CO.causal_conv1d_varlen(y, w, None, st2, [0, 11], [0], [True], activation=None)
    o3, _ = CO.causal_conv1d_varlen(a * x + c * y, w, None, a * st + c * st2, [0, 11], [0], [True],
                                    activation=None)
    np.testing.assert_allclose(o3, a * o1 + c * o2, rtol=0, atol=1e-13)


def test_decode_pack_splits_q_k_v_in_channel_order():
    # The packed channels are q (H*K), then k (H*K), then v (HV*V), each in
    # row-major head order.  Catches a swapped q/k block or a head-major error.
    H, HV, K, V, R = 2, 4, 3, 2, 3
    dim = 2 * H * K + HV * V
    r = RNG(10)
    x = r.standard_normal((R, dim))
    w = r.uniform(-0.5, 0.5, (dim, 4))
    st = r.standard_normal((2, dim, 3))
    idx = [1, -1, 0]
    q, k, v, new = CO.conv_decode_pack(x, st, w, None, idx, H, HV, K, V)
    out, new2 = CO.causal_conv1d_update(x, st, w, None, idx)
    np.testing.assert_array_equal(q[:, 0].reshape(R, -1), out[:, :H * K])
    np.testing.assert_array_equal(k[:, 0].reshape(R, -1), out[:, H * K:2 * H * K])
    np.testing.assert_array_equal(v[:, 0].reshape(R, -1), out[:, 2 * H * K:])
    np.testing.assert_array_equal(new, new2)
    assert q[0, 0, 1, 2] == out[0, 1 * K + 2]


# ------------------------------------------------------------ MTP decode conv

def _spec_case(seed, N, m, dim, W, S, A=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(((m + 1) * N, dim))
    weight = rng.uniform(-0.5, 0.5, (dim, W))
    bias = rng.normal(0, 0.1, dim)
    states = rng.standard_normal((N + 2, dim, S))
    qsl = np.arange(0, (m + 1) * N + 1, m + 1)
    acc = np.asarray(A if A is not None else rng.integers(1, m + 2, N))
    return x, weight, bias, states, qsl, acc


def test_spec_with_no_draft_is_the_single_token_update():
    """mtp_step = 0, one token, one accepted: exactly causal_conv1d_update."""
    x, w, b, st, qsl, _ = _spec_case(1, 5, 0, 6, 4, 3)
    idx = np.array([3, 0, -1, 4, 1])
    o1, s1 = CO.causal_conv1d_update_spec(x, st, w, b, idx, np.ones(5, int), qsl, 0)
    o2, s2 = CO.causal_conv1d_update(x, st, w, b, idx)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


def test_spec_all_accepted_continues_the_plain_stream():
    """Two MTP steps with every token accepted give the plain stream's outputs
    and leave the plain stream's last S inputs in the slot."""
    m, W, dim = 3, 4, 5
    S = W - 1 + m
    rng = np.random.default_rng(2)
    hist = rng.standard_normal((dim, S))
    x1, x2 = rng.standard_normal((m + 1, dim)), rng.standard_normal((m + 1, dim))
    w, b = rng.uniform(-0.5, 0.5, (dim, W)), rng.normal(0, 0.1, dim)
    st = hist[None].copy()
    qsl = np.array([0, m + 1])
    o1, st = CO.causal_conv1d_update_spec(x1, st, w, b, [0], [m + 1], qsl, m)
    o2, st = CO.causal_conv1d_update_spec(x2, st, w, b, [0], [m + 1], qsl, m)
    # the first step starts from a slot whose last m + 1 entries were all accepted
    stream = np.concatenate([hist[:, S - (W - 1):], x1.T, x2.T], axis=1)
    ref = CO.conv_stream(stream, w, b, "silu")
    np.testing.assert_allclose(np.concatenate([o1, o2]).T, ref, rtol=1e-13, atol=1e-13)
    whole = np.concatenate([hist, x1.T, x2.T], axis=1)
    np.testing.assert_array_equal(st[0], whole[:, -S:])


def test_spec_rejected_drafts_never_reach_later_outputs():
    """Speculative decoding's defining property: after a step of m + 1 tokens of
    which A were accepted, the next step's outputs equal those of a plain stream
    that only ever saw the A accepted tokens."""
    m, W, dim = 3, 4, 6
    S = W - 1 + m
    rng = np.random.default_rng(3)
    w, b = rng.uniform(-0.5, 0.5, (dim, W)), rng.normal(0, 0.1, dim)
    hist = rng.standard_normal((dim, W - 1))
    for A in range(1, m + 2):
        x1, x2 = rng.standard_normal((m + 1, dim)), rng.standard_normal((m + 1, dim))
        # a slot as prefill leaves it: the first W - 1 entries, then m unused ones
        st = np.concatenate([hist, rng.standard_normal((dim, m)) * 1e6], axis=1)[None]
        qsl = np.array([0, m + 1])
        _, st = CO.causal_conv1d_update_spec(x1, st, w, b, [0], [1], qsl, m)
        o2, _ = CO.causal_conv1d_update_spec(x2, st, w, b, [0], [A], qsl, m)
        stream = np.concatenate([hist, x1[:A].T, x2.T], axis=1)
        ref = CO.conv_stream(stream, w, b, "silu")[:, A:]
        np.testing.assert_allclose(o2.T, ref, rtol=1e-12, atol=1e-12)


def test_spec_after_prefill_reads_only_the_prefill_state():
    """num_accepted = 1 on a freshly prefilled slot (prefill writes slot[:W - 1]
    through the sliced view) ignores the mtp_step unused entries."""
    m, W, dim = 2, 4, 3
    rng = np.random.default_rng(4)
    w, b = rng.uniform(-0.5, 0.5, (dim, W)), None
    prefill_state = rng.standard_normal((dim, W - 1))
    junk = rng.standard_normal((dim, m)) * 1e9
    st = np.concatenate([prefill_state, junk], axis=1)[None]
    x = rng.standard_normal((m + 1, dim))
    o, _ = CO.causal_conv1d_update_spec(x, st, w, b, [0], [1], [0, m + 1], m, activation=None)
    ref = CO.conv_stream(np.concatenate([prefill_state, x.T], axis=1), w, b, None)
    np.testing.assert_allclose(o.T, ref, rtol=1e-13, atol=1e-13)


def test_spec_pad_request_and_linearity():
    x, w, b, st, qsl, acc = _spec_case(5, 4, 2, 5, 3, 5)
    idx = np.array([1, -1, 0, 3])
    o, s = CO.causal_conv1d_update_spec(x, st, w, None, idx, acc, qsl, 2, activation=None)
    assert (o[qsl[1]:qsl[2]] == 0).all()
    np.testing.assert_array_equal(s[[2, 4, 5]], st[[2, 4, 5]])      # untouched slots
    o2, s2 = CO.causal_conv1d_update_spec(2 * x, 2 * st, w, None, idx, acc, qsl, 2, activation=None)
    np.testing.assert_allclose(o2, 2 * o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s2[[0, 1, 3]], 2 * s[[0, 1, 3]], rtol=1e-13, atol=1e-13)
