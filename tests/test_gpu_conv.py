"""GPU parity of the causal conv1d entry points against the fp64 oracle.

Outputs are bf16 rounded from fp32 accumulation, so the bound is one bf16
rounding of the exact value plus fp32 noise: |gpu - ref| <= 2^-8 |ref| + 1e-5.
The conv states are copies of bf16 inputs and must match bit for bit, as must
every slot a call is not supposed to touch.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_chunked_chunk_gb300 as gdn
from gated_deltanet_chunked_chunk_gb300 import workloads as W
from oracle import conv_oracle as CO

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RTOL, ATOL = 2.0 ** -8, 1e-5


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def close(gpu, ref):
    gpu = f64(gpu)
    err = np.abs(gpu - ref) - (RTOL * np.abs(ref) + ATOL)
    assert err.max() <= 0.0, f"max excess {err.max():.3e}"


def run_prefill(case, activation="silu", use_bias=True, use_init=True):
    d = lambda t: t.to(DEV).contiguous()
    states = d(case.conv_states)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_fwd(d(case.x), d(case.weight), d(case.bias) if use_bias else None, states,
                                    d(case.query_start_loc), d(case.cache_indices),
                                    d(case.has_initial_state) if use_init else None, activation=activation,
                                    dev_status=status)
    torch.cuda.synchronize()
    init = case.has_initial_state.numpy() if use_init else np.zeros(len(case.cache_indices), bool)
    ref_out, ref_states = CO.causal_conv1d_varlen(
        f64(case.x), f64(case.weight), f64(case.bias) if use_bias else None, f64(case.conv_states),
        case.query_start_loc.numpy(), case.cache_indices.numpy(), init, activation=activation)
    return out, states, status, ref_out, ref_states


@pytest.mark.parametrize("Wd,S", [(4, 3), (4, 6), (2, 1), (8, 7), (3, 8)])
def test_prefill_varlen_matches_oracle(Wd, S):
    # ragged lengths: empty, shorter than W - 1, crossing the 2048-token tile, PAD slot
    case = W.conv_prefill_case("t", 21 + Wd, 40, [5, 0, 70, 2, 2049, 1], W=Wd, S=S, pad_slot_every=4)
    out, states, status, ref_out, ref_states = run_prefill(case)
    close(out, ref_out)
    np.testing.assert_array_equal(f64(states), ref_states)
    assert int(status.item()) == 0


def test_prefill_without_activation_bias_or_initial_state():
    case = W.conv_prefill_case("t", 31, 33, [17, 300, 4])
    out, states, status, ref_out, ref_states = run_prefill(case, activation=None, use_bias=False, use_init=False)
    close(out, ref_out)
    np.testing.assert_array_equal(f64(states), ref_states)


def test_prefill_long_sampled_channels():
    # The benchmark's workload (8192 channels x 65536 tokens, one sequence
    # with an initial state); the oracle runs on 12 sampled channels (the conv
    # is per channel) over the whole sequence.
    case = W.conv_prefill_long()
    out, states, status, _, _ = run_prefill_full_only(case)
    chans = [0, 1, 2047, 2048, 4095, 4096, 5000, 6143, 6144, 7000, 8190, 8191]
    ref_out, ref_states = CO.causal_conv1d_varlen(
        f64(case.x[chans]), f64(case.weight[chans]), f64(case.bias[chans]), f64(case.conv_states[:, chans]),
        case.query_start_loc.numpy(), case.cache_indices.numpy(), case.has_initial_state.numpy())
    close(out[chans], ref_out)
    np.testing.assert_array_equal(f64(states[:, chans]), ref_states)
    assert int(status.item()) == 0


def run_prefill_full_only(case):
    d = lambda t: t.to(DEV).contiguous()
    states = d(case.conv_states)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_fwd(d(case.x), d(case.weight), d(case.bias), states, d(case.query_start_loc),
                                    d(case.cache_indices), d(case.has_initial_state), dev_status=status)
    torch.cuda.synchronize()
    return out, states, status, None, None


def test_prefill_bad_offsets_set_status():
    case = W.conv_prefill_case("t", 41, 16, [10, 10])
    d = lambda t: t.to(DEV).contiguous()
    bad = torch.tensor([0, 12, 15], dtype=torch.int32)   # last offset short of total = 20
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_fwd(d(case.x), d(case.weight), d(case.bias), d(case.conv_states), d(bad),
                                    d(case.cache_indices), d(case.has_initial_state), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gdn.DEV_BAD_CU_SEQLENS
    assert torch.all(out[:, 15:] == 0)


@pytest.mark.parametrize("R,P,dim,S", [(37, 50, 300, 3), (256, 512, 8192, 3), (5, 9, 64, 5)])
def test_decode_update_matches_oracle(R, P, dim, S):
    case = W.conv_decode_case("d", 51 + R, R, P, dim, S=S)
    d = lambda t: t.to(DEV).contiguous()
    states = d(case.conv_state)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_update(d(case.x), states, d(case.weight), d(case.bias), d(case.indices),
                                       dev_status=status)
    torch.cuda.synchronize()
    ref_out, ref_states = CO.causal_conv1d_update(f64(case.x), f64(case.conv_state), f64(case.weight),
                                                  f64(case.bias), case.indices.numpy())
    close(out, ref_out)
    np.testing.assert_array_equal(f64(states), ref_states)   # touched and untouched slots, bit for bit
    pad = (case.indices == -1).nonzero().flatten().tolist()
    if R >= 37:
        assert pad, "workload should contain PAD rows"
    assert torch.all(out[pad] == 0)
    assert int(status.item()) == 0


def test_decode_bad_slot_is_flagged_and_treated_as_pad():
    case = W.conv_decode_case("d", 61, 6, 8, 32)
    idx = torch.tensor([0, 8, -1, 3, -5, 7], dtype=torch.int32)
    d = lambda t: t.to(DEV).contiguous()
    states = d(case.conv_state)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_update(d(case.x), states, d(case.weight), d(case.bias), d(idx), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gdn.DEV_BAD_SLOT
    ref_idx = np.where((idx.numpy() < 0) | (idx.numpy() >= 8), -1, idx.numpy())
    ref_out, ref_states = CO.causal_conv1d_update(f64(case.x), f64(case.conv_state), f64(case.weight),
                                                  f64(case.bias), ref_idx)
    close(out, ref_out)
    np.testing.assert_array_equal(f64(states), ref_states)


def test_decode_pack_splits_into_recurrent_decode_layouts():
    H, HV, K, V = 2, 4, 64, 64
    dim = 2 * H * K + HV * V
    case = W.conv_decode_case("p", 71, 19, 24, dim)
    d = lambda t: t.to(DEV).contiguous()
    states = d(case.conv_state)
    q, k, v = gdn.gdn_conv_decode_pack(d(case.x), states, d(case.weight), d(case.bias), d(case.indices), H, HV, K, V)
    torch.cuda.synchronize()
    rq, rk, rv, rst = CO.conv_decode_pack(f64(case.x), f64(case.conv_state), f64(case.weight), f64(case.bias),
                                          case.indices.numpy(), H, HV, K, V)
    assert q.shape == (19, 1, H, K) and v.shape == (19, 1, HV, V)
    close(q, rq)
    close(k, rk)
    close(v, rv)
    np.testing.assert_array_equal(f64(states), rst)
    # the split buffers go straight into the recurrent decode
    pool = torch.zeros(24, HV, K, V, dtype=torch.float32, device=DEV)
    o = gdn.gdn_recurrent_decode(q, k, v, pool, d(case.indices), g=torch.zeros(19, HV, device=DEV),
                                 beta=torch.full((19, HV), 0.5, device=DEV))
    torch.cuda.synchronize()
    assert o.shape == (19, 1, HV, V) and torch.isfinite(o.float()).all()


def test_prefill_then_decode_continue_the_same_stream():
    # prefill T tokens, then decode token T+1 from the updated slot == prefill of T+1 tokens
    dim, T = 48, 37
    case = W.conv_prefill_case("c", 81, dim, [T + 1], P=2, init_every=1)
    d = lambda t: t.to(DEV).contiguous()
    st_a = d(case.conv_states)
    out_a = gdn.gdn_causal_conv1d_fwd(d(case.x[:, :T]), d(case.weight), d(case.bias), st_a,
                                      d(torch.tensor([0, T], dtype=torch.int32)), d(case.cache_indices),
                                      d(case.has_initial_state))
    dec = gdn.gdn_causal_conv1d_update(d(case.x[:, T:].t()), st_a, d(case.weight), d(case.bias),
                                       d(case.cache_indices))
    st_b = d(case.conv_states)
    out_b = gdn.gdn_causal_conv1d_fwd(d(case.x), d(case.weight), d(case.bias), st_b, d(case.query_start_loc),
                                      d(case.cache_indices), d(case.has_initial_state))
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b[:, :T])
    assert torch.equal(dec[0], out_b[:, T])
    assert torch.equal(st_a, st_b)


# ------------------------------------------------------------ MTP decode conv

def _spec_inputs(seed, N, m, P, dim, Wd, S, short=True, pad=True):
    gen = torch.Generator().manual_seed(seed)
    lens = [m + 1 if not (short and n % 3 == 2) else max(1, m - 1) for n in range(N)]
    qsl = torch.tensor(W.cu_from_lengths(lens), dtype=torch.int32)
    Tt = int(qsl[-1])
    x = torch.randn(Tt, dim, generator=gen).to(torch.bfloat16)
    weight = (torch.rand(dim, Wd, generator=gen) - 0.5).to(torch.bfloat16)
    bias = (torch.randn(dim, generator=gen) * 0.1).to(torch.bfloat16)
    states = torch.randn(P, dim, S, generator=gen).to(torch.bfloat16)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    if pad:
        idx[1] = -1
    acc = torch.randint(1, m + 2, (N,), generator=gen, dtype=torch.int32)
    return x, weight, bias, states, idx, acc, qsl


@pytest.mark.parametrize("N,m,P,dim,Wd,S", [(12, 3, 20, 200, 4, 6), (7, 1, 9, 64, 4, 8), (256, 3, 512, 1024, 4, 6)])
def test_spec_decode_update_matches_oracle(N, m, P, dim, Wd, S):
    x, w, b, st, idx, acc, qsl = _spec_inputs(70 + N, N, m, P, dim, Wd, S)
    states = st.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_update_spec(x.to(DEV), states, w.to(DEV), b.to(DEV), idx.to(DEV), acc.to(DEV),
                                            qsl.to(DEV), m, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_out, ref_states = CO.causal_conv1d_update_spec(f64(x), f64(st), f64(w), f64(b), idx.numpy(), acc.numpy(),
                                                       qsl.numpy(), m)
    close(out, ref_out)
    np.testing.assert_array_equal(f64(states), ref_states)   # every slot, bit for bit
    assert torch.all(out[int(qsl[1]):int(qsl[2])] == 0)       # the PAD request


def test_spec_decode_two_steps_carry_the_accepted_stream():
    """Two MTP steps in a row on the device against two oracle steps (the second
    step's accepted counts locate the history inside the first step's state)."""
    N, m, P, dim, Wd, S = 16, 3, 24, 256, 4, 6
    x1, w, b, st, idx, acc1, qsl = _spec_inputs(81, N, m, P, dim, Wd, S, short=False, pad=False)
    x2 = torch.randn(tuple(x1.shape), generator=torch.Generator().manual_seed(82)).to(torch.bfloat16)
    acc2 = torch.randint(1, m + 2, (N,), generator=torch.Generator().manual_seed(83), dtype=torch.int32)
    states = st.to(DEV)
    o1 = gdn.gdn_causal_conv1d_update_spec(x1.to(DEV), states, w.to(DEV), b.to(DEV), idx.to(DEV), acc1.to(DEV),
                                           qsl.to(DEV), m)
    o2 = gdn.gdn_causal_conv1d_update_spec(x2.to(DEV), states, w.to(DEV), b.to(DEV), idx.to(DEV), acc2.to(DEV),
                                           qsl.to(DEV), m)
    torch.cuda.synchronize()
    r1, rs = CO.causal_conv1d_update_spec(f64(x1), f64(st), f64(w), f64(b), idx.numpy(), acc1.numpy(), qsl.numpy(), m)
    r2, rs = CO.causal_conv1d_update_spec(f64(x2), rs, f64(w), f64(b), idx.numpy(), acc2.numpy(), qsl.numpy(), m)
    close(o1, r1)
    close(o2, r2)
    np.testing.assert_array_equal(f64(states), rs)


def test_spec_decode_bad_counts_flagged():
    x, w, b, st, idx, acc, qsl = _spec_inputs(91, 5, 2, 8, 32, 4, 5, short=False, pad=False)
    acc[3] = 0                                             # outside [1, m + 1]: treated as PAD
    bad_q = qsl.clone()
    states = st.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gdn.gdn_causal_conv1d_update_spec(x.to(DEV), states, w.to(DEV), b.to(DEV), idx.to(DEV), acc.to(DEV),
                                            bad_q.to(DEV), 2, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gdn.DEV_BAD_SLOT
    assert torch.all(out[int(qsl[3]):int(qsl[4])] == 0)
    assert torch.equal(states[int(idx[3])].cpu(), st[int(idx[3])])
