"""The method's own edge cases on the CUDA path (through the C ABI), each held
to the same bars as the oracle pins of test_oracle_pins.py.

"NPU Training Operators - GDN", section "Operator semantics": g is the
log-space forget gate (a very negative g wipes the state) and beta the strength
of the delta update (beta = 0 writes nothing, beta = 1 with a unit key stores
v exactly under that key).  The FastDeploy PR "support fla triton kernel for
qwen3.5", accuracy table, checks the chunked kernel against the recurrent one;
here both are checked against the fp64 per-token oracle.
"""
import numpy as np
import pytest
import torch

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


def _d(t):
    return None if t is None else t.cuda().contiguous()


def _run(case, g, beta):
    return P.run_chunk_gpu(case, g, beta)


def _oracle(case, g, beta):
    return P.run_chunk_oracle(case, g, beta)


def _case(seed, T, H, HV, K, V, init="all"):
    return W.prefill_case("edge", seed, 1, T, H, HV, K, V, init=init)


@pytest.mark.parametrize("t0", [100, 128])
def test_forget_gate_wipes_state(t0):
    """g = -1e3 at token t0 (mid-chunk: 100, chunk boundary: 128): e^g is 0 in
    fp32, so every later output equals that of a fresh start at t0 with a zero
    state; the chunk holding t0 takes the unfactored decay branch."""
    case = _case(31 + t0, 320, 2, 4, 128, 128)
    g, beta = P.oracle_gates(case)
    g[:, t0] = -1e3
    o_gpu, ht_gpu = _run(case, g, beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)
    # the same tokens from t0 on, started fresh (no initial state)
    fresh = W.PrefillCase("fresh", case.q[:, t0:].contiguous(), case.k[:, t0:].contiguous(),
                          case.v[:, t0:].contiguous(), case.A_log, case.a, case.b, case.dt_bias,
                          None, None, None)
    o_f, ht_f = _run(fresh, g[:, t0:].contiguous(), beta[:, t0:].contiguous())
    P.assert_o_close(o_gpu[:, t0:], o_f, what="o after the wipe vs fresh start")
    P.assert_state_close(ht_gpu, ht_f, what="final state vs fresh start")
    if t0 % 64 == 0:
        # same chunk alignment: the wiped state enters every product multiplied
        # by an exact zero, so the two runs agree bit for bit
        np.testing.assert_array_equal(o_gpu[:, t0:], o_f)
        np.testing.assert_array_equal(ht_gpu, ht_f)


def test_beta_zero_gate_zero_keeps_state():
    """beta = 0, g = 0: nothing is written and nothing decays, so the final state
    is the initial one bit for bit and o_t = scale S0^T q_hat_t."""
    case = _case(41, 200, 2, 4, 128, 128)
    g = torch.zeros(1, case.T, case.HV)
    beta = torch.zeros(1, case.T, case.HV)
    o_gpu, ht_gpu = _run(case, g, beta)
    np.testing.assert_array_equal(ht_gpu, case.initial_state.numpy())
    o_ref, ht_ref = _oracle(case, g, beta)
    np.testing.assert_array_equal(ht_ref, case.initial_state.numpy().astype(np.float64))
    P.assert_o_close(o_gpu, o_ref)


def test_beta_one_unit_key_recalls_last_value():
    """beta = 1 with unit keys (L2 norm on): after token t the state maps k_hat_t
    to v_t exactly, whatever g is: S_T^T k_hat_T = v_T."""
    case = _case(43, 193, 2, 4, 128, 128)
    g, _ = P.oracle_gates(case)
    beta = torch.ones(1, case.T, case.HV)
    o_gpu, ht_gpu = _run(case, g, beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)
    G = case.HV // case.H
    for hv in range(case.HV):
        k = case.k[0, -1, hv // G].double().numpy()
        kh = k / np.sqrt((k * k).sum() + 1e-6)
        recall = ht_gpu[0, hv].astype(np.float64).T @ kh
        np.testing.assert_allclose(recall, case.v[0, -1, hv].double().numpy(), atol=P.STATE_MAX_ABS)


def test_orthonormal_keys_recall_every_value():
    """Keys e_0, e_1, ... (exactly orthonormal in bf16) across two chunks, g = 0,
    beta = 1, zero initial state: every stored pair is recalled, S_T^T e_t = v_t,
    i.e. row t of the final state is v_t."""
    T, K, V = 128, 128, 64
    case = _case(47, T, 1, 2, K, V, init="none")
    eye = torch.zeros(1, T, 1, K)
    eye[0, torch.arange(T), 0, torch.arange(T)] = 1.0
    case.k = eye.to(torch.bfloat16)
    g = torch.zeros(1, T, case.HV)
    beta = torch.ones(1, T, case.HV)
    o_gpu, ht_gpu = _run(case, g, beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)
    for hv in range(case.HV):
        np.testing.assert_allclose(ht_gpu[0, hv], case.v[0, :, hv].float().numpy(), atol=P.STATE_MAX_ABS)


def test_zero_query_and_key_rows_stay_finite():
    """All-zero q and k rows with the L2 norm on: the normalised vectors are 0
    (not NaN); a zero query gives a zero output row, a zero key writes nothing."""
    case = _case(53, 150, 2, 4, 64, 64)
    case.q[0, 3::7] = 0
    case.k[0, 5::11] = 0
    case.q[0, 64:70] = 0
    case.k[0, 64:70] = 0
    g, beta = P.oracle_gates(case)
    o_gpu, ht_gpu = _run(case, g, beta)
    assert np.isfinite(o_gpu).all() and np.isfinite(ht_gpu).all()
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)
    G = case.HV // case.H
    for hv in range(case.HV):
        zero_q = (case.q[0, :, hv // G].float() == 0).all(-1).numpy()
        assert (o_gpu[0, zero_q, hv] == 0).all()


def test_large_and_moderate_chunk_decay():
    """One head whose per-chunk decay is e^-126 (too wide to factor into row and
    column terms in fp32: the element-by-element branch) next to one at e^-63
    (factored): both against the oracle."""
    case = _case(59, 256, 1, 2, 128, 128)
    g = torch.empty(1, case.T, case.HV)
    g[..., 0] = -2.0
    g[..., 1] = -1.0
    beta = torch.sigmoid(torch.randn(1, case.T, case.HV, generator=torch.Generator().manual_seed(5)))
    o_gpu, ht_gpu = _run(case, g, beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    for hv in range(2):
        P.assert_o_close(o_gpu[..., hv, :], o_ref[..., hv, :], what=f"o[hv={hv}]")
        P.assert_state_close(ht_gpu[:, hv], ht_ref[:, hv], what=f"final_state[hv={hv}]")


def test_gate_mix_per_chunk_branches():
    """Random per-chunk mixes: each 64-token chunk of each head draws its gate
    scale so that chunks land on both sides of the factoring limit, with an
    initial state, against the oracle."""
    case = _case(61, 64 * 12 + 17, 2, 4, 128, 128)
    gen = torch.Generator().manual_seed(61)
    nchunk = (case.T + 63) // 64
    scale = torch.exp(torch.empty(nchunk, case.HV).uniform_(np.log(0.05), np.log(3.0), generator=gen))
    g = -(torch.rand(1, case.T, case.HV, generator=gen) * 2.0) * scale.repeat_interleave(64, 0)[:case.T][None]
    beta = torch.rand(1, case.T, case.HV, generator=gen)
    o_gpu, ht_gpu = _run(case, g.contiguous(), beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)


def test_decode_edge_cases_match_oracle():
    """Decode with beta = 0 and g = 0 leaves the pool slot bit-unchanged, and
    g = -1e3 with beta = 1 and unit keys stores v under k exactly."""
    gdn = _gdn()
    import oracle
    case = W.decode_case("dec_edge", 71, 6, 8, 2, 4, 64, 64, pad_prob=0.0)
    pool = case.ssm_pool.cuda()
    before = pool.clone()
    idx = case.ssm_indices.cuda()
    g = torch.zeros(case.R, case.HV)
    b = torch.zeros(case.R, case.HV)
    o = gdn.gdn_recurrent_decode(_d(case.q), _d(case.k), _d(case.v), pool, idx, g=_d(g), beta=_d(b))
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    o_ref, _, _ = oracle.decode(case.q, case.k, case.v, g, b, case.ssm_pool, case.ssm_indices.numpy())
    P.assert_o_close(o.float().cpu().numpy()[:, 0], o_ref)
    g = torch.full((case.R, case.HV), -1e3)
    b = torch.ones(case.R, case.HV)
    gdn.gdn_recurrent_decode(_d(case.q), _d(case.k), _d(case.v), pool, idx, g=_d(g), beta=_d(b))
    torch.cuda.synchronize()
    G = case.HV // case.H
    for r, s in enumerate(case.ssm_indices.tolist()):
        for hv in range(case.HV):
            k = case.k[r, 0, hv // G].double().numpy()
            kh = k / np.sqrt((k * k).sum() + 1e-6)
            S = pool[s, hv].double().cpu().numpy()
            np.testing.assert_allclose(S, np.outer(kh, case.v[r, 0, hv].double().numpy()), atol=1e-5)


@pytest.mark.slow
def test_config3_long_context_all_heads():
    """T = 65536 (1024 serial chunks), every value head, against the whole
    oracle; the last 4096 tokens also on their own (errors must not grow along T)."""
    case = W.config3()
    g, beta = P.oracle_gates(case)
    o_gpu, ht_gpu = _run(case, g, beta)
    o_ref, ht_ref = _oracle(case, g, beta)
    P.assert_o_close(o_gpu, o_ref)
    P.assert_state_close(ht_gpu, ht_ref)
    P.assert_o_close(o_gpu[:, -4096:], o_ref[:, -4096:], what="o tail")
    for hv in range(case.HV):
        P.assert_o_close(o_gpu[..., hv, :], o_ref[..., hv, :], what=f"o[hv={hv}]")
