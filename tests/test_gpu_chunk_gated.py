"""GPU parity of gdn_chunk_fwd_gated (gating fused into the prefill) against
the fp64 oracle, through the C ABI.

The oracle side computes the gates in fp64 from the same raw inputs
(A_log, a, b, dt_bias) and runs the per-token recurrence; the GPU side gets
only the raw inputs.  Outputs must meet the prefill tolerances, the gates the
gating tolerance and equal gdn_gating's bit for bit (the same expressions),
and -- given those gates -- the plain prefill entry point must reproduce the
fused one bit for bit (both run the same two kernels on the same values)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_chunk_gb300 import workloads as W
import parity_util as P

pytestmark = pytest.mark.gpu
DEV = "cuda"
GATE_RTOL, GATE_ATOL = 1e-5, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_chunked_chunk_gb300 import build
    build.build()


def _run(case):
    import gated_deltanet_chunked_chunk_gb300 as gdn
    d = P.to_dev
    shp = (case.B, case.T, case.HV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, ht, g, beta = gdn.gdn_chunk_fwd_gated(
        d(case.q), d(case.k), d(case.v), d(case.A_log), d(case.a.reshape(shp)), d(case.b.reshape(shp)),
        d(case.dt_bias), scale=case.scale, initial_state=d(case.initial_state),
        output_final_state=case.output_final_state, cu_seqlens=d(case.cu_seqlens),
        use_qk_l2norm=case.use_qk_l2norm, return_gates=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, ht, g, beta


def _check(case):
    o, ht, g, beta = _run(case)
    g_ref, b_ref = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    shp = (case.B, case.T, case.HV)
    rows = slice(None)
    if case.cu_seqlens is not None:
        rows = slice(0, int(case.cu_seqlens[-1]))
    np.testing.assert_allclose(g.cpu().numpy()[:, rows], g_ref.reshape(shp)[:, rows], rtol=GATE_RTOL,
                               atol=GATE_ATOL)
    np.testing.assert_allclose(beta.cpu().numpy()[:, rows], b_ref.reshape(shp)[:, rows], rtol=GATE_RTOL,
                               atol=GATE_ATOL)
    # Parity against the oracle fed its own fp64 gates (rounded to fp32).
    g64, b64 = P.oracle_gates(case)
    o_ref, ht_ref = P.run_chunk_oracle(case, g64, b64)
    P.assert_o_close(o.float().cpu().numpy(), o_ref)
    if case.output_final_state:
        P.assert_state_close(ht.cpu().numpy(), ht_ref)
    # gdn_gating computes the same gates bit for bit ...
    import gated_deltanet_chunked_chunk_gb300 as gdn
    g2, b2 = gdn.gdn_gating(P.to_dev(case.A_log), P.to_dev(case.a), P.to_dev(case.b), P.to_dev(case.dt_bias))
    assert torch.equal(g[:, rows].reshape(-1, case.HV), g2.reshape(shp)[:, rows].reshape(-1, case.HV))
    assert torch.equal(beta[:, rows].reshape(-1, case.HV), b2.reshape(shp)[:, rows].reshape(-1, case.HV))
    # ... and the unfused entry point on those gates gives bit-identical results.
    o2, ht2 = P.run_chunk_gpu(case, g.cpu(), beta.cpu())
    assert np.array_equal(o.float().cpu().numpy(), o2)
    if ht is not None:
        assert np.array_equal(ht.cpu().numpy(), ht2)


def test_gated_config0_tiny():
    _check(W.config0())


def test_gated_ragged_gva_with_state():
    _check(W.prefill_case("gated_ragged", 51, 2, 200, 2, 4, 128, 128, init="all"))


def test_gated_long_single_sequence_two_ranges():
    # 71 chunks of one dense sequence: the two-range path, each range's prep
    # computing the gates of its own chunks.
    _check(W.prefill_case("gated_long", 54, 1, 64 * 70 + 20, 2, 4, 128, 128, init="all"))


def test_gated_varlen_with_empty_sequence():
    lengths = [70, 0, 5, 129]
    _check(W.prefill_case("gated_var", 52, 1, sum(lengths), 2, 4, 64, 128, init="even",
                          cu_seqlens=W.cu_from_lengths(lengths)))


def test_gated_without_gate_copies():
    import gated_deltanet_chunked_chunk_gb300 as gdn
    case = W.prefill_case("gated_nocopy", 53, 1, 96, 2, 2, 64, 64)
    d = P.to_dev
    shp = (case.B, case.T, case.HV)
    o, ht = gdn.gdn_chunk_fwd_gated(d(case.q), d(case.k), d(case.v), d(case.A_log), d(case.a.reshape(shp)),
                                    d(case.b.reshape(shp)), d(case.dt_bias))
    o_full, ht_full, _, _ = _run(case)
    assert torch.equal(o, o_full) and torch.equal(ht, ht_full)
