"""gdn_chunk_fwd_noalloc: the chunked prefill for callers that cannot allocate
device memory at call time (their device memory is reserved up front by their
own pool, or their hot loop must stay off the allocation path).  Its workspace
is a fixed buffer inside the library; this test checks, through the C ABI, that
two calls in a row give bit for bit what gdn_chunk_fwd gives with a caller
workspace (the same kernels on the same inputs), and
that inputs too large for the fixed buffer are refused before any launch.

Kept in a file that pytest collects last, so a run that stops at the first
failure has run every other test before this one."""
import ctypes

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


def _inputs(case):
    g, beta = P.oracle_gates(case)
    d = lambda t: None if t is None else t.cuda().contiguous()
    return (d(case.q), d(case.k), d(case.v), d(g), d(beta), d(case.initial_state), d(case.cu_seqlens))


@pytest.mark.parametrize("varlen", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(varlen):
    gdn = _gdn()
    if varlen:
        cu = W.cu_from_lengths([70, 1, 0, 130, 64])
        case = W.prefill_case("noalloc_varlen", 31, 1, cu[-1], 2, 4, 128, 128, cu_seqlens=cu, init="even")
    else:
        case = W.prefill_case("noalloc_dense", 30, 2, 300, 2, 4, 128, 128, init="all")
    q, k, v, g, beta, h0, cu_t = _inputs(case)
    need = gdn.chunk_fwd_workspace_size(case.B, case.T, case.H, case.HV, case.K, case.V, case.N, varlen)
    assert 0 < need <= gdn.NOALLOC_SCRATCH_BYTES
    o_ref, h_ref = gdn.gdn_chunk_fwd(q, k, v, g, beta, initial_state=h0, cu_seqlens=cu_t)
    torch.cuda.synchronize()
    for _ in range(2):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        o, h = gdn.gdn_chunk_fwd_noalloc(q, k, v, g, beta, initial_state=h0, cu_seqlens=cu_t, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # the same kernels on the same inputs: identical bits, only the
        # workspace's address differs
        assert torch.equal(o, o_ref), "o (noalloc vs workspace) differs"
        assert torch.equal(h, h_ref), "final_state (noalloc vs workspace) differs"
        # and both within the parity tolerances of the oracle's result
        P.assert_o_close(o.float().cpu().numpy(), o_ref.float().cpu().numpy(), what="o (noalloc vs workspace)")


def test_noalloc_refuses_inputs_beyond_its_scratch():
    gdn = _gdn()
    lib = gdn.load_library()
    B, T, H, HV, K, V = 1, 65536, 16, 32, 128, 128
    assert gdn.chunk_fwd_workspace_size(B, T, H, HV, K, V, 1, False) > gdn.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    rc = lib.gdn_chunk_fwd_noalloc(fake, fake, fake, fake, fake, -1.0, None, None, 1, B, T, H, HV, K, V, 1,
                                   fake, None, None, None)
    assert rc == gdn.GDN_ESCRATCH_LIMIT
    assert "no-allocation" in gdn.status_string(rc)
