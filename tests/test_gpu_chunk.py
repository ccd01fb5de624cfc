"""GPU parity of gdn_chunk_fwd against the fp64 oracle (through the C ABI)."""
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


def _check_case(case, items=None):
    g, beta = P.oracle_gates(case)
    o_gpu, ht_gpu = P.run_chunk_gpu(case, g, beta)
    o_ref, ht_ref = P.run_chunk_oracle(case, g, beta, items=items)
    if items is None:
        P.assert_o_close(o_gpu, o_ref)
        if case.output_final_state:
            P.assert_state_close(ht_gpu, ht_ref)
        else:
            assert ht_gpu is None
    return o_gpu, ht_gpu, o_ref, ht_ref


GRID = []
for i, (K, V) in enumerate([(64, 64), (128, 128), (64, 128), (128, 64)]):
    for j, T in enumerate([1, 63, 64, 65, 200]):
        G = (1, 2, 4)[(i + j) % 3]
        GRID.append((K, V, T, G, (i + j) % 2 == 0, (i * 5 + j) % 3 != 1))


@pytest.mark.parametrize("K,V,T,G,init,final", GRID)
def test_shape_grid(K, V, T, G, init, final):
    case = W.prefill_case(f"grid", 100 + K + V + T + G, 2, T, 2, 2 * G, K, V,
                          init="all" if init else "none", output_final_state=final)
    _check_case(case)


def test_config0_tiny():
    _check_case(W.config0())


def test_config1_dense_gva_with_state():
    _check_case(W.config1())


def test_config2_varlen_packed():
    _check_case(W.config2())


def test_no_l2norm_and_explicit_scale():
    case = W.prefill_case("nol2", 7, 1, 130, 2, 4, 64, 64, init="all", scale=0.05,
                          use_qk_l2norm=False)
    case.q = (case.q.float() / 8).to(torch.bfloat16)
    case.k = (case.k.float() / 8).to(torch.bfloat16)
    _check_case(case)


def test_varlen_with_empty_and_short_sequences():
    lens = [0, 1, 64, 0, 65, 130, 7]
    cu = W.cu_from_lengths(lens)
    case = W.prefill_case("varlen_edge", 8, 1, cu[-1], 2, 4, 128, 128, cu_seqlens=cu, init="all")
    o_gpu, ht_gpu, o_ref, ht_ref = _check_case(case)
    h0 = case.initial_state.numpy()
    for n, L in enumerate(lens):
        if L == 0:
            np.testing.assert_array_equal(ht_gpu[n], h0[n])


def test_varlen_many_sequences():
    # 1500 sequences of 0..150 tokens (every kind of ragged tail, a fifth of them
    # empty): exercises the chunk-start table that maps chunk slots to sequences.
    rng = np.random.default_rng(21)
    lens = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(1, 151, 1500)]
    cu = W.cu_from_lengths(lens)
    case = W.prefill_case("varlen_many", 21, 1, cu[-1], 1, 2, 64, 64, cu_seqlens=cu, init="all")
    o_gpu, ht_gpu, o_ref, ht_ref = _check_case(case)
    h0 = case.initial_state.numpy()
    for n, L in enumerate(lens):
        if L == 0:
            np.testing.assert_array_equal(ht_gpu[n], h0[n])


def test_varlen_equals_separate_dense_calls_bitwise():
    lens = [70, 1, 129, 64]
    cu = W.cu_from_lengths(lens)
    case = W.prefill_case("packed", 9, 1, cu[-1], 2, 4, 128, 128, cu_seqlens=cu, init="all")
    g, beta = P.oracle_gates(case)
    o_p, ht_p = P.run_chunk_gpu(case, g, beta)
    import gated_deltanet_chunked_chunk_gb300 as gdn
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        o1, h1 = gdn.gdn_chunk_fwd(case.q[:, sl].cuda(), case.k[:, sl].cuda(), case.v[:, sl].cuda(),
                                   g[:, sl].contiguous().cuda(), beta[:, sl].contiguous().cuda(),
                                   initial_state=case.initial_state[n:n + 1].cuda())
        np.testing.assert_array_equal(o1.float().cpu().numpy()[0], o_p[0, sl])
        np.testing.assert_array_equal(h1.cpu().numpy()[0], ht_p[n])


def test_split_at_chunk_boundary_with_state_carry_is_bitwise():
    case = W.prefill_case("split", 10, 1, 320, 2, 4, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    import gated_deltanet_chunked_chunk_gb300 as gdn
    d = lambda t: t.cuda().contiguous()
    o_full, h_full = gdn.gdn_chunk_fwd(d(case.q), d(case.k), d(case.v), d(g), d(beta),
                                       initial_state=d(case.initial_state))
    cut = 192
    oa, ha = gdn.gdn_chunk_fwd(d(case.q[:, :cut]), d(case.k[:, :cut]), d(case.v[:, :cut]),
                               d(g[:, :cut]), d(beta[:, :cut]), initial_state=d(case.initial_state))
    ob, hb = gdn.gdn_chunk_fwd(d(case.q[:, cut:]), d(case.k[:, cut:]), d(case.v[:, cut:]),
                               d(g[:, cut:]), d(beta[:, cut:]), initial_state=ha)
    assert torch.equal(torch.cat([oa, ob], 1), o_full)
    assert torch.equal(hb, h_full)


@pytest.mark.parametrize("K", [128, 64])
def test_long_single_sequence_two_ranges_match_batched_call_bitwise(K):
    # One dense sequence of 71 chunks (a ragged last one) is walked in two
    # chunk ranges (16 walk CTAs leave most SMs free, so the ranges are about
    # even), the walk of the first overlapping the prep of the second, with
    # the fp32 state handed over in the workspace.  The same sequence as
    # one of a batch of two takes the single-range path: the same bits, and
    # parity with the oracle.  The workspace starts as NaN bytes, so a second
    # range that read the handed-over state before the first range wrote it
    # would show.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    T = 64 * 70 + 20
    case = W.prefill_case("two_ranges", 11, 1, T, 2, 4, K, 128, init="all")
    _check_case(case)
    g, beta = P.oracle_gates(case)
    d = lambda t: t.cuda().contiguous()
    two = lambda t: torch.cat([t, t.flip(1)], 0)
    ws = torch.full((gdn.chunk_fwd_workspace_size(1, T, 2, 4, K, 128, 1, False),), 255, dtype=torch.uint8,
                    device="cuda")
    o1, h1 = gdn.gdn_chunk_fwd(d(case.q), d(case.k), d(case.v), d(g), d(beta),
                               initial_state=d(case.initial_state), workspace=ws)
    o2, h2 = gdn.gdn_chunk_fwd(d(two(case.q)), d(two(case.k)), d(two(case.v)), d(two(g)), d(two(beta)),
                               initial_state=d(torch.cat([case.initial_state, case.initial_state], 0)))
    assert torch.equal(o2[:1], o1)
    assert torch.equal(h2[:1], h1)
    # The same sequence given with cu_seqlens = [0, T] (one varlen sequence)
    # takes the same ranges after the chunk-start table.
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    ws3 = torch.full((gdn.chunk_fwd_workspace_size(1, T, 2, 4, K, 128, 1, True),), 255, dtype=torch.uint8,
                     device="cuda")
    o3, h3 = gdn.gdn_chunk_fwd(d(case.q), d(case.k), d(case.v), d(g), d(beta), initial_state=d(case.initial_state),
                               cu_seqlens=cu, workspace=ws3)
    assert torch.equal(o3, o1)
    assert torch.equal(h3, h1)
    # Two ranges: four launches (five with the chunk-start table); the batch
    # of two (and a 63-chunk sequence) takes two.
    assert gdn.chunk_fwd_kernel_launches(1, T, 2, 4, K, 128, 1, False) == 4
    assert gdn.chunk_fwd_kernel_launches(1, T, 2, 4, K, 128, 1, True) == 5
    assert gdn.chunk_fwd_kernel_launches(2, T, 2, 4, K, 128, 2, False) == 2
    assert gdn.chunk_fwd_kernel_launches(1, 63 * 64, 2, 4, K, 128, 1, False) == 2


def test_three_ranges_reuse_the_hand_over_buffer_bitwise():
    # 300 chunks at HV = 32 (128 walk CTAs, 24 SMs free): three chunk ranges,
    # the hand-over state rewritten in place twice.  NaN-filled workspace; the
    # same sequence in a batch of two (one range) gives the same bits.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    T = 64 * 300
    case = W.prefill_case("three_ranges", 12, 1, T, 16, 32, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    d = lambda t: t.cuda().contiguous()
    two = lambda t: torch.cat([t, t.flip(1)], 0)
    assert gdn.chunk_fwd_kernel_launches(1, T, 16, 32, 128, 128, 1, False) == 6
    ws = torch.full((gdn.chunk_fwd_workspace_size(1, T, 16, 32, 128, 128, 1, False),), 255, dtype=torch.uint8,
                    device="cuda")
    o1, h1 = gdn.gdn_chunk_fwd(d(case.q), d(case.k), d(case.v), d(g), d(beta),
                               initial_state=d(case.initial_state), workspace=ws)
    o2, h2 = gdn.gdn_chunk_fwd(d(two(case.q)), d(two(case.k)), d(two(case.v)), d(two(g)), d(two(beta)),
                               initial_state=d(torch.cat([case.initial_state, case.initial_state], 0)))
    assert torch.equal(o2[:1], o1)
    assert torch.equal(h2[:1], h1)


def test_multi_range_call_captured_in_a_cuda_graph_matches_eager():
    # A serving loop captures the prefill into a CUDA graph.  Three chunk
    # ranges (six launches, the later preps programmatic dependents of the
    # walks before them) captured and replayed give the eager call's bits.
    import gated_deltanet_chunked_chunk_gb300 as gdn
    T = 64 * 300
    case = W.prefill_case("graph", 13, 1, T, 16, 32, 128, 128, init="all")
    g, beta = P.oracle_gates(case)
    d = lambda t: t.cuda().contiguous()
    q, k, v, gg, bb, h0 = d(case.q), d(case.k), d(case.v), d(g), d(beta), d(case.initial_state)
    ws = torch.empty(gdn.chunk_fwd_workspace_size(1, T, 16, 32, 128, 128, 1, False), dtype=torch.uint8,
                     device="cuda")
    o_e, h_e = gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, workspace=ws)
    o_g = torch.empty_like(o_e)
    h_g = torch.empty_like(h_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, workspace=ws, o=o_g, final_state=h_g)
    torch.cuda.current_stream().wait_stream(side)
    o_g.zero_()
    h_g.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, workspace=ws, o=o_g, final_state=h_g)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e)
    assert torch.equal(h_g, h_e)


def test_varlen_maximum_sequence_count():
    # 65535 packed sequences (the largest count the walk's grid takes; one
    # more is refused on the host) of 0 to 3 tokens each, every one with its
    # own initial state: sampled sequences against the oracle, and the empty
    # ones carry their initial state through unchanged.
    N = 65535
    rng = np.random.default_rng(60)
    lens = [int(x) for x in rng.integers(0, 4, N)]
    cu = W.cu_from_lengths(lens)
    case = W.prefill_case("max_n", 60, 1, cu[-1], 1, 1, 64, 64, cu_seqlens=cu, init="all")
    g, beta = P.oracle_gates(case)
    o_gpu, ht_gpu = P.run_chunk_gpu(case, g, beta)
    assert np.isfinite(o_gpu).all() and np.isfinite(ht_gpu).all()
    empty = [n for n in range(N) if lens[n] == 0]
    assert len(empty) > 1000
    np.testing.assert_array_equal(ht_gpu[empty[:2000]], case.initial_state[empty[:2000]].numpy())
    for n in [0, 1, 2, 3, 77, 4096, 32767, 40000, N - 2, N - 1] + [int(x) for x in rng.integers(0, N, 20)]:
        o_ref, h_ref, (b0, sl) = P.oracle_single_head(case, g, beta, n, 0)
        if lens[n]:
            P.assert_o_close(o_gpu[b0:b0 + 1, sl, 0:1], o_ref[None, :, None], f"o seq {n}")
        P.assert_state_close(ht_gpu[n:n + 1, 0:1], h_ref[None, None], f"state seq {n}")


def test_deterministic_and_guard_bands():
    case = W.config1()
    g, beta = P.oracle_gates(case)
    import gated_deltanet_chunked_chunk_gb300 as gdn
    d = lambda t: t.cuda().contiguous()
    q, k, v, gg, bb, h0 = map(d, (case.q, case.k, case.v, g, beta, case.initial_state))
    pad = 4096
    o_buf = torch.full((case.B * case.T * case.HV * case.V + 2 * pad,), 0x7FBF, dtype=torch.int16,
                       device="cuda").view(torch.bfloat16)
    s_buf = torch.full((h0.numel() + 2 * pad,), 12345.0, device="cuda")
    o = o_buf[pad:-pad].view(case.B, case.T, case.HV, case.V)
    ht = s_buf[pad:-pad].view_as(h0)
    gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0, o=o, final_state=ht)
    o2, h2 = gdn.gdn_chunk_fwd(q, k, v, gg, bb, initial_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(ht, h2)
    canary = o_buf.view(torch.int16)
    assert bool((canary[:pad] == 0x7FBF).all()) and bool((canary[-pad:] == 0x7FBF).all())
    assert bool((s_buf[:pad] == 12345.0).all()) and bool((s_buf[-pad:] == 12345.0).all())


def test_bad_cu_seqlens_sets_device_status():
    import gated_deltanet_chunked_chunk_gb300 as gdn
    T, H, HV, K = 100, 2, 2, 64
    x = torch.zeros(1, T, H, K, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(1, T, HV, K, dtype=torch.bfloat16, device="cuda")
    gz = torch.zeros(1, T, HV, device="cuda")
    cu = torch.tensor([0, 60, 40, 100], dtype=torch.int32, device="cuda")  # decreasing
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_fwd(x, x, v, gz, gz, cu_seqlens=cu, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gdn.DEV_BAD_CU_SEQLENS


def test_chunk_entry_points_from_a_fresh_thread():
    # The first CUDA work of a new host thread is the library call (outputs and
    # workspace allocated beforehand on the main thread): the entry points make
    # the device's context current before their tensor-map encode, and give the
    # same bits as on the main thread.
    import threading
    import gated_deltanet_chunked_chunk_gb300 as gdn
    case = W.prefill_case("thread", 71, 1, 150, 2, 4, 64, 128, init="all")
    g, beta = P.oracle_gates(case)
    d = lambda t: t.to("cuda").contiguous()
    args = (d(case.q), d(case.k), d(case.v), d(g), d(beta))
    h0 = d(case.initial_state)
    ws = torch.empty(gdn.chunk_fwd_workspace_size(1, 150, 2, 4, 64, 128, 1, False), dtype=torch.uint8,
                     device="cuda")
    o_main, ht_main = gdn.gdn_chunk_fwd(*args, initial_state=h0, workspace=ws)
    o = torch.empty_like(o_main)
    ht = torch.empty_like(ht_main)
    torch.cuda.synchronize()
    errors = []

    def work():
        try:
            gdn.gdn_chunk_fwd(*args, initial_state=h0, o=o, final_state=ht, workspace=ws)
        except Exception as ex:  # reported on the main thread below
            errors.append(ex)

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert torch.equal(o, o_main) and torch.equal(ht, ht_main)
