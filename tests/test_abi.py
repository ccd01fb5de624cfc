"""CPU-side checks of the C ABI: the library builds/loads, exports every symbol
include/gdn.h declares, and rejects bad arguments on the host (these calls
return before any CUDA work, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_chunked_chunk_gb300 as gdn
from gated_deltanet_chunked_chunk_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(gdn.EXPORTED_SYMBOLS) == _declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        s = gdn.status_string(code)
        assert isinstance(s, str) and s
    assert gdn.status_string(999) == "unknown status"
    assert lib.gdn_version() >= 100


NULL = None


def _chunk(lib, **kw):
    a = dict(q=NULL, k=NULL, v=NULL, g=NULL, beta=NULL, scale=-1.0, h0=NULL, cu=NULL, N=1, B=1, T=8,
             H=2, HV=4, K=128, V=128, l2=1, o=NULL, ht=NULL, ws=NULL, wsb=0, st=NULL, stream=NULL)
    a.update(kw)
    return lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["cu"],
                             a["N"], a["B"], a["T"], a["H"], a["HV"], a["K"], a["V"], a["l2"], a["o"],
                             a["ht"], a["ws"], a["wsb"], a["st"], a["stream"])


def test_chunk_fwd_host_validation(lib):
    fake = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    assert _chunk(lib) == gdn.GDN_EINVAL                      # null tensors
    assert _chunk(lib, HV=3) == gdn.GDN_EINVAL                # HV % H != 0
    assert _chunk(lib, K=96, q=fake, k=fake, v=fake, g=fake, beta=fake, o=fake) == gdn.GDN_EUNSUPPORTED
    assert _chunk(lib, V=32) == gdn.GDN_EUNSUPPORTED
    assert _chunk(lib, cu=fake, B=2, N=3) == gdn.GDN_EINVAL   # varlen needs B == 1
    assert _chunk(lib, N=3) == gdn.GDN_EINVAL                 # dense needs N == B
    assert _chunk(lib, T=-1) == gdn.GDN_EINVAL
    assert _chunk(lib, N=0, B=0, T=0) == gdn.GDN_OK           # nothing to do, nothing launched


def test_chunk_fwd_launch_count_without_a_device(lib):
    # Shapes that never take the two-range path are answered on the host.
    assert gdn.chunk_fwd_kernel_launches(1, 8, 2, 4, 96, 128, 1, False) == -1   # K unsupported
    assert gdn.chunk_fwd_kernel_launches(1, 8, 2, 4, 128, 32, 1, False) == -1   # V unsupported
    assert gdn.chunk_fwd_kernel_launches(0, 0, 2, 4, 128, 128, 0, False) == 0
    assert gdn.chunk_fwd_kernel_launches(2, 100, 2, 4, 128, 128, 2, False) == 2  # prep + walk
    assert gdn.chunk_fwd_kernel_launches(1, 100, 2, 4, 128, 128, 3, True) == 3   # + the chunk-start table
    assert gdn.chunk_fwd_kernel_launches(2, 0, 2, 4, 128, 128, 2, False) == 1    # states only: the walk
    assert gdn.chunk_fwd_kernel_launches(1, 63 * 64, 2, 4, 128, 128, 1, False) == 2  # under 64 chunks


def test_chunk_misaligned_buffers_refused_before_launch(lib):
    """The prefill and backward move q, k, v, o, the states and their gradients
    with TMA, bulk copies and 16-byte accesses: a buffer that is only 8-byte
    aligned is refused on the host (the fake pointers are never dereferenced)."""
    ok = ctypes.c_void_p(64)
    odd = ctypes.c_void_p(64 + 8)
    base = dict(q=ok, k=ok, v=ok, g=ok, beta=ok, o=ok, ws=ok, wsb=1 << 40)
    for name in ("q", "k", "v", "o", "h0", "ht", "ws"):
        kw = dict(base)
        kw[name] = odd
        assert _chunk(lib, **kw) == gdn.GDN_EINVAL, name
    F = ctypes.c_float

    def bwd(**kw):
        a = dict(q=ok, k=ok, v=ok, g=ok, beta=ok, h0=NULL, cu=NULL, do=ok, dht=NULL, dq=ok, dk=ok, dv=ok, dg=ok,
                 dbeta=ok, dh0=NULL, ws=ok)
        a.update(kw)
        return lib.gdn_chunk_bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], F(-1.0), a["h0"], a["cu"], 1, 1, 8, 2,
                                 4, 128, 128, 1, a["do"], a["dht"], a["dq"], a["dk"], a["dv"], a["dg"], a["dbeta"],
                                 a["dh0"], a["ws"], ctypes.c_size_t(1 << 40), NULL, NULL)
    for name in ("q", "k", "v", "do", "dht", "h0", "dq", "dk", "dh0", "ws"):
        assert bwd(**{name: odd}) == gdn.GDN_EINVAL, name


def test_chunk_fwd_gated_host_validation(lib):
    fake = ctypes.c_void_p(16)

    def call(**kw):
        a = dict(q=fake, k=fake, v=fake, A_log=fake, a=fake, b=fake, dt=fake, scale=-1.0, h0=NULL, cu=NULL,
                 N=1, B=1, T=8, H=2, HV=4, K=128, V=128, l2=1, o=fake, ht=NULL, gout=NULL, bout=NULL,
                 ws=NULL, wsb=0, st=NULL, stream=NULL)
        a.update(kw)
        return lib.gdn_chunk_fwd_gated(a["q"], a["k"], a["v"], a["A_log"], a["a"], a["b"], a["dt"], a["scale"],
                                       a["h0"], a["cu"], a["N"], a["B"], a["T"], a["H"], a["HV"], a["K"],
                                       a["V"], a["l2"], a["o"], a["ht"], a["gout"], a["bout"], a["ws"],
                                       a["wsb"], a["st"], a["stream"])
    assert call(A_log=NULL) == gdn.GDN_EINVAL                 # no gate inputs at all
    assert call(b=NULL) == gdn.GDN_EINVAL                     # part of the gate group
    assert call(dt=NULL) == gdn.GDN_EINVAL
    assert call(gout=fake) == gdn.GDN_EINVAL                  # g copy without the beta copy
    assert call(bout=fake) == gdn.GDN_EINVAL
    assert call(HV=3) == gdn.GDN_EINVAL
    assert call(K=96) == gdn.GDN_EUNSUPPORTED
    assert call() == gdn.GDN_EWORKSPACE                       # T = 8 needs the record workspace
    assert call(N=0, B=0, T=0, A_log=NULL, a=NULL, b=NULL, dt=NULL) == gdn.GDN_OK


def test_decode_host_validation(lib):
    fake = ctypes.c_void_p(16)

    def call(**kw):
        a = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, A_log=NULL, a=NULL, b=NULL, dt=NULL,
                 scale=-1.0, l2=1, pool=fake, P=4, idx=fake, R=2, H=2, HV=4, K=128, V=128, o=fake,
                 st=NULL, stream=NULL)
        a.update(kw)
        return lib.gdn_recurrent_decode(a["q"], a["k"], a["v"], a["g"], a["beta"], a["A_log"], a["a"],
                                        a["b"], a["dt"], a["scale"], a["l2"], a["pool"], a["P"],
                                        a["idx"], a["R"], a["H"], a["HV"], a["K"], a["V"], a["o"],
                                        a["st"], a["stream"])
    assert call(pool=NULL) == gdn.GDN_EINVAL                  # missing pool: readable error, no crash
    assert call(idx=NULL) == gdn.GDN_EINVAL                   # missing indices
    assert call(A_log=fake, a=fake, b=fake, dt=fake) == gdn.GDN_EINVAL  # both gate groups
    assert call(g=NULL, beta=NULL) == gdn.GDN_EINVAL          # no gate group
    assert call(beta=NULL) == gdn.GDN_EINVAL                  # half a group
    assert call(HV=6, H=4) == gdn.GDN_EINVAL
    assert call(K=32) == gdn.GDN_EUNSUPPORTED
    assert call(R=0) == gdn.GDN_OK


def test_gating_host_validation(lib):
    assert lib.gdn_gating(NULL, NULL, NULL, NULL, 0, 4, NULL, NULL, NULL) == gdn.GDN_OK
    assert lib.gdn_gating(NULL, NULL, NULL, NULL, 5, 4, NULL, NULL, NULL) == gdn.GDN_EINVAL
    assert lib.gdn_gating(NULL, NULL, NULL, NULL, 5, 0, NULL, NULL, NULL) == gdn.GDN_EINVAL


def test_python_binding_checks_before_calling():
    import torch
    q = torch.zeros(1, 4, 2, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        gdn.gdn_chunk_fwd(q, q, q, q[..., 0], q[..., 0])
    with pytest.raises(ValueError):
        gdn.gdn_recurrent_decode(q, q, q, None, None)


def test_conv_host_validation(lib):
    NULL = None
    fake = ctypes.c_void_p(16)
    I64 = ctypes.c_int64

    def fwd(x=fake, w=fake, st=fake, P=2, S=3, qsl=fake, cache=fake, N=1, dim=8, total=5, W=4, act=1,
            out=fake):
        return lib.gdn_causal_conv1d_fwd(x, w, NULL, st, P, S, qsl, cache, NULL, N, dim, I64(total), W, act,
                                         out, NULL, NULL)

    assert fwd(N=0, total=0) == gdn.GDN_OK                     # nothing to do, nothing launched
    assert fwd(N=0) == gdn.GDN_EINVAL                          # tokens without a sequence
    assert fwd(qsl=NULL) == gdn.GDN_EINVAL
    assert fwd(w=NULL) == gdn.GDN_EINVAL
    assert fwd(x=NULL) == gdn.GDN_EINVAL
    assert fwd(st=NULL) == gdn.GDN_EINVAL                      # slots given but no pool
    assert fwd(act=2) == gdn.GDN_EINVAL
    assert fwd(W=9) == gdn.GDN_EUNSUPPORTED                    # width above 8
    assert fwd(S=2) == gdn.GDN_EUNSUPPORTED                    # state shorter than W - 1
    assert fwd(S=65) == gdn.GDN_EUNSUPPORTED

    def upd(x=fake, st=fake, w=fake, idx=fake, R=3, dim=8, W=4, S=3, out=fake):
        return lib.gdn_causal_conv1d_update(x, st, 2, S, w, NULL, idx, R, dim, W, 1, out, NULL, NULL)

    assert upd(R=0) == gdn.GDN_OK
    assert upd(idx=NULL) == gdn.GDN_EINVAL
    assert upd(st=NULL) == gdn.GDN_EINVAL
    assert upd(W=0) == gdn.GDN_EUNSUPPORTED
    assert upd(dim=0) == gdn.GDN_EINVAL

    def pack(q=fake, R=2, H=2, HV=4, K=8, V=8, W=4, S=3):
        return lib.gdn_conv_decode_pack(fake, fake, 2, S, fake, NULL, fake, R, H, HV, K, V, W, 1, q, fake, fake,
                                        NULL, NULL)

    assert pack(R=0) == gdn.GDN_OK
    assert pack(q=NULL) == gdn.GDN_EINVAL
    assert pack(H=0) == gdn.GDN_EINVAL
    assert pack(S=1) == gdn.GDN_EUNSUPPORTED


def test_decode_variants_host_validation(lib):
    NULL = None
    fake = ctypes.c_void_p(16)
    F = ctypes.c_float

    def bf16(pool=fake, idx=fake, R=2, K=128, g=fake):
        return lib.gdn_recurrent_decode_bf16(fake, fake, fake, g, fake, NULL, NULL, NULL, NULL, F(-1.0), 1, pool,
                                             4, idx, R, 2, 4, K, 128, fake, NULL, NULL)

    assert bf16(R=0) == gdn.GDN_OK
    assert bf16(pool=NULL) == gdn.GDN_EINVAL
    assert bf16(idx=NULL) == gdn.GDN_EINVAL
    assert bf16(K=96) == gdn.GDN_EUNSUPPORTED
    assert bf16(g=NULL) == gdn.GDN_EINVAL                      # half a gate group

    def mtp(cu=fake, rd=fake, wr=fake, N=2, Tt=6, ld=3, pool=fake):
        return lib.gdn_recurrent_decode_mtp(fake, fake, fake, fake, fake, NULL, NULL, NULL, NULL, F(-1.0), 1,
                                            pool, 8, cu, N, Tt, rd, wr, ld, NULL, 2, 4, 64, 64, fake, NULL, NULL)

    assert mtp(N=0) == gdn.GDN_OK
    assert mtp(cu=NULL) == gdn.GDN_EINVAL
    assert mtp(rd=NULL) == gdn.GDN_EINVAL
    assert mtp(wr=NULL) == gdn.GDN_EINVAL
    assert mtp(ld=0) == gdn.GDN_EINVAL
    assert mtp(pool=NULL) == gdn.GDN_EINVAL
    assert mtp(N=70000) == gdn.GDN_EUNSUPPORTED


def test_backward_binding_checks_shapes_before_calling():
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    v = torch.zeros(1, 8, 4, 64, dtype=torch.bfloat16)
    g = torch.zeros(1, 8, 4)
    with pytest.raises(ValueError):   # do has the wrong head count
        gdn.gdn_chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):   # g, beta must be [B,T,HV]
        gdn.gdn_chunk_bwd(q, q, v, g[..., :2], g[..., :2], v)
    with pytest.raises(ValueError):   # dht must be [N,HV,K,V]
        gdn.gdn_chunk_bwd(q, q, v, g, g, v, dht=torch.zeros(1, 4, 64, 32))


def test_misaligned_pool_and_grid_limits_refused_before_launch(lib):
    """A pool that is not 16-byte aligned (a view at an odd offset) would meet
    16-byte vector accesses and bulk copies on the device: every decode entry
    point refuses it on the host.  Request / sequence counts beyond the grid's
    65535 come back as GDN_EUNSUPPORTED.  No call below reaches a launch."""
    NULL = None
    fake = ctypes.c_void_p(16)
    odd = ctypes.c_void_p(16 + 8)     # 8-byte aligned, not 16
    F = ctypes.c_float

    def dec(pool=fake, R=2):
        return lib.gdn_recurrent_decode(fake, fake, fake, fake, fake, NULL, NULL, NULL, NULL, F(-1.0), 1, pool, 4,
                                        fake, R, 2, 4, 128, 128, fake, NULL, NULL)

    def bf16(pool=fake, R=2):
        return lib.gdn_recurrent_decode_bf16(fake, fake, fake, fake, fake, NULL, NULL, NULL, NULL, F(-1.0), 1, pool,
                                             4, fake, R, 2, 4, 128, 128, fake, NULL, NULL)

    def mtp(pool=fake):
        return lib.gdn_recurrent_decode_mtp(fake, fake, fake, fake, fake, NULL, NULL, NULL, NULL, F(-1.0), 1,
                                            pool, 8, fake, 2, 6, fake, fake, 3, NULL, 2, 4, 64, 64, fake, NULL,
                                            NULL)

    assert dec(pool=odd) == gdn.GDN_EINVAL
    assert bf16(pool=odd) == gdn.GDN_EINVAL
    assert mtp(pool=odd) == gdn.GDN_EINVAL
    assert dec(R=70000) == gdn.GDN_EUNSUPPORTED
    assert bf16(R=70000) == gdn.GDN_EUNSUPPORTED
    assert _chunk(lib, cu=fake, B=1, N=70000, q=fake, k=fake, v=fake, g=fake, beta=fake,
                  o=fake) == gdn.GDN_EUNSUPPORTED
    assert "65535" in gdn.status_string(gdn.GDN_EUNSUPPORTED)


def test_wait_expiry_hook_toggles(lib):
    assert lib.gdn_testing_force_wait_expiry(0) == 0
    assert lib.gdn_testing_force_wait_expiry(1) == 0
    assert gdn.testing_force_wait_expiry(False) is True
    assert lib.gdn_testing_force_wait_expiry(0) == 0


def test_conv_spec_host_validation(lib):
    NULL = None
    fake = ctypes.c_void_p(16)

    def call(S=6, m=3, Wd=4, N=2, x=fake, qsl=fake):
        return lib.gdn_causal_conv1d_update_spec(x, fake, 4, S, fake, NULL, fake, NULL, qsl, N, 8, m, 64, Wd, 1,
                                                 fake, NULL, NULL)

    assert call(N=0) == gdn.GDN_OK
    assert call(S=5) == gdn.GDN_EUNSUPPORTED        # state too short for width - 1 + mtp_step
    assert call(m=-1) == gdn.GDN_EINVAL
    assert call(x=NULL) == gdn.GDN_EINVAL
    assert call(qsl=NULL) == gdn.GDN_EINVAL
    assert call(N=70000) == gdn.GDN_EUNSUPPORTED
