"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/decgemm.h declares, and rejects bad arguments with the
documented codes before touching CUDA."""
import ctypes
import os

import pytest

import moe_decode_gemm_gb300 as dg
from _util import header_functions
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "decgemm.h")


@pytest.fixture(scope="module")
def L():
    from moe_decode_gemm_gb300 import build
    build.build()
    return dg.lib()


def test_exports_every_declared_function(L):
    declared = header_functions(HEADER)
    assert len(declared) >= 18
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(declared) == sorted(dg.EXPORTS)


def test_version_and_strerror(L):
    assert L.dec_version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6, -99):
        assert isinstance(dg.strerror(code), str) and dg.strerror(code)


A = ctypes.c_void_p(1 << 20)        # aligned fake pointers: never dereferenced
MIS = ctypes.c_void_p((1 << 20) + 8)


@pytest.mark.parametrize("args,code", [
    ((None, A, A, 1, 16, 64), dg.DEC_EINVAL),
    ((A, None, A, 1, 16, 64), dg.DEC_EINVAL),
    ((A, A, None, 1, 16, 64), dg.DEC_EINVAL),
    ((A, A, A, 0, 16, 64), dg.DEC_EINVAL),
    ((A, A, A, 1, 0, 64), dg.DEC_EINVAL),
    ((A, A, A, 1, 16, 12), dg.DEC_EINVAL),     # K % 8 != 0
    ((A, A, A, 1, 16, 4), dg.DEC_EINVAL),
    ((MIS, A, A, 1, 16, 64), dg.DEC_EINVAL),   # misaligned
    ((A, MIS, A, 1, 16, 64), dg.DEC_EINVAL),
    ((A, A, A, 65, 16, 64), dg.DEC_EUNSUPPORTED),
])
def test_linear_rejects(L, args, code):
    assert L.dec_linear(*args, None) == code


@pytest.mark.parametrize("ldx", [0, -8, 32, 68, 100])
def test_linear_ex_rejects_bad_row_stride(L, ldx):
    # K = 64: the row stride must be >= K and a multiple of 8
    assert L.dec_linear_ex(A, ldx, A, None, A, 1, 16, 64, None) == dg.DEC_EINVAL


def test_splitk_rejects_bad_split(L):
    assert L.dec_linear_splitk(A, A, A, 4, 16, 64, 0, None) == dg.DEC_EINVAL
    assert L.dec_linear_splitk(A, A, A, 4, 16, 64, 2, None) == dg.DEC_EINVAL  # S > K/64


def test_residual_requires_residual(L):
    assert L.dec_linear_residual(A, A, None, A, 1, 16, 64, None) == dg.DEC_EINVAL


def _moe(L, **kw):
    a = dict(x=A, Wr=A, W13=A, W2=A, Ws13=A, Ws2=A, out=A, M=4, H=64, E=16, topk=4, I=64,
             idx=None, w=None)
    a.update(kw)
    return L.moe_decode(a["x"], a["Wr"], a["W13"], a["W2"], a["Ws13"], a["Ws2"], a["out"],
                        a["M"], a["H"], a["E"], a["topk"], a["I"], a["idx"], a["w"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), dg.DEC_EINVAL),
    (dict(W2=None), dg.DEC_EINVAL),
    (dict(Ws13=None), dg.DEC_EINVAL),          # shared expert half given
    (dict(M=0), dg.DEC_EINVAL),
    (dict(H=60), dg.DEC_EINVAL),
    (dict(I=12), dg.DEC_EINVAL),
    (dict(topk=0), dg.DEC_EINVAL),
    (dict(out=MIS), dg.DEC_EINVAL),
    (dict(M=65), dg.DEC_EUNSUPPORTED),
    (dict(topk=17, E=16), dg.DEC_EUNSUPPORTED),
    (dict(topk=33, E=64), dg.DEC_EUNSUPPORTED),
    (dict(E=1025), dg.DEC_EUNSUPPORTED),
])
def test_moe_rejects(L, kw, code):
    assert _moe(L, **kw) == code


def test_moe_residual_requires_residual(L):
    rc = L.moe_decode_residual(A, A, A, A, None, None, None, A, 4, 64, 16, 4, 64, None, None, None)
    assert rc == dg.DEC_EINVAL


def test_prefetch_and_add_reject(L):
    assert L.l2_prefetch(None, 4096, None) == dg.DEC_EINVAL
    assert L.l2_prefetch(MIS, 4096, None) == dg.DEC_EINVAL
    assert L.l2_prefetch(A, 8, None) == dg.DEC_OK       # rounds down to nothing
    assert L.dec_add(None, A, A, 16, None) == dg.DEC_EINVAL
    assert L.dec_add(A, A, A, 0, None) == dg.DEC_OK


def test_regime_report_before_any_call(L):
    import threading
    out = []
    t = threading.Thread(target=lambda: out.append(L.dec_last_choice()))
    t.start()
    t.join()
    assert out == [dg.REGIME_NONE]


def test_wait_timeout_setting_round_trips(L):
    old = L.dec_set_wait_timeout_ns(123456)
    assert L.dec_set_wait_timeout_ns(old) == 123456
