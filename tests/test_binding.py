"""The binding rejects tensors the C ABI would misread, before any C call.

The ABI sees only pointers and sizes: a float32 or transposed weight, an
output of the wrong shape or a host tensor would be silently misread there.
CPU only: every check runs before the library is touched.
"""
import pytest

import moe_decode_gemm_gb300 as dg

torch = pytest.importorskip("torch")

bf = torch.bfloat16


def _t(*shape, dtype=bf):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("kw,exc,msg", [
    (dict(x=_t(2, 64, dtype=torch.float32)), TypeError, "x: expected torch.bfloat16"),
    (dict(W=_t(16, 64, dtype=torch.float16)), TypeError, "W: expected torch.bfloat16"),
    (dict(W=_t(16, 32)), ValueError, "W: expected [N, 64]"),
    (dict(W=_t(64, 16).t()), ValueError, "W: must be contiguous"),
    (dict(y=_t(2, 15)), ValueError, "y: expected shape (2, 16)"),
    (dict(residual=_t(3, 16)), ValueError, "residual: expected shape (2, 16)"),
    (dict(x=_t(64, 2).t()), ValueError, "unit column stride"),
    (dict(), ValueError, "expected a CUDA tensor"),
])
def test_dec_linear_rejects(kw, exc, msg):
    a = dict(x=_t(2, 64), W=_t(16, 64), y=_t(2, 16), residual=None)
    a.update(kw)
    with pytest.raises(exc) as e:
        dg.dec_linear(a["x"], a["W"], a["y"], residual=a["residual"])
    assert msg in str(e.value)


@pytest.mark.parametrize("fn", [dg.dec_linear_splitk, dg.dec_linear_noalloc])
def test_splitk_and_noalloc_reject(fn):
    args = (_t(2, 64), _t(16, 64, dtype=torch.float32))
    with pytest.raises(TypeError):
        fn(*args, 2, _t(2, 16)) if fn is dg.dec_linear_splitk else fn(*args, _t(2, 16))
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        fn(_t(2, 64), _t(16, 64), 2, _t(2, 16)) if fn is dg.dec_linear_splitk else \
            fn(_t(2, 64), _t(16, 64), _t(2, 16))


def _moe_args(**kw):
    M, H, E, I, k = 3, 64, 8, 32, 2
    a = dict(x=_t(M, H), Wr=_t(E, H), W13=_t(E, 2 * I, H), W2=_t(E, H, I), Ws13=_t(2 * I, H),
             Ws2=_t(H, I), topk=k, out=_t(M, H), topk_idx=_t(M, k, dtype=torch.int32),
             topk_w=_t(M, k, dtype=torch.float32), residual=None)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,exc,msg", [
    (dict(Wr=_t(8, 63)), ValueError, "Wr: expected [E, 64]"),
    (dict(W13=_t(8, 64, 64).transpose(1, 2)), ValueError, "W13: must be contiguous"),
    (dict(W13=_t(7, 64, 64)), ValueError, "W13: expected [8, 2I, 64]"),
    (dict(W2=_t(8, 32, 64)), ValueError, "W2: expected shape (8, 64, 32)"),
    (dict(W2=_t(8, 64, 32, dtype=torch.float32)), TypeError, "W2: expected torch.bfloat16"),
    (dict(Ws2=None), ValueError, "give both or neither"),
    (dict(Ws13=_t(32, 64)), ValueError, "Ws13: expected shape (64, 64)"),
    (dict(out=_t(3, 32)), ValueError, "out: expected shape (3, 64)"),
    (dict(topk_idx=_t(3, 2, dtype=torch.int64)), TypeError, "topk_idx: expected torch.int32"),
    (dict(topk_w=_t(3, 3, dtype=torch.float32)), ValueError, "topk_w: expected shape (3, 2)"),
    (dict(residual=_t(2, 64)), ValueError, "residual: expected shape (3, 64)"),
    (dict(), ValueError, "expected a CUDA tensor"),
])
def test_moe_decode_rejects(kw, exc, msg):
    a = _moe_args(**kw)
    with pytest.raises(exc) as e:
        dg.moe_decode(a["x"], a["Wr"], a["W13"], a["W2"], a["Ws13"], a["Ws2"], a["topk"],
                      out=a["out"], topk_idx=a["topk_idx"], topk_w=a["topk_w"],
                      residual=a["residual"])
    assert msg in str(e.value)


def test_dec_add_rejects():
    with pytest.raises(ValueError, match="expected shape"):
        dg.dec_add(_t(8), _t(9))
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        dg.dec_add(_t(8), _t(8))
