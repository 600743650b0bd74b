"""dec_linear_noalloc, the projection entry point that allocates nothing.

Callers that cannot allocate device memory -- a framework whose caching
allocator already owns the GPU, an engine with a memory budget fixed up front,
or a latency-critical loop where cudaMalloc may not run -- use this entry
point; its split-K scratch is a fixed array inside the library. Its output must
match dec_linear's within the tolerance the other tests use, call after call.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_within_tol, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_decode_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"


import moe_decode_gemm_gb300 as dg  # noqa: E402


def _call_noalloc(x, W, y):
    """Through the C ABI directly."""
    M, K = x.shape
    N = W.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return dg.lib().dec_linear_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                       ctypes.c_void_p(y.data_ptr()), M, N, K, stream)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (2, 1000, 4104), (5, 2048, 7168),
                                   (16, 640, 1536)])
def test_no_alloc_matches_dec_linear_on_two_calls(M, N, K):
    xb = wl.normal_bf16((M, K), 1.0, "noalloc", M, N, "x")
    Wb = wl.normal_bf16((N, K), 0.02, "noalloc", M, N, "W")
    x, W = wl.bits_to_torch(xb), wl.bits_to_torch(Wb)
    ref = dg.dec_linear(x, W)                      # the allocating entry point
    assert dg.sync_check() == dg.DEC_OK
    _, A = oracle.linear(xb, Wb)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(x, W, y) == dg.DEC_OK
        torch.cuda.synchronize()
        assert_within_tol(to_f64(y), to_f64(ref), A, "noalloc call %d M=%d" % (call, M))


def test_no_alloc_rejects_sizes_beyond_its_limits():
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected first
    p = ctypes.c_void_p(fake.data_ptr())
    L = dg.lib()
    assert L.dec_linear_noalloc(p, p, p, 17, 128, 128, None) == dg.DEC_EUNSUPPORTED
    assert L.dec_linear_noalloc(p, p, p, 1, 16384 * 128 + 1, 128, None) == dg.DEC_EUNSUPPORTED
    assert L.dec_linear_noalloc(None, p, p, 1, 128, 128, None) == dg.DEC_EINVAL
