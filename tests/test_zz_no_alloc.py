"""dec_linear_noalloc, the projection entry point that allocates nothing.

Some callers of this library cannot allocate device memory: a framework whose
caching allocator has already reserved the GPU, an engine whose memory budget
is fixed before the first request, or a latency-critical loop in which
cudaMalloc (which may synchronise the device) must never run. This entry point
keeps its split-K scratch in a fixed array inside the library instead. Its
output must match the fp64 oracle within the tolerance every projection test
uses, call after call; a call must leave the device's free memory unchanged;
and dec_sync_check must report its status without setting anything up.

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
                                   (16, 640, 1536), (16, 16384, 7168)])
def test_no_alloc_matches_oracle_on_two_calls(M, N, K):
    xb = wl.normal_bf16((M, K), 1.0, "noalloc", M, N, "x")
    Wb = wl.normal_bf16((N, K), 0.02, "noalloc", M, N, "W")
    x, W = wl.bits_to_torch(xb), wl.bits_to_torch(Wb)
    ref, A = oracle.linear(xb, Wb)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(x, W, y) == dg.DEC_OK
        torch.cuda.synchronize()
        assert dg.sync_check() == dg.DEC_OK
        assert_within_tol(to_f64(y), ref, A, "noalloc call %d M=%d N=%d K=%d" % (call, M, N, K))


@pytest.mark.parametrize("M", [2, 16])
def test_no_alloc_leaves_free_memory_unchanged(M):
    # One call on a small shape first (the same kernel, so that its code is
    # loaded), then a call on the largest shape the entry point takes: the
    # device's free memory is the same before and after it. Every tensor is
    # allocated before the first reading.
    small = [wl.bits_to_torch(wl.normal_bf16(s, 0.02, "noalloc-mem", M, i))
             for i, s in enumerate([(M, 512), (256, 512)])]
    ys = torch.empty((M, 256), dtype=torch.bfloat16, device="cuda")
    N, K = 16384, 7168
    xb = wl.normal_bf16((M, K), 1.0, "noalloc-mem", M, "x")
    Wb = wl.normal_bf16((N, K), 0.02, "noalloc-mem", M, "W")
    x, W = wl.bits_to_torch(xb), wl.bits_to_torch(Wb)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(small[0], small[1], ys) == dg.DEC_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _call_noalloc(x, W, y) == dg.DEC_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "free device memory changed by %d bytes" % (free0 - free1)
    cols = np.arange(0, N, 97)
    ref, A = oracle.linear(xb, Wb[cols])
    assert_within_tol(to_f64(y)[:, cols], ref, A, "noalloc largest shape M=%d" % M)


def test_no_alloc_rejects_sizes_beyond_its_limits():
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected first
    p = ctypes.c_void_p(fake.data_ptr())
    L = dg.lib()
    assert L.dec_linear_noalloc(p, p, p, 17, 128, 128, None) == dg.DEC_EUNSUPPORTED
    assert L.dec_linear_noalloc(p, p, p, 1, 16384 * 128 + 1, 128, None) == dg.DEC_EUNSUPPORTED
    assert L.dec_linear_noalloc(None, p, p, 1, 128, 128, None) == dg.DEC_EINVAL
