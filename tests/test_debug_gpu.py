"""The index-checking build (libdecgemm_debug.so) on every kernel path, and
guard bands around the MoE block's outputs.

In the DEC_DEBUG build every index a kernel computes into a global buffer is
checked against the buffer's extent; an out-of-range access is skipped and
dec_sync_check returns DEC_EBOUNDS with the source line and index. These tests
run small cases of every projection regime and split, the MoE block (with and
without the shared expert, under skewed routing, with growing workspace
layouts) and the latent block through it, and expect no failed check and
results within the tolerance.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_within_tol, gap_rows, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_decode_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"


import moe_decode_gemm_gb300 as dg  # noqa: E402


_DEBUG = {}


@pytest.fixture
def debug_lib():
    """Route the binding to the index-checking build for one test."""
    if "lib" not in _DEBUG:
        _DEBUG["lib"] = dg._load(dg.DEBUG_LIB_PATH)
    old = dg.use_library(_DEBUG["lib"])
    assert dg.lib().dec_debug_build() == 1
    yield
    torch.cuda.synchronize()
    dg.use_library(old)


def _ok(what):
    rc = dg.sync_check()
    assert rc == dg.DEC_OK, "%s: %s, first failed check %s" % (what, dg.strerror(rc),
                                                             dg.check_site())


# projections: CUDA-core (whole-row slabs, cluster, stream-K), mma.sync (whole-row slabs,
# cluster, stream-K, 256-row tiles, forced split), tcgen05 (cluster, tile-aligned, stream-K),
# residual, row-strided input
PROJ = [(1, 4000, 1000, None), (2, 1000, 4104, None), (1, 7168, 7168, None),
        (5, 2048, 7168, None), (4, 7168, 7168, None), (16, 640, 1536, None),
        (9, 2048, 2048, 5), (33, 1900, 904, None), (64, 2048, 7168, None),
        (48, 7168, 2048, None), (17, 16384, 1024, None), (64, 300, 520, 3),
        (2, 2048, 4096, None), (1, 1100, 1024, None), (3, 2000, 7168, None),
        (4, 4096, 1088, None), (12, 4096, 1088, None), (16, 2000, 7168, None),
        (24, 1900, 6200, None), (6, 6000, 2048, None), (8, 8192, 2048, None)]


@pytest.mark.parametrize("M,N,K,S", PROJ)
@pytest.mark.parametrize("residual", [False, True])
def test_projection_paths_pass_the_index_checks(debug_lib, M, N, K, S, residual):
    if S is not None and residual:
        pytest.skip("forced splits take no residual")
    key = ("dbg", M, N, K)
    xb = wl.normal_bf16((M, K + 8), 1.0, *key, "x")
    Wb = wl.normal_bf16((N, K), 0.02, *key, "W")
    rb = wl.normal_bf16((M, N), 1.0, *key, "r") if residual else None
    xt = wl.bits_to_torch(xb)[:, :K]          # rows K + 8 apart: read in place
    W = wl.bits_to_torch(Wb)
    if S is None:
        y = dg.dec_linear(xt, W, residual=None if rb is None else wl.bits_to_torch(rb))
    else:
        y = dg.dec_linear_splitk(xt.contiguous(), W, S)
    _ok("projection M=%d N=%d K=%d S=%s" % (M, N, K, S))
    ref, A = oracle.linear(xb[:, :K], Wb)
    if residual:
        ref, A = oracle.residual(rb, ref, A)
    assert_within_tol(to_f64(y), ref, A, "debug projection")


def _block(M, H, E, I, k, key, shared=True, skew=0.0):
    Wr = (wl.skewed_router_bf16(E, H, skew, *key, "Wr") if skew else
          wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr"))
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"),
          wl.normal_bf16((H, I), 0.02, *key, "Ws2")) if shared else None
    return x, Wr, W13, W2, Ws


@pytest.mark.parametrize("M,H,E,I,k,shared,skew", [
    (1, 256, 32, 128, 8, True, 0.0), (5, 200, 24, 72, 3, True, 0.0),
    (16, 256, 64, 128, 8, False, 0.0), (33, 256, 64, 128, 8, True, 0.0),
    (64, 256, 64, 128, 8, True, 1.0), (64, 128, 1024, 64, 32, True, 0.0)])
def test_moe_block_passes_the_index_checks(debug_lib, M, H, E, I, k, shared, skew):
    x, Wr, W13, W2, Ws = _block(M, H, E, I, k, ("dbg-moe", M, E), shared, skew)
    t = wl.bits_to_torch
    res = wl.normal_bf16((M, H), 1.0, "dbg-moe", M, "res")
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    out = dg.moe_decode(t(x), t(Wr), t(W13), t(W2), None if Ws is None else t(Ws[0]),
                        None if Ws is None else t(Ws[1]), k, topk_idx=idx, residual=t(res))
    _ok("moe M=%d E=%d" % (M, E))
    r = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=Ws)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    ref, A = oracle.residual(res, r["out"], r["absref"])
    assert_within_tol(to_f64(out), ref, A, "debug moe")


def test_latent_blocks_with_a_growing_layout_pass_the_index_checks(debug_lib):
    # latent widths 128 then 200 (a larger layout inside the same workspace)
    for M, H, L, E, I, k in [(12, 256, 128, 32, 128, 4), (12, 128, 200, 24, 64, 3)]:
        key = ("dbg-latent", L)
        Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
        Wd = wl.normal_bf16((L, H), 1.0 / math.sqrt(H), *key, "Wd")
        x, _ = gap_rows(Wr, M, H, k, *key, "x")
        W13 = np.stack([wl.normal_bf16((2 * I, L), 0.02, *key, "W13", e) for e in range(E)])
        W2 = np.stack([wl.normal_bf16((L, I), 0.02, *key, "W2", e) for e in range(E)])
        Wup = wl.normal_bf16((H, L), 0.02, *key, "Wup")
        Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"),
              wl.normal_bf16((H, I), 0.02, *key, "Ws2"))
        t = wl.bits_to_torch
        Wrl = np.concatenate([Wr, Wd])
        out = dg.moe_decode_latent(t(x), t(Wrl), t(W13), t(W2), t(Wup), t(Ws[0]), t(Ws[1]), k)
        _ok("latent L=%d" % L)
        r = oracle.moe_latent(x, Wrl, E, lambda e: (W13[e], W2[e]), k, I, Wup, shared=Ws)
        assert_within_tol(to_f64(out), r["out"], r["absref"], "debug latent L=%d" % L)


# ---------------------------------------------------------------- guard bands
def test_moe_outputs_guard_bands_untouched():
    # the block writes exactly out [M,H], topk_idx [M,k] and topk_w [M,k]:
    # sentinel words around each stay intact (release build)
    M, H, E, I, k = 7, 256, 32, 128, 4
    x, Wr, W13, W2, Ws = _block(M, H, E, I, k, ("guard-moe",))
    t = wl.bits_to_torch
    pad = 4096
    bo = torch.full((pad + M * H + pad,), 12345, dtype=torch.int16, device="cuda")
    bi = torch.full((pad + M * k + pad,), 777, dtype=torch.int32, device="cuda")
    bw = torch.full((pad + M * k + pad,), -3.0, dtype=torch.float32, device="cuda")
    out = bo[pad:pad + M * H].view(torch.bfloat16).view(M, H)
    idx = bi[pad:pad + M * k].view(M, k)
    gw = bw[pad:pad + M * k].view(M, k)
    dg.moe_decode(t(x), t(Wr), t(W13), t(W2), t(Ws[0]), t(Ws[1]), k, out=out, topk_idx=idx,
                  topk_w=gw)
    assert dg.sync_check() == dg.DEC_OK
    for b, v in ((bo, 12345), (bi, 777)):
        assert torch.all(b[:pad] == v) and torch.all(b[-pad:] == v)
    assert torch.all(bw[:pad] == -3.0) and torch.all(bw[-pad:] == -3.0)
    r = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=Ws)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert_within_tol(to_f64(out), r["out"], r["absref"], "guarded moe")
