"""GPU parity of the latent MoE block against the fp64 oracle.

The router scores and the latent input projection are one product over a
stacked [E + L, H] weight; the routed experts work on the latent width L;
their gate-weighted sum is projected back to the hidden width, and the shared
expert (on x) and the residual are added. Token rows are drawn so that the
router scores of every token have gaps of at least 1e-3 among the k+1
largest: the chosen experts must equal the oracle's exactly.
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


def _block(M, H, L, E, I, k, key, shared=True):
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    Wd = wl.normal_bf16((L, H), 1.0 / math.sqrt(H), *key, "Wd")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, L), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((L, I), 0.02, *key, "W2", e) for e in range(E)])
    Wup = wl.normal_bf16((H, L), 0.02, *key, "Wup")
    Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"),
          wl.normal_bf16((H, I), 0.02, *key, "Ws2")) if shared else None
    return x, np.concatenate([Wr, Wd]), W13, W2, Wup, Ws


def _check(x, Wrl, W13, W2, Wup, Ws, k, what, res=None):
    t = wl.bits_to_torch
    M = x.shape[0]
    E = W13.shape[0]
    I = W13.shape[1] // 2
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    gw = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    out = dg.moe_decode_latent(t(x), t(Wrl), t(W13), t(W2), t(Wup),
                               None if Ws is None else t(Ws[0]), None if Ws is None else t(Ws[1]),
                               k, topk_idx=idx, topk_w=gw,
                               residual=None if res is None else t(res))
    assert dg.sync_check() == dg.DEC_OK
    r = oracle.moe_latent(x, Wrl, E, lambda e: (W13[e], W2[e]), k, I, Wup, shared=Ws)
    assert np.array_equal(idx.cpu().numpy(), r["idx"]), what + ": chosen experts differ"
    np.testing.assert_allclose(gw.cpu().numpy(), r["gates"], rtol=2e-5, atol=1e-7)
    ref, A = r["out"], r["absref"]
    if res is not None:
        ref, A = oracle.residual(res, ref, A)
    assert_within_tol(to_f64(out), ref, A, what)


@pytest.mark.parametrize("M", [1, 2, 5, 16, 33, 64])
@pytest.mark.parametrize("shared", [True, False])
def test_small_latent_block(M, shared):
    # a latent width of 128: the rounding of z and of the experts' hidden
    # vectors is absorbed by the 1e-3 * A term when the contractions after
    # them are a hundred terms long or more (at 64 the bf16 rounding points
    # alone reach the bound)
    blk = _block(M, 256, 128, 32, 128, 4, ("latent", M, shared), shared=shared)
    _check(*blk, 4, "latent M=%d shared=%s" % (M, shared))


def test_latent_wider_than_hidden_and_residual():
    # L > H is allowed (the experts' width is the latent one); residual fused
    M, H, L, E, I, k = 12, 128, 200, 24, 64, 3
    blk = _block(M, H, L, E, I, k, ("latent-wide",))
    res = wl.normal_bf16((M, H), 1.0, "latent-wide", "res")
    _check(*blk, k, "L > H with residual", res=res)


def test_latent_bad_arguments_are_rejected():
    fake = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    p = fake.data_ptr()
    L = dg.lib()
    import ctypes
    P = ctypes.c_void_p
    args = lambda Lw, Wup: (P(p), P(p), P(p), P(p), Wup, None, None, None, P(p), 4, 64, Lw, 16,
                            4, 64, None, None, None)
    assert L.moe_decode_latent(*args(0, P(p))) == dg.DEC_EINVAL
    assert L.moe_decode_latent(*args(12, P(p))) == dg.DEC_EINVAL      # L % 8
    assert L.moe_decode_latent(*args(64, None)) == dg.DEC_EINVAL      # no up-projection


# ---------------------------------------------------------------- full hidden size
H, E, K8, I = wl.HIDDEN, wl.EXPERTS, wl.TOPK, wl.INTER
LAT = 512


@pytest.fixture(scope="module")
def latent_bank():
    """A full-size block (hidden 7168, 384 experts, top-8, intermediate 2048,
    shared expert) with the routed experts on a 512-wide latent."""
    W13 = wl.normal_bf16_cuda((E, 2 * I, LAT), wl.WEIGHT_STD, "latent-bank", "W13")
    W2 = wl.normal_bf16_cuda((E, LAT, I), wl.WEIGHT_STD, "latent-bank", "W2")
    Ws13 = wl.normal_bf16_cuda((2 * I, H), wl.WEIGHT_STD, "latent-bank", "Ws13")
    Ws2 = wl.normal_bf16_cuda((H, I), wl.WEIGHT_STD, "latent-bank", "Ws2")
    Wup = wl.normal_bf16_cuda((H, LAT), wl.WEIGHT_STD, "latent-bank", "Wup")
    Wr = wl.normal_bf16((E, H), wl.ROUTER_STD, "latent-bank", "Wr")
    Wd = wl.normal_bf16((LAT, H), wl.ROUTER_STD, "latent-bank", "Wd")
    yield W13, W2, Ws13, Ws2, Wup, np.concatenate([Wr, Wd])
    del W13, W2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_full_hidden_latent_block(latent_bank, M):
    W13, W2, Ws13, Ws2, Wup, Wrl_bits = latent_bank
    x_bits, _ = gap_rows(Wrl_bits[:E], M, H, K8, "latent-full", M)
    t = wl.bits_to_torch
    idx = torch.empty((M, K8), dtype=torch.int32, device="cuda")
    res_bits = wl.normal_bf16((M, H), 1.0, "latent-full", M, "res")
    out = dg.moe_decode_latent(t(x_bits), t(Wrl_bits), W13, W2, Wup, Ws13, Ws2, K8,
                               topk_idx=idx, residual=t(res_bits))
    assert dg.sync_check() == dg.DEC_OK
    tokens = sorted(set([0, M // 3, M // 2, M - 1]))
    fetch = lambda e: (wl.torch_to_bits(W13[e]), wl.torch_to_bits(W2[e]))
    r = oracle.moe_latent(x_bits, Wrl_bits, E, fetch, K8, I, wl.torch_to_bits(Wup),
                          shared=(wl.torch_to_bits(Ws13), wl.torch_to_bits(Ws2)), tokens=tokens)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    ref, A = oracle.residual(res_bits, r["out"], r["absref"])
    assert_within_tol(to_f64(out)[tokens], ref[tokens], A[tokens], "latent full M=%d" % M)


@pytest.mark.parametrize("shared,residual", [(False, False), (True, False), (False, True)])
def test_full_hidden_latent_block_slab_tail_variants(latent_bank, shared, residual):
    # 1-16 tokens at hidden 7168: the up-projection runs on whole-row slabs
    # after the join, adding the shared expert's output (when there is one)
    # and the residual (when given) in its epilogue
    W13, W2, Ws13, Ws2, Wup, Wrl_bits = latent_bank
    M = 8
    x_bits, _ = gap_rows(Wrl_bits[:E], M, H, K8, "latent-tail", shared, residual)
    t = wl.bits_to_torch
    idx = torch.empty((M, K8), dtype=torch.int32, device="cuda")
    res_bits = wl.normal_bf16((M, H), 1.0, "latent-tail", "res") if residual else None
    out = dg.moe_decode_latent(t(x_bits), t(Wrl_bits), W13, W2, Wup, Ws13 if shared else None,
                               Ws2 if shared else None, K8, topk_idx=idx,
                               residual=t(res_bits) if residual else None)
    assert dg.sync_check() == dg.DEC_OK
    tokens = [0, 3, 7]
    fetch = lambda e: (wl.torch_to_bits(W13[e]), wl.torch_to_bits(W2[e]))
    sh = (wl.torch_to_bits(Ws13), wl.torch_to_bits(Ws2)) if shared else None
    r = oracle.moe_latent(x_bits, Wrl_bits, E, fetch, K8, I, wl.torch_to_bits(Wup), shared=sh,
                          tokens=tokens)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    ref, A = r["out"], r["absref"]
    if residual:
        ref, A = oracle.residual(res_bits, ref, A)
    assert_within_tol(to_f64(out)[tokens], ref[tokens], A[tokens],
                      "latent tail shared=%s residual=%s" % (shared, residual))
