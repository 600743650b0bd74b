"""Seeded random projection shapes through every dispatcher path.

Each case draws M (1-64), N, K (a multiple of 8; often of 64, so that the
whole-row slabs apply), an optional residual and an optional row stride for x,
runs dec_linear through the C ABI, and compares a sample of output columns
with the fp64 oracle at the stated tolerance. The shapes are chosen so that
every kernel family appears: whole-row slabs (CUDA cores and mma.sync), the
cluster splits, stream-K on CUDA cores / mma.sync / tcgen05, and the
tile-aligned tcgen05 split.
"""
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


def _shape(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 17, 24, 32, 40, 64]))
    N = int(rng.choice([int(rng.integers(1, 600)), int(rng.integers(900, 5000)), 2048, 4096]))
    K = int(rng.choice([64 * int(rng.integers(1, 128)), 8 * int(rng.integers(1, 1024))]))
    residual = bool(rng.integers(0, 2))
    ldx = K + 8 * int(rng.integers(0, 4)) if rng.integers(0, 3) == 0 else 0
    return M, N, K, residual, ldx


SEEDS = list(range(48))


@pytest.mark.parametrize("seed", SEEDS)
def test_random_projection_matches_oracle(seed):
    M, N, K, residual, ldx = _shape(seed)
    key = ("fuzz", seed)
    wide = wl.normal_bf16((M, ldx or K), 1.0, *key, "x")
    W = wl.normal_bf16((N, K), 0.02, *key, "W")
    r = wl.normal_bf16((M, N), 1.0, *key, "r") if residual else None
    xt = wl.bits_to_torch(wide)[:, :K]
    y = dg.dec_linear(xt, wl.bits_to_torch(W), residual=None if r is None else wl.bits_to_torch(r))
    assert dg.sync_check() == dg.DEC_OK
    cols = np.sort(np.random.default_rng(seed + 1000).choice(N, min(N, 256), replace=False))
    ref, A = oracle.linear(wide[:, :K], W[cols])
    if r is not None:
        ref, A = oracle.residual(r[:, cols], ref, A)
    assert_within_tol(to_f64(y)[:, cols], ref, A,
                      "fuzz seed %d: M=%d N=%d K=%d residual=%s ldx=%d %s" %
                      (seed, M, N, K, residual, ldx, dg.last_choice()))


def test_random_shapes_reach_every_kernel_family():
    # the draws above cover slabs, clusters and stream-K in every regime
    seen = set()
    for seed in SEEDS:
        M, N, K, residual, ldx = _shape(seed)
        x = torch.zeros((M, ldx or K), dtype=torch.bfloat16, device="cuda")[:, :K]
        W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
        dg.dec_linear(x, W)
        regime, _ = dg.last_choice()
        seen.add((regime, "slab" if dg.last_slab() else "cluster" if dg.last_cluster() else "split"))
    assert dg.sync_check() == dg.DEC_OK
    for want in [("mma", "slab"), ("smallm", "split"), ("mma", "split"), ("tc", "split"),
                 ("tc", "cluster")]:
        assert want in seen, (want, sorted(seen))


def _wide_shape(seed):
    # 1-16 tokens over 4865-9728 rows: the 48- and 64-row slabs, and split-K
    # where K is not a multiple of 64
    rng = np.random.default_rng(20_000 + seed)
    M = int(rng.integers(1, 17))
    N = int(rng.integers(4865, 9729))
    K = int(rng.choice([64 * int(rng.integers(8, 128)), 8 * int(rng.integers(64, 1024))]))
    residual = bool(rng.integers(0, 2))
    ldx = K + 8 * int(rng.integers(1, 4)) if rng.integers(0, 3) == 0 else 0
    return M, N, K, residual, ldx


WIDE_SEEDS = list(range(16))


@pytest.mark.parametrize("seed", WIDE_SEEDS)
def test_random_wide_projection_matches_oracle(seed):
    M, N, K, residual, ldx = _wide_shape(seed)
    key = ("fuzz-wide", seed)
    wide = wl.normal_bf16((M, ldx or K), 1.0, *key, "x")
    W = wl.normal_bf16((N, K), 0.02, *key, "W")
    r = wl.normal_bf16((M, N), 1.0, *key, "r") if residual else None
    xt = wl.bits_to_torch(wide)[:, :K]
    y = dg.dec_linear(xt, wl.bits_to_torch(W), residual=None if r is None else wl.bits_to_torch(r))
    assert dg.sync_check() == dg.DEC_OK
    if K % 64 == 0:
        rows = -(-N // dg.last_grid())
        assert dg.last_slab() and rows in (48, 64), (M, N, K, rows)
    cols = np.sort(np.random.default_rng(seed + 3000).choice(N, 256, replace=False))
    ref, A = oracle.linear(wide[:, :K], W[cols])
    if r is not None:
        ref, A = oracle.residual(r[:, cols], ref, A)
    assert_within_tol(to_f64(y)[:, cols], ref, A,
                      "wide fuzz seed %d: M=%d N=%d K=%d residual=%s ldx=%d %s" %
                      (seed, M, N, K, residual, ldx, dg.last_choice()))


def test_random_wide_shapes_reach_both_slab_widths():
    seen = set()
    for seed in WIDE_SEEDS:
        M, N, K, _, _ = _wide_shape(seed)
        if K % 64 == 0:
            seen.add(48 if N <= 48 * 152 else 64)
    assert seen == {48, 64}, seen


# ---------------------------------------------------------------- MoE blocks
def _moe_shape(seed):
    rng = np.random.default_rng(10_000 + seed)
    M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 24, 33, 48, 64]))
    E = int(rng.choice([8, 16, 40, 64, 128, 200, 384]))
    k = int(min(E, rng.choice([1, 2, 4, 6, 8, 12])))
    H = 8 * int(rng.integers(16, 80))        # 128-632
    I = 8 * int(rng.integers(16, 48))        # 128-376
    shared = bool(rng.integers(0, 2))
    residual = bool(rng.integers(0, 2))
    return M, E, k, H, I, shared, residual


@pytest.mark.parametrize("seed", list(range(16)))
def test_random_moe_block_matches_oracle(seed):
    import math
    from _util import gap_rows
    M, E, k, H, I, shared, residual = _moe_shape(seed)
    key = ("fuzz-moe", seed)
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"),
          wl.normal_bf16((H, I), 0.02, *key, "Ws2")) if shared else None
    res = wl.normal_bf16((M, H), 1.0, *key, "res") if residual else None
    t = wl.bits_to_torch
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    out = dg.moe_decode(t(x), t(Wr), t(W13), t(W2), None if Ws is None else t(Ws[0]),
                        None if Ws is None else t(Ws[1]), k, topk_idx=idx,
                        residual=None if res is None else t(res))
    assert dg.sync_check() == dg.DEC_OK
    r = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=Ws)
    what = "fuzz moe seed %d: M=%d E=%d k=%d H=%d I=%d shared=%s residual=%s" % (
        seed, M, E, k, H, I, shared, residual)
    assert np.array_equal(idx.cpu().numpy(), r["idx"]), what + ": chosen experts differ"
    ref, A = r["out"], r["absref"]
    if res is not None:
        ref, A = oracle.residual(res, ref, A)
    assert_within_tol(to_f64(out), ref, A, what)
