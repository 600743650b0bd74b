"""GPU parity of the decode projection y = x·Wᵀ against the fp64 oracle.

Every call goes through the C ABI (the ctypes binding). Each test asserts the
kernel regime the dispatcher chose, so a silent change of path shows.
"""
import os

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


def _expect_regime(M):
    """The split-K kernels' regime for M tokens."""
    return "smallm" if M <= 2 else ("mma" if M <= 16 else "tc")


def _expect_path(M):
    """The regime of the last call: whole-row slabs of 1-16 tokens run on mma.sync."""
    return "mma" if dg.last_slab() and M <= 16 else _expect_regime(M)


def _gpu_linear(x_bits, W_bits, S=None, res_bits=None):
    x = wl.bits_to_torch(x_bits)
    W = wl.bits_to_torch(W_bits)
    res = None if res_bits is None else wl.bits_to_torch(res_bits)
    if S is None:
        y = dg.dec_linear(x, W, residual=res)
    else:
        y = dg.dec_linear_splitk(x, W, S)
    choice = dg.last_choice()
    assert dg.sync_check() == dg.DEC_OK
    return y, choice


def _check_random(M, N, K, key, cols=None, S=None):
    x = wl.normal_bf16((M, K), 1.0, *key, "x")
    W = wl.normal_bf16((N, K), 0.02, *key, "W")
    y, choice = _gpu_linear(x, W, S=S)
    if cols is None:
        ref, A = oracle.linear(x, W)
        got = to_f64(y)
    else:
        ref, A = oracle.linear(x, W[cols])
        got = to_f64(y)[:, cols]
    assert_within_tol(got, ref, A, "M=%d N=%d K=%d S=%s" % (M, N, K, S))
    return y, choice


def test_single_projection_m1_4096():
    # M=1, K=N=4096, x ~N(0,1), W ~N(0,0.02), seed 0
    _, (regime, split) = _check_random(1, 4096, 4096, ("cfg1", 0))
    assert regime == "mma" and dg.last_slab() and split == 1   # 32-row tensor-core slabs


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 15, 16, 17, 32, 33, 64])
def test_ragged_shapes_every_regime(M):
    # N not a multiple of the 128-row tile, K not a multiple of the 64-wide block
    _, (regime, _) = _check_random(M, 300, 520, ("ragged", M))
    assert regime == _expect_regime(M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (2, 1, 8), (3, 5, 16), (64, 1, 8), (1, 129, 72),
                                   (16, 127, 4096), (64, 7, 24)])
def test_degenerate_shapes(M, N, K):
    _check_random(M, N, K, ("degenerate", M, N, K))


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 64])
@pytest.mark.parametrize("S", [None, 1, 2, 3, 4, 7, 16])
def test_integer_inputs_bit_exact(M, S):
    # integer-valued bf16 inputs: fp32 accumulation is exact, so the only
    # rounding is the final bf16 one, taken on the exact value on both sides
    K, N = 2048, 384
    x = wl.integer_bf16((M, K), -2, 2, "int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "int", M, "W")
    y, _ = _gpu_linear(x, W, S=S)
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))


@pytest.mark.parametrize("M", [1, 2, 5, 16, 64])
def test_one_hot_rows_reproduce_x(M):
    K, N = 2048, 520
    x = wl.normal_bf16((M, K), 1.0, "onehot", M, "x")
    W, perm = wl.one_hot_rows(N, K, "onehot", M, "W")
    y, _ = _gpu_linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), x[:, perm])


@pytest.mark.parametrize("M", [8, 32, 64])
def test_wide_k_split_factors(M):
    # M in {8,32,64}, K=16384, N=2048, forced split factors 2..16 and the
    # dispatcher's own choice; each run twice must be bit-identical
    K, N = 16384, 2048
    cols = np.random.default_rng(M).choice(N, 256, replace=False)
    x = wl.normal_bf16((M, K), 1.0, "cfg3", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "cfg3", M, "W")
    ref, A = oracle.linear(x, W[cols])
    for S in [None, 2, 4, 8, 12, 16]:
        y1, (_, s_used) = _gpu_linear(x, W, S=S)
        y2, _ = _gpu_linear(x, W, S=S)
        assert torch.equal(y1, y2), "split %s not deterministic" % S
        if S is not None:
            assert s_used == S
        assert_within_tol(to_f64(y1)[:, cols], ref, A, "M=%d S=%s" % (M, S))


@pytest.mark.parametrize("N", [2048, 7168, 16384])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_batch_sweep_k7168(M, N):
    # K=7168 decode projections at every batch size; the oracle checks a
    # sample of 384 output columns
    cols = np.random.default_rng(N + M).choice(N, 384, replace=False)
    _, (regime, _) = _check_random(M, N, 7168, ("cfg2", M, N), cols=cols)
    assert regime == _expect_path(M)
    assert dg.last_slab() == (N in (2048, 7168) and M <= 16)


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_residual_epilogue(M):
    K, N = 1536, 640
    x = wl.normal_bf16((M, K), 1.0, "res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "res", M, "r")
    y, _ = _gpu_linear(x, W, res_bits=r)
    f, A = oracle.linear(x, W)
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), ref, Aref, "residual M=%d" % M)


@pytest.mark.parametrize("M,forces", [(2, ["smallm", "mma"]), (16, ["mma", "tc"]),
                                      (40, ["mma", "tc"])])
def test_forced_regimes_agree(M, forces):
    # integer inputs: every regime must give the same bits
    N, K = 512, 1024
    x = wl.integer_bf16((M, K), -2, 2, "force", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "force", M, "W")
    outs = {}
    for f in forces:
        os.environ["DEC_FORCE"] = f
        try:
            y, (regime, _) = _gpu_linear(x, W)
        finally:
            del os.environ["DEC_FORCE"]
        assert regime == f
        outs[f] = wl.torch_to_bits(y)
    assert np.array_equal(outs[forces[0]], outs[forces[1]])


# ---------------------------------------------------------------- tcgen05 grid
def _tc_aligned_split(N, K, sms):
    # the dispatcher's tile-aligned split for the tcgen05 kernel, or 0 for a
    # split over every SM
    KB, tiles = (K + 127) // 128, (N + 127) // 128
    for sa in range(min(KB, 16), 0, -1):
        if tiles * sa <= sms and KB % sa == 0:
            return sa if tiles * sa * 4 >= 3 * sms else 0
    return 0


@pytest.mark.parametrize("M,N,K", [(64, 2048, 7168), (32, 2048, 16384), (64, 16384, 7168),
                                   (17, 4096, 4096), (64, 7168, 7168)])
def test_tc_tile_aligned_split(M, N, K):
    # 17..64 tokens on the tcgen05 kernel at full size: a tile-aligned split
    # (tiles * sa CTAs, sa dividing the k chunks; sa = 1 has no fixup at all)
    # where it keeps three quarters of the SMs busy, else stream-K over every
    # SM; sampled output features of every tile against the oracle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cols = np.arange(0, N, 61)
    y, (regime, split) = _check_random(M, N, K, ("tcgrid", M, N, K), cols=cols)
    assert regime == "tc"
    sa = _tc_aligned_split(N, K, sms)
    tiles = (N + 127) // 128
    if sa:
        assert split == sa and dg.last_grid() == tiles * sa
    else:
        assert dg.last_grid() == min(sms, tiles * ((K + 127) // 128))


# ---------------------------------------------------------------- cluster split
# Narrow projections with few 128-row tiles (M <= 16) split each tile's k
# chunks over the CTAs of one thread-block cluster and sum the partial tiles
# through distributed shared memory.


@pytest.fixture
def split_k_only(monkeypatch):
    """1-2 tokens on the split-K kernels (the slab kernel would take some of
    these shapes)."""
    monkeypatch.setenv("DEC_FORCE", "splitk")


@pytest.mark.parametrize("M,N,K", [(1, 4000, 1000), (3, 4000, 1288), (8, 2048, 1160),
                                   (15, 1900, 904), (2, 4096, 4096)])
def test_cluster_split_shapes(split_k_only, M, N, K):
    # ragged last tile and last k chunk; uneven k shares between the ranks
    y, (regime, cl) = _check_random(M, N, K, ("cluster", M, N, K))
    assert dg.last_cluster() and cl >= 2 and regime == _expect_regime(M)
    y2, _ = _gpu_linear(wl.normal_bf16((M, K), 1.0, "cluster", M, N, K, "x"),
                        wl.normal_bf16((N, K), 0.02, "cluster", M, N, K, "W"))
    assert torch.equal(y, y2), "cluster split not deterministic"


@pytest.mark.parametrize("M", [1, 4, 15])
def test_cluster_split_integer_inputs_match_stream_k(split_k_only, M):
    # exact fp32 sums: the cluster split, the stream-K split and the oracle
    # give the same bits
    K, N = 2048, 4096
    x = wl.integer_bf16((M, K), -2, 2, "cl-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "cl-int", M, "W")
    y, _ = _gpu_linear(x, W)
    assert dg.last_cluster()
    ys, (_, s_used) = _gpu_linear(x, W, S=4)
    assert not dg.last_cluster() and s_used == 4
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M", [1, 4])
def test_cluster_split_residual(split_k_only, M):
    K, N = 1024, 4096
    x = wl.normal_bf16((M, K), 1.0, "cl-res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "cl-res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "cl-res", M, "r")
    y, _ = _gpu_linear(x, W, res_bits=r)
    assert dg.last_cluster()
    f, A = oracle.linear(x, W)
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), ref, Aref, "cluster residual M=%d" % M)


# 17-64 tokens (tcgen05) take the same cluster split when N has few tiles:
# each rank accumulates its k share in tensor memory, drains it to shared
# memory, and the ranks sum the partials through distributed shared memory.
@pytest.mark.parametrize("M,N,K", [(33, 1900, 904), (17, 2000, 1288), (64, 1920, 1024),
                                   (48, 2304, 4096), (64, 2048, 7168), (40, 2048, 16384),
                                   (24, 1900, 6200)])
def test_tc_cluster_split_shapes(M, N, K):
    # ragged last tile and last k chunk, uneven k shares, token counts not a
    # multiple of 16; 128-k stages (up to 512 k per rank) and 64-k stages
    y, (regime, cl) = _check_random(M, N, K, ("tccluster", M, N, K))
    assert regime == "tc" and dg.last_cluster() and cl >= 2
    y2, _ = _gpu_linear(wl.normal_bf16((M, K), 1.0, "tccluster", M, N, K, "x"),
                        wl.normal_bf16((N, K), 0.02, "tccluster", M, N, K, "W"))
    assert torch.equal(y, y2), "tcgen05 cluster split not deterministic"


@pytest.mark.parametrize("M,K", [(17, 2048), (32, 2048), (64, 2048), (64, 8192)])
def test_tc_cluster_integer_inputs_match_stream_k(M, K):
    # exact fp32 sums: the cluster split, the stream-K tcgen05 split and the
    # oracle give the same bits
    N = 2048
    x = wl.integer_bf16((M, K), -2, 2, "tccl-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "tccl-int", M, "W")
    y, (regime, _) = _gpu_linear(x, W)
    assert regime == "tc" and dg.last_cluster()
    ys, (_, s_used) = _gpu_linear(x, W, S=4)
    assert not dg.last_cluster() and s_used == 4
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M,K", [(17, 1024), (64, 1024), (32, 4096)])
def test_tc_cluster_residual(M, K):
    N = 2048
    x = wl.normal_bf16((M, K), 1.0, "tccl-res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "tccl-res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "tccl-res", M, "r")
    y, (regime, _) = _gpu_linear(x, W, res_bits=r)
    assert regime == "tc" and dg.last_cluster()
    f, A = oracle.linear(x, W)
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), ref, Aref, "tcgen05 cluster residual M=%d" % M)


@pytest.mark.parametrize("M,N,K,ldx", [(1, 7168, 7168, 8192), (4, 4096, 2048, 2056),
                                       (16, 1024, 2048, 4096), (64, 640, 1536, 1544),
                                       (2, 4096, 4096, 8192), (64, 2048, 1024, 1032)])
def test_row_strided_input_reads_a_column_slice(M, N, K, ldx):
    # x is the first K columns of a [M, ldx] activation (the q part of a fused
    # q|kv output, say): read in place, with and without a residual
    wide = wl.normal_bf16((M, ldx), 1.0, "ldx", M, N, K, "xw")
    W = wl.normal_bf16((N, K), 0.02, "ldx", M, N, K, "W")
    r = wl.normal_bf16((M, N), 1.0, "ldx", M, N, K, "r")
    xt = wl.bits_to_torch(wide)[:, :K]
    assert xt.stride(0) == ldx
    f, A = oracle.linear(wide[:, :K], W)
    y = dg.dec_linear(xt, wl.bits_to_torch(W))
    assert dg.sync_check() == dg.DEC_OK
    assert_within_tol(to_f64(y), f, A, "ldx=%d" % ldx)
    y2 = dg.dec_linear(xt, wl.bits_to_torch(W), residual=wl.bits_to_torch(r))
    assert dg.sync_check() == dg.DEC_OK
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y2), ref, Aref, "ldx=%d residual" % ldx)
    # the same bits as on a contiguous copy
    y3 = dg.dec_linear(xt.contiguous(), wl.bits_to_torch(W))
    assert torch.equal(y, y3)


def test_output_guard_bands_untouched():
    # the kernel writes exactly [M,N]: sentinel bytes around y stay intact
    M, N, K = 3, 200, 256
    x = wl.bits_to_torch(wl.normal_bf16((M, K), 1.0, "guard", "x"))
    W = wl.bits_to_torch(wl.normal_bf16((N, K), 0.02, "guard", "W"))
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    dg.dec_linear(x, W, y)
    assert dg.sync_check() == dg.DEC_OK
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345)


@pytest.mark.parametrize("M", [4, 16])
@pytest.mark.parametrize("residual", [True, False])
def test_wide_tiles_full_size_7168(split_k_only, M, residual):
    # N = K = 7168 at 4 and 16 tokens on split-K takes the 256-row-tile
    # instance (the dispatcher gives this shape 48-row slabs): every element
    # against the oracle
    N = K = 7168
    x = wl.normal_bf16((M, K), 1.0, "wide", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "wide", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "wide", M, "r") if residual else None
    y, (regime, _) = _gpu_linear(x, W, res_bits=r)
    assert regime == "mma" and dg.last_wide() and not dg.last_cluster()
    f, A = oracle.linear(x, W)
    if residual:
        f, A = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), f, A, "wide tiles M=%d residual=%s" % (M, residual))


# ---------------------------------------------------------------- whole-row slabs
# 1-2 tokens on the CUDA cores: each CTA owns 8, 16 or 32 whole weight rows
# over all of K (no split over K, no partial sums leave the CTA) when such
# slabs fill the SMs. The dispatcher takes them where only 8-row slabs fill
# the SMs (else the tensor-core slabs below); DEC_FORCE=smallm takes them
# wherever they fit.


@pytest.fixture
def core_slabs(monkeypatch):
    monkeypatch.setenv("DEC_FORCE", "smallm")


@pytest.mark.parametrize("M,N,K", [(1, 2048, 7168), (2, 2048, 7168), (1, 4096, 4096),
                                   (2, 1024, 1024), (2, 1100, 4096), (1, 4000, 16384),
                                   (1, 3700, 2048), (2, 2048, 16384)])
def test_slab_shapes(core_slabs, M, N, K):
    # rows per CTA 8 / 16 / 32, a ragged last slab, K up to 16384
    y, (regime, split) = _check_random(M, N, K, ("slab", M, N, K))
    assert regime == "smallm" and dg.last_slab() and split == 1 and not dg.last_cluster()
    y2, _ = _gpu_linear(wl.normal_bf16((M, K), 1.0, "slab", M, N, K, "x"),
                        wl.normal_bf16((N, K), 0.02, "slab", M, N, K, "W"))
    assert torch.equal(y, y2), "slab kernel not deterministic"


@pytest.mark.parametrize("M", [1, 2])
def test_slab_integer_inputs_match_oracle_and_split_k(M, monkeypatch):
    monkeypatch.setenv("DEC_FORCE", "smallm")
    K, N = 4096, 2048
    x = wl.integer_bf16((M, K), -2, 2, "slab-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "slab-int", M, "W")
    y, _ = _gpu_linear(x, W)
    assert dg.last_slab()
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    monkeypatch.setenv("DEC_FORCE", "splitk")
    ys, _ = _gpu_linear(x, W)
    assert not dg.last_slab()
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M", [1, 2])
def test_slab_residual_and_row_strided_input(core_slabs, M):
    K, N, ldx = 4096, 2048, 4160
    wide = wl.normal_bf16((M, ldx), 1.0, "slab-res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "slab-res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "slab-res", M, "r")
    xt = wl.bits_to_torch(wide)[:, :K]
    y = dg.dec_linear(xt, wl.bits_to_torch(W), residual=wl.bits_to_torch(r))
    assert dg.last_slab()
    assert dg.sync_check() == dg.DEC_OK
    f, A = oracle.linear(wide[:, :K], W)
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), ref, Aref, "slab residual M=%d" % M)


@pytest.mark.parametrize("M,N", [(1, 1024), (2, 1100)])
def test_dispatcher_takes_cuda_core_slabs_of_8_rows(M, N):
    # 16-row slabs would leave half the SMs idle: 8-row ones on the CUDA cores
    y, (regime, split) = _check_random(M, N, 4096, ("slab8", M, N))
    assert regime == "smallm" and dg.last_slab() and split == 1


def test_slab_declines_shapes_it_does_not_fill(core_slabs):
    # too few rows for three quarters of the SMs, or K not a multiple of 64
    for M, N, K in [(1, 384, 2048), (1, 4096, 1000), (2, 6000, 2048)]:
        _check_random(M, N, K, ("slab-no", M, N, K))
        assert not dg.last_slab(), (M, N, K)


# ---------------------------------------------------------------- tensor-core slabs
# 1-16 tokens: the same whole-row slabs (16 or 32 rows per CTA) with the dot
# products on the tensor cores (mma.sync), 4, 8 or 16 token rows per stage.


@pytest.mark.parametrize("M,N,K", [(1, 2048, 7168), (2, 2048, 7168), (3, 2048, 7168),
                                   (4, 4096, 4096), (1, 4096, 4096), (3, 3700, 2048),
                                   (4, 2000, 1024), (2, 2048, 16384), (4, 4096, 1088),
                                   (5, 2048, 7168), (8, 2048, 7168), (16, 2048, 7168),
                                   (12, 4096, 4096), (9, 2048, 16384), (16, 3700, 2048),
                                   (7, 4096, 1088), (13, 2000, 1024)])
def test_mma_slab_shapes(M, N, K):
    # 16 / 32 rows per CTA, 4 / 8 / 16 token rows, ragged last slab, K from
    # 1024 to 16384 (1088: a last stage with one k block of 64)
    y, (regime, split) = _check_random(M, N, K, ("mslab", M, N, K))
    assert regime == "mma" and dg.last_slab() and split == 1 and not dg.last_cluster()
    y2, _ = _gpu_linear(wl.normal_bf16((M, K), 1.0, "mslab", M, N, K, "x"),
                        wl.normal_bf16((N, K), 0.02, "mslab", M, N, K, "W"))
    assert torch.equal(y, y2), "mma slab kernel not deterministic"


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 11, 16])
def test_mma_slab_integer_inputs_match_oracle_and_split_k(M, monkeypatch):
    K, N = 4096, 2048
    x = wl.integer_bf16((M, K), -2, 2, "mslab-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "mslab-int", M, "W")
    y, _ = _gpu_linear(x, W)
    assert dg.last_slab()
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    monkeypatch.setenv("DEC_FORCE", "splitk")
    ys, _ = _gpu_linear(x, W)
    assert not dg.last_slab()
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M", [1, 4, 6, 16])
def test_mma_slab_residual_and_row_strided_input(M):
    K, N, ldx = 4096, 2048, 4160
    wide = wl.normal_bf16((M, ldx), 1.0, "mslab-res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "mslab-res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "mslab-res", M, "r")
    xt = wl.bits_to_torch(wide)[:, :K]
    y = dg.dec_linear(xt, wl.bits_to_torch(W), residual=wl.bits_to_torch(r))
    assert dg.last_slab() and dg.last_choice()[0] == "mma"
    assert dg.sync_check() == dg.DEC_OK
    f, A = oracle.linear(wide[:, :K], W)
    ref, Aref = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), ref, Aref, "mma slab residual M=%d" % M)


@pytest.mark.parametrize("M", [1, 2])
def test_mma_slab_for_one_or_two_tokens_matches_the_cuda_core_slab(M, monkeypatch):
    K, N = 7168, 2048
    x = wl.integer_bf16((M, K), -2, 2, "mslab-12", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "mslab-12", M, "W")
    ym, (regime, _) = _gpu_linear(x, W)
    assert regime == "mma" and dg.last_slab()
    monkeypatch.setenv("DEC_FORCE", "smallm")
    y, (regime, _) = _gpu_linear(x, W)
    assert regime == "smallm" and dg.last_slab()
    assert torch.equal(y, ym)


def test_mma_slab_declines_shapes_it_does_not_fill():
    # too few rows for three quarters of the SMs, K not a multiple of 64,
    # too many rows for 64 per CTA, more than 16 tokens
    for M, N, K in [(4, 1024, 4096), (3, 4096, 1000), (8, 9800, 7168), (17, 2048, 4096)]:
        _check_random(M, N, K, ("mslab-no", M, N, K))
        assert not dg.last_slab(), (M, N, K)


@pytest.mark.parametrize("M,N,K", [(1, 7168, 7168), (5, 7168, 7168), (16, 7168, 4096),
                                   (3, 6000, 7168), (12, 5800, 1088), (2, 7168, 16384)])
def test_mma_slabs_of_48_rows(M, N, K):
    # three 16-row groups per CTA (N from 4865 to 7296 rows): warps 0, 3, 6 /
    # 1, 4, 7 / 2, 5 share a group's k blocks; ragged last slab; deep ring
    cols = np.random.default_rng(N + K + M).choice(N, 512, replace=False)
    y, (regime, split) = _check_random(M, N, K, ("mslab48", M, N, K), cols=cols)
    assert regime == "mma" and dg.last_slab() and split == 1 and dg.last_grid() == (N + 47) // 48


@pytest.mark.parametrize("M", [1, 8, 16])
def test_mma_slabs_of_48_rows_integer_inputs_match_oracle_and_split_k(M, monkeypatch):
    K, N = 2048, 7168
    x = wl.integer_bf16((M, K), -2, 2, "mslab48-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "mslab48-int", M, "W")
    y, _ = _gpu_linear(x, W)
    assert dg.last_slab()
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    monkeypatch.setenv("DEC_FORCE", "splitk")
    ys, _ = _gpu_linear(x, W)
    assert not dg.last_slab()
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M,N,K", [(1, 8192, 7168), (4, 8192, 7168), (16, 8192, 7168),
                                   (3, 7400, 7168), (8, 9728, 2048), (12, 9000, 1088),
                                   (2, 8192, 16384)])
def test_mma_slabs_of_64_rows(M, N, K):
    # four 16-row groups per CTA (N from 7297 to 9728 rows, the fused q|kv
    # projection among them): warps w and w + 4 share group w's k blocks;
    # ragged last slab; deep ring
    cols = np.random.default_rng(N + K + M).choice(N, 512, replace=False)
    y, (regime, split) = _check_random(M, N, K, ("mslab64", M, N, K), cols=cols)
    assert regime == "mma" and dg.last_slab() and split == 1 and dg.last_grid() == (N + 63) // 64


@pytest.mark.parametrize("M", [1, 5, 16])
def test_mma_slabs_of_64_rows_integer_inputs_match_oracle_and_split_k(M, monkeypatch):
    K, N = 2048, 8192
    x = wl.integer_bf16((M, K), -2, 2, "mslab64-int", M, "x")
    W = wl.integer_bf16((N, K), -2, 2, "mslab64-int", M, "W")
    y, _ = _gpu_linear(x, W)
    assert dg.last_slab() and dg.last_grid() == N // 64
    ref, _ = oracle.linear(x, W)
    assert np.array_equal(wl.torch_to_bits(y), oracle.f64_to_bf16_bits(ref))
    monkeypatch.setenv("DEC_FORCE", "splitk")
    ys, _ = _gpu_linear(x, W)
    assert not dg.last_slab()
    assert torch.equal(y, ys)


@pytest.mark.parametrize("M", [1, 16])
def test_mma_slabs_of_64_rows_residual(M):
    # every element of a 64-row slab call with the residual epilogue
    N, K = 8192, 2048
    x = wl.normal_bf16((M, K), 1.0, "mslab64-res", M, "x")
    W = wl.normal_bf16((N, K), 0.02, "mslab64-res", M, "W")
    r = wl.normal_bf16((M, N), 1.0, "mslab64-res", M, "r")
    y, (regime, _) = _gpu_linear(x, W, res_bits=r)
    assert regime == "mma" and dg.last_slab() and dg.last_grid() == N // 64
    f, A = oracle.linear(x, W)
    f, A = oracle.residual(r, f, A)
    assert_within_tol(to_f64(y), f, A, "64-row slabs M=%d residual" % M)
