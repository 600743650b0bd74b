"""GPU parity of the MoE decode block against the fp64 oracle.

Router inputs are drawn so that the fp64 router scores of every token have
adjacent gaps of at least 1e-3 among the k+1 largest: the expert choice is
then unique and the GPU's top-k indices must equal the oracle's exactly.
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


def _small_block(M, H, E, I, k, key, std=0.02, shared=True):
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, H), std, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), std, *key, "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), std, *key, "Ws13"),
          wl.normal_bf16((H, I), std, *key, "Ws2")) if shared else None
    return x, Wr, W13, W2, Ws


def _gpu_moe(x, Wr, W13, W2, Ws, k, res=None):
    t = wl.bits_to_torch
    M = x.shape[0]
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    gw = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    out = dg.moe_decode(t(x), t(Wr), t(W13), t(W2), None if Ws is None else t(Ws[0]),
                        None if Ws is None else t(Ws[1]), k, topk_idx=idx, topk_w=gw,
                        residual=None if res is None else t(res))
    assert dg.sync_check() == dg.DEC_OK
    return out, idx.cpu().numpy(), gw.cpu().numpy()


def _check(x, Wr, W13, W2, Ws, k, what, res=None):
    I = W13.shape[1] // 2
    out, idx, gw = _gpu_moe(x, Wr, W13, W2, Ws, k, res=res)
    r = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=Ws)
    assert np.array_equal(idx, r["idx"]), what + ": top-k indices differ"
    np.testing.assert_allclose(gw, r["gates"], rtol=2e-5, atol=1e-7, err_msg=what + ": gates")
    ref, A = r["out"], r["absref"]
    if res is not None:
        ref, A = oracle.residual(res, ref, A)
    assert_within_tol(to_f64(out), ref, A, what)
    return out


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 33, 64])
@pytest.mark.parametrize("shared", [True, False])
def test_small_block_against_oracle(M, shared):
    blk = _small_block(M, 256, 64, 128, 8, ("moe-small", M, shared), shared=shared)
    _check(*blk, 8, "M=%d shared=%s" % (M, shared))


def test_ragged_intermediate_and_hidden():
    # I not a multiple of 64 and H not a multiple of 128: tiles overhang
    blk = _small_block(9, 200, 24, 72, 3, ("moe-ragged",))
    _check(*blk, 3, "ragged")


def test_every_token_same_expert_pool():
    # 64 tokens over 8 experts with k = 8: every expert serves all 64 tokens
    blk = _small_block(64, 128, 8, 64, 8, ("moe-dense",))
    _check(*blk, 8, "all experts, all tokens")


def test_topk_equals_E_with_zero_router_is_dense_mean():
    E, H, I, M = 16, 128, 64, 5
    x, Wr, W13, W2, _ = _small_block(M, H, E, I, 8, ("moe-uniform",), shared=False)
    Wr0 = np.zeros_like(Wr)
    out, idx, gw = _gpu_moe(x, Wr0, W13, W2, None, E)
    assert np.all(idx == np.arange(E))                  # ties: smaller index first
    np.testing.assert_allclose(gw, 1.0 / E, rtol=1e-6)
    r = oracle.moe(x, Wr0, lambda e: (W13[e], W2[e]), E, I, shared=None)
    assert_within_tol(to_f64(out), r["out"], r["absref"], "uniform")


def test_single_expert_block():
    blk = _small_block(7, 192, 1, 64, 1, ("moe-one",))
    _check(*blk, 1, "E=1")


def test_zero_routed_down_projection_leaves_shared_expert():
    x, Wr, W13, W2, Ws = _small_block(6, 256, 32, 128, 4, ("moe-zero",))
    _check(x, Wr, W13, np.zeros_like(W2), Ws, 4, "zero W2")


def test_residual_combine():
    x, Wr, W13, W2, Ws = _small_block(12, 256, 48, 128, 6, ("moe-res",))
    res = wl.normal_bf16((12, 256), 1.0, "moe-res", "r")
    _check(x, Wr, W13, W2, Ws, 6, "residual", res=res)


def test_routing_limits_topk32_of_1024_experts_64_tokens():
    # the largest routing problem the block accepts: 2048 (token, slot) pairs
    # over 1024 experts, 32 chosen per token
    M, H, E, I, k = 64, 128, 1024, 64, 32
    blk = _small_block(M, H, E, I, k, ("moe-limits",), shared=True)
    _check(*blk, k, "E=1024 k=32 M=64")


@pytest.mark.parametrize("M", [16, 40])
@pytest.mark.parametrize("H", [320, 520, 696, 840])
def test_router_clusters_of_any_size_cover_every_expert_row(H, M):
    # The router runs one thread-block cluster of min(H/128 rounded up, 8)
    # CTAs per 128 experts: 3, 5, 6 and 7 CTAs here, which do not divide the
    # 128 rows of a tile. Experts 125-127 (the last rows of the first tile)
    # are made the likeliest choices, so most tokens' top-k depends on them.
    # 16 tokens: mma.sync dot products; 40: tcgen05 (tensor-memory partials
    # pushed to the rows' owners).
    E, I, k = 160, 128, 4
    key = ("router-rows", H) if M == 16 else ("router-rows", H, M)
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    Wr[125:128] = wl.normal_bf16((3, H), 6.0 / math.sqrt(H), *key, "Wr-hot")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)])
    idx = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=None)["idx"]
    assert np.isin(idx, [125, 126, 127]).any(axis=1).mean() >= 0.5, idx
    _check(x, Wr, W13, W2, None, k, "router rows H=%d" % H)


def test_skewed_routing_shares_experts_across_groups():
    # power-law expert popularity at 64 tokens (32-row expert groups): experts
    # serving 17-32 tokens (one wide group), one serving more than 32 (two
    # groups), experts of at most 16 (the narrow token box), and many serving
    # none
    M, H, E, I, k = 64, 256, 64, 128, 8
    key = ("moe-skew",)
    Wr = wl.skewed_router_bf16(E, H, 1.0, *key, "Wr")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"), wl.normal_bf16((H, I), 0.02, *key, "Ws2"))
    idx = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=None)["idx"]
    counts = np.bincount(idx.ravel(), minlength=E)
    assert counts.max() > 32 and ((counts > 16) & (counts <= 32)).any(), counts
    assert ((counts > 0) & (counts <= 16)).any() and (counts == 0).sum() > 0, counts
    _check(x, Wr, W13, W2, Ws, k, "skewed routing")


def test_repeat_calls_bit_identical():
    x, Wr, W13, W2, Ws = _small_block(33, 256, 64, 128, 8, ("moe-det",))
    a, _, _ = _gpu_moe(x, Wr, W13, W2, Ws, 8)
    b, _, _ = _gpu_moe(x, Wr, W13, W2, Ws, 8)
    assert torch.equal(a, b)


# ---------------------------------------------------------------- full size
H, E, K8, I = wl.HIDDEN, wl.EXPERTS, wl.TOPK, wl.INTER


@pytest.fixture(scope="module")
def full_bank():
    """Routed experts (33.8 GB) and shared expert on the device, ~N(0, 0.02)."""
    W13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device="cuda")
    W2 = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
    for e in range(E):
        wl.normal_bf16_cuda((2 * I, H), wl.WEIGHT_STD, "bank", 0, "W13", e, out=W13[e])
        wl.normal_bf16_cuda((H, I), wl.WEIGHT_STD, "bank", 0, "W2", e, out=W2[e])
    Ws13 = wl.normal_bf16_cuda((2 * I, H), wl.WEIGHT_STD, "bank", 0, "Ws13")
    Ws2 = wl.normal_bf16_cuda((H, I), wl.WEIGHT_STD, "bank", 0, "Ws2")
    Wr = wl.normal_bf16((E, H), wl.ROUTER_STD, "bank", 0, "Wr")
    yield W13, W2, Ws13, Ws2, Wr
    del W13, W2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_full_size_block(full_bank, M):
    # hidden 7168, 384 experts, top-8, intermediate 2048, shared expert;
    # indices of every token exact, outputs of sampled tokens within tolerance
    W13, W2, Ws13, Ws2, Wr_bits = full_bank
    x_bits, _ = gap_rows(Wr_bits, M, H, K8, "full", M)
    t = wl.bits_to_torch
    x, Wr = t(x_bits), t(Wr_bits)
    idx = torch.empty((M, K8), dtype=torch.int32, device="cuda")
    gw = torch.empty((M, K8), dtype=torch.float32, device="cuda")
    out = dg.moe_decode(x, Wr, W13, W2, Ws13, Ws2, K8, topk_idx=idx, topk_w=gw)
    assert dg.sync_check() == dg.DEC_OK
    logits, _ = oracle.linear(x_bits, Wr_bits)
    ridx, rg = oracle.topk(logits, K8)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(gw.cpu().numpy(), rg, rtol=2e-5, atol=1e-7)
    tokens = sorted(set([0, M - 1, M // 2]))
    fetch = lambda e: (wl.torch_to_bits(W13[e]), wl.torch_to_bits(W2[e]))
    r = oracle.moe(x_bits, Wr_bits, fetch, K8, I,
                   shared=(wl.torch_to_bits(Ws13), wl.torch_to_bits(Ws2)), tokens=tokens)
    got = to_f64(out)
    assert_within_tol(got[tokens], r["out"][tokens], r["absref"][tokens], "full M=%d" % M)


# ---------------------------------------------------------------- decode layer
@pytest.mark.parametrize("M", [1, 5, 33])
def test_decode_layer_composition(M):
    """The layer as the benchmark composes it: one fused q|kv projection, the o
    projection reading q in place with the residual fused, then the MoE block
    with its residual; every stage against the oracle on the GPU's own input
    to that stage."""
    H, KV, E, I, k = 256, 64, 32, 128, 4
    key = ("layer", M)
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    x, _ = gap_rows(Wr, M, H, k, *key, "x")
    Wq = wl.normal_bf16((H, H), 0.02, *key, "Wq")
    Wkv = wl.normal_bf16((KV, H), 0.02, *key, "Wkv")
    Wo = wl.normal_bf16((H, H), 0.02, *key, "Wo")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"), wl.normal_bf16((H, I), 0.02, *key, "Ws2"))
    t = wl.bits_to_torch
    xt = t(x)
    qkv = dg.dec_linear(xt, t(np.concatenate([Wq, Wkv])))
    assert dg.sync_check() == dg.DEC_OK
    ref, A = oracle.linear(x, np.concatenate([Wq, Wkv]))
    assert_within_tol(to_f64(qkv), ref, A, "q|kv")
    q_bits = wl.torch_to_bits(qkv)[:, :H]
    # o projection on the q columns of the fused output, residual x
    r = dg.dec_linear(qkv[:, :H], t(Wo), residual=xt)
    assert dg.sync_check() == dg.DEC_OK
    o, oA = oracle.linear(q_bits, Wo)
    rref, rA = oracle.residual(x, o, oA)
    assert_within_tol(to_f64(r), rref, rA, "o + residual")
    # MoE block on r with its residual; with Wo = 0 the block's input is x
    # exactly, whose router scores satisfy the gap rule, so the chosen experts
    # must match the oracle's bit for bit
    r0 = dg.dec_linear(qkv[:, :H], t(np.zeros_like(Wo)), residual=xt)
    assert torch.equal(r0, xt)
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    out = dg.moe_decode(r0, t(Wr), t(W13), t(W2), t(Ws[0]), t(Ws[1]), k, topk_idx=idx,
                        residual=r0)
    assert dg.sync_check() == dg.DEC_OK
    mo = oracle.moe(x, Wr, lambda e: (W13[e], W2[e]), k, I, shared=Ws)
    assert np.array_equal(idx.cpu().numpy(), mo["idx"])
    oref, oA2 = oracle.residual(x, mo["out"], mo["absref"])
    assert_within_tol(to_f64(out), oref, oA2, "moe + residual")


def test_decode_layer_replays_from_a_cuda_graph():
    """A decode layer captured into a CUDA graph (after one eager warm-up call,
    so that the library's workspace exists) replays to the same bits: the
    shared expert's side-stream fork and join, programmatic dependent launches
    and cluster launches all capture."""
    M, H, KV, E, I, k = 5, 256, 64, 32, 128, 4
    key = ("graph",)
    t = wl.bits_to_torch
    Wr = t(wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr"))
    x = t(wl.normal_bf16((M, H), 1.0, *key, "x"))
    Wqkv = t(wl.normal_bf16((H + KV, H), 0.02, *key, "Wqkv"))
    Wo = t(wl.normal_bf16((H, H), 0.02, *key, "Wo"))
    W13 = t(np.stack([wl.normal_bf16((2 * I, H), 0.02, *key, "W13", e) for e in range(E)]))
    W2 = t(np.stack([wl.normal_bf16((H, I), 0.02, *key, "W2", e) for e in range(E)]))
    Ws13 = t(wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13"))
    Ws2 = t(wl.normal_bf16((H, I), 0.02, *key, "Ws2"))
    qkv = torch.empty((M, H + KV), dtype=torch.bfloat16, device="cuda")
    r = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def layer():
        dg.dec_linear(x, Wqkv, qkv, stream=s)
        dg.dec_linear(qkv[:, :H], Wo, r, stream=s, residual=x)
        dg.moe_decode(r, Wr, W13, W2, Ws13, Ws2, k, out=out, stream=s, residual=r)

    layer()
    torch.cuda.synchronize()
    assert dg.sync_check() == dg.DEC_OK
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert dg.sync_check() == dg.DEC_OK


def test_workspace_relayout_within_its_capacity():
    # A larger block that still fits the workspace allocated for a smaller one
    # (it is allocated with slack) changes the workspace's layout without a
    # new allocation: the arrival counters must still start at zero. Three
    # blocks of growing E, each checked against the oracle. The workspace is
    # freed first, so that the first block sizes it.
    torch.cuda.synchronize()
    dg.shutdown()
    for E in (40, 44, 48):
        blk = _small_block(6, 192, E, 96, 4, ("moe-relayout", E))
        _check(*blk, 4, "E=%d after a smaller block" % E)


@pytest.mark.parametrize("M,H,I", [(17, 7168, 2048), (33, 7168, 2048), (64, 7168, 2048),
                                   (20, 520, 328), (48, 1032, 584)])
def test_shared_expert_on_tensor_cores(M, H, I):
    # From 17 tokens the shared expert's gate/up (SwiGLU, gate and up
    # accumulators in tensor memory) and down projections run on tcgen05. With
    # the routed down projections zero the block is the shared expert alone:
    # every element against the oracle, at the full hidden and intermediate
    # sizes and at ragged ones (tiles and k chunks overhanging). The ragged
    # intermediate widths are a few hundred: below about 200 the bf16 rounding
    # of the hidden vector alone (the oracle with that rounding applied)
    # exceeds the 1e-3 * A term on some elements.
    E, k = 8, 2
    key = ("shared-tc", M, H, I)
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), *key, "Wr")
    x = wl.normal_bf16((M, H), 1.0, *key, "x")
    t = wl.bits_to_torch
    W13 = torch.zeros((E, 2 * I, H), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((E, H, I), dtype=torch.bfloat16, device="cuda")
    Ws13 = wl.normal_bf16((2 * I, H), 0.02, *key, "Ws13")
    Ws2 = wl.normal_bf16((H, I), 0.02, *key, "Ws2")
    out = dg.moe_decode(t(x), t(Wr), W13, W2, t(Ws13), t(Ws2), k)
    assert dg.sync_check() == dg.DEC_OK
    s, sA = oracle.expert_mlp(x, Ws13, Ws2, I)
    assert_within_tol(to_f64(out), s, sA, "shared expert M=%d H=%d I=%d" % (M, H, I))
