"""Full-size parity of the decode layer stack that the benchmark times.

A layer is built and run exactly as the benchmark does, through
``moe_decode_gemm_gb300.stack.decode_layer``: the fused [8192, 7168] q|kv
projection, the o projection reading q in place with the residual fused, the
L2 prefetch of the next layer's weights on a side stream, and the MoE block
(hidden 7168, 384 experts, top-8, intermediate 2048, shared expert on the
library's side stream) with its residual. Each stage is checked against the
fp64 oracle fed the GPU's own bf16 input to that stage, so that errors do not
compound: every element of q|kv and of r, the chosen experts of every token,
and the block's output for at least 8 tokens.

Where the oracle's scores of two experts are closer than the gap the
workload guarantees (1e-3), fp32 may legitimately choose the other one: there
the GPU's choice is checked to be a valid top-k, and the output is checked for
the choice it made. After four layers the drift against the oracle's own
four-layer chain is reported, not gated.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import GAP, assert_within_tol, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_decode_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"


import moe_decode_gemm_gb300 as dg  # noqa: E402
from moe_decode_gemm_gb300.stack import decode_layer  # noqa: E402

H, KV, E, K8, I = wl.HIDDEN, wl.KV_WIDTH, wl.EXPERTS, wl.TOPK, wl.INTER
NL = 4


class _Host:
    """Host copies (bf16 bits) of a layer's dense weights, and its experts on demand."""

    def __init__(self, L):
        self.L = L
        self.Wqkv = wl.torch_to_bits(L.Wqkv)
        self.Wq, self.Wo, self.Wr = self.Wqkv[:H], wl.torch_to_bits(L.Wo), wl.torch_to_bits(L.Wr)
        self.shared = (wl.torch_to_bits(L.Ws13), wl.torch_to_bits(L.Ws2))
        self._experts = {}

    def expert(self, e):
        if e not in self._experts:
            self._experts[e] = (wl.torch_to_bits(self.L.W13[e]), wl.torch_to_bits(self.L.W2[e]))
        return self._experts[e]


@pytest.fixture(scope="module")
def stack():
    layers = [wl.LayerWeights(l, "cuda") for l in range(NL)]
    torch.cuda.synchronize()
    hosts = [_Host(L) for L in layers]
    yield layers, hosts
    del layers, hosts
    torch.cuda.empty_cache()


def _oracle_r(h, x_bits):
    """The layer's MoE input r = bf16(x + bf16(x·Wqᵀ)·Woᵀ), in fp64."""
    q, _ = oracle.linear(x_bits, h.Wq)
    o, _ = oracle.linear(oracle.f64_to_bf16_bits(q), h.Wo)
    return oracle.f64_to_bf16_bits(oracle.bf16_to_f64(x_bits) + o)


def _layer_gap_rows(h, M, *key):
    """Token rows x ~N(0,1) whose layer-input r has router scores with gaps of
    at least 1e-3 among the 9 largest (rows that fail are redrawn)."""
    attempts = [0] * M
    for _ in range(64):
        x = wl.token_rows(M, H, *key, attempts=attempts)
        logits, _ = oracle.linear(_oracle_r(h, x), h.Wr)
        bad = np.where(~np.all(oracle.sorted_gaps(logits, K8 + 1) >= GAP, axis=1))[0]
        if bad.size == 0:
            return x
        for m in bad:
            attempts[m] += 1
    raise RuntimeError("could not draw gap-separated rows")


def _check_choice(logits, gidx, what):
    """Chosen experts: exactly the oracle's where the gap rule holds, else a
    valid top-k (distinct, within fp32 reach of the k-th score, ordered)."""
    ridx, _ = oracle.topk(logits, K8)
    sure = np.all(oracle.sorted_gaps(logits, K8 + 1) >= GAP, axis=1)
    assert np.array_equal(gidx[sure], ridx[sure]), what + ": chosen experts differ"
    for m in np.where(~sure)[0]:
        row = logits[m]
        kth = np.sort(row)[::-1][K8 - 1]
        sel = row[gidx[m]]
        assert len(set(gidx[m].tolist())) == K8, what
        assert np.all(sel >= kth - 1e-4), what + ": token %d chose a score below the k-th" % m
        assert np.all(np.diff(sel) <= 1e-4), what + ": token %d out of order" % m
    return int(sure.sum())


def _check_layer(h, x_bits, qkv, r, out, idx, tokens, what):
    """Every stage of one layer against the oracle on the GPU's own inputs."""
    ref, A = oracle.linear(x_bits, h.Wqkv)
    assert_within_tol(to_f64(qkv), ref, A, what + " q|kv")
    q_bits = wl.torch_to_bits(qkv)[:, :H]
    o, oA = oracle.linear(q_bits, h.Wo)
    rref, rA = oracle.residual(x_bits, o, oA)
    assert_within_tol(to_f64(r), rref, rA, what + " r = x + o")
    r_bits = wl.torch_to_bits(r)
    logits, _ = oracle.linear(r_bits, h.Wr)
    gidx = idx.cpu().numpy()
    nsure = _check_choice(logits, gidx, what)
    mo = oracle.moe(r_bits, h.Wr, h.expert, K8, I, shared=h.shared, tokens=tokens, route=gidx)
    oref, oA2 = oracle.residual(r_bits, mo["out"], mo["absref"])
    got = to_f64(out)
    assert_within_tol(got[tokens], oref[tokens], oA2[tokens], what + " x' = r + moe(r)")
    return nsure


def _sample_tokens(M):
    if M <= 8:
        return list(range(M))
    return sorted(set([0, M - 1] + np.random.default_rng(M).choice(M, 10, replace=False).tolist()))


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_full_size_layer_every_stage(stack, M):
    layers, hosts = stack
    L, h = layers[0], hosts[0]
    x_bits = _layer_gap_rows(h, M, "stack-parity", M)
    x = wl.bits_to_torch(x_bits)
    main = torch.cuda.Stream(priority=-1)
    pref = torch.cuda.Stream()
    ev = torch.cuda.Event()
    pf_bytes = min(H * H * 2, torch.cuda.get_device_properties(0).L2_cache_size // 2)
    qkv = torch.empty((M, H + KV), dtype=torch.bfloat16, device="cuda")
    r = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((M, K8), -1, dtype=torch.int32, device="cuda")
    decode_layer(L, x, qkv, r, out, K8, idx=idx, stream=main,
                 prefetch=(pref, ev, layers[1].Wq.data_ptr(), pf_bytes))
    main.wait_stream(pref)
    torch.cuda.synchronize()
    assert dg.sync_check(main) == dg.DEC_OK
    tokens = _sample_tokens(M)
    nsure = _check_layer(h, x_bits, qkv, r, out, idx, tokens, "layer 0 M=%d" % M)
    assert nsure == M      # the input rows were drawn so that every token's choice is unique
    assert len(tokens) >= min(M, 8)


@pytest.mark.parametrize("M", [4, 64])
def test_four_layer_stack_every_layer_and_drift(stack, M):
    """The benchmark's four layers back to back (prefetch of each next layer's
    q weights on a side stream), then every layer checked on its own GPU
    input; and the same stack with the benchmark's shared q|kv and r buffers
    gives the same bits. The drift of the last layer's output against the
    oracle's own four-layer chain is reported."""
    layers, hosts = stack
    x_bits = wl.token_rows(M, H, "stack-x", M)
    main = torch.cuda.Stream(priority=-1)
    pref = torch.cuda.Stream()
    evs = [torch.cuda.Event() for _ in range(NL)]
    pf_bytes = min(H * H * 2, torch.cuda.get_device_properties(0).L2_cache_size // 2)
    xs = [wl.bits_to_torch(x_bits)] + [torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
                                      for _ in range(NL)]
    qkvs = [torch.empty((M, H + KV), dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    rs = [torch.empty((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(NL)]
    idxs = [torch.full((M, K8), -1, dtype=torch.int32, device="cuda") for _ in range(NL)]

    def run(shared_bufs):
        for l in range(NL):
            pf = (pref, evs[l], layers[(l + 1) % NL].Wq.data_ptr(), pf_bytes)
            decode_layer(layers[l], xs[l], qkvs[0] if shared_bufs else qkvs[l],
                         rs[0] if shared_bufs else rs[l], xs[l + 1], K8, idx=idxs[l],
                         stream=main, prefetch=pf)
        main.wait_stream(pref)
        torch.cuda.synchronize()
        assert dg.sync_check(main) == dg.DEC_OK

    run(shared_bufs=True)
    bench_like = xs[NL].clone()
    run(shared_bufs=False)
    assert torch.equal(xs[NL], bench_like)
    tokens = _sample_tokens(M)[:8]
    for l in range(NL):
        _check_layer(hosts[l], wl.torch_to_bits(xs[l]), qkvs[l], rs[l], xs[l + 1], idxs[l],
                     tokens, "layer %d M=%d" % (l, M))
    # drift: the oracle's own chain (each layer fed the oracle's rounded output)
    xo = x_bits[tokens]
    for l in range(NL):
        h = hosts[l]
        lay = oracle.decoder_layer(xo, h.Wq, h.Wqkv[H:], h.Wo, h.Wr, h.expert, K8, I, h.shared)
        xo = lay["out"]
    gpu = to_f64(xs[NL])[tokens]
    ref = oracle.bf16_to_f64(xo)
    drift = np.abs(gpu - ref)
    scale = np.abs(ref) + lay["out_abs"]
    rel = float(np.max(drift / scale))
    print("4-layer drift at M=%d over tokens %s: max |gpu - oracle chain| = %.4g, "
          "max relative to |ref| + A = %.4g" % (M, tokens, float(drift.max()), rel))
    assert np.all(np.isfinite(gpu)) and math.isfinite(rel)


@pytest.mark.parametrize("M", [1, 16])
def test_stack_replayed_as_one_cuda_graph_gives_the_eager_bits(stack, M):
    """The benchmark times the step as one captured CUDA graph: the four
    layers captured (prefetch and shared-expert side streams included) and
    replayed twice give the same bits as the same calls launched one by one,
    whose every stage the tests above check against the oracle."""
    layers, _ = stack
    x_bits = wl.token_rows(M, H, "stack-graph", M)
    main = torch.cuda.Stream(priority=-1)
    pref = torch.cuda.Stream()
    evs = [torch.cuda.Event() for _ in range(NL)]
    pf_bytes = min(H * H * 2, torch.cuda.get_device_properties(0).L2_cache_size // 2)
    xs = [wl.bits_to_torch(x_bits)] + [torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
                                      for _ in range(NL)]
    qkv = torch.empty((M, H + KV), dtype=torch.bfloat16, device="cuda")
    r = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    idxs = [torch.full((M, K8), -1, dtype=torch.int32, device="cuda") for _ in range(NL)]

    def run():
        for l in range(NL):
            pf = (pref, evs[l], layers[(l + 1) % NL].Wq.data_ptr(), pf_bytes)
            decode_layer(layers[l], xs[l], qkv, r, xs[l + 1], K8, idx=idxs[l], stream=main,
                         prefetch=pf)
        main.wait_stream(pref)

    run()
    torch.cuda.synchronize()
    assert dg.sync_check(main) == dg.DEC_OK
    eager = [x.clone() for x in xs[1:]] + [i.clone() for i in idxs]
    for t in xs[1:] + idxs:
        t.fill_(-1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        run()
    for _ in range(2):
        with torch.cuda.stream(main):
            g.replay()
        torch.cuda.synchronize()
        assert dg.sync_check(main) == dg.DEC_OK
        for a, b in zip(eager, xs[1:] + idxs):
            assert torch.equal(a, b)
        for t in xs[1:] + idxs:
            t.fill_(-1)
        torch.cuda.synchronize()
