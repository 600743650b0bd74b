"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a hand-worked fixture (tests/golden), a
closed form, an invariant, or a special case that reduces to a library
routine (numpy matmul, scipy's expit/softmax, torch.topk). Chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them. CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads as wl


def _golden(name):
    from conftest import GOLDEN
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _dec(bits):
    return oracle.bf16_to_f64(bits)


# ------------------------------------------------------------------ bf16 codec
def test_bf16_decode_golden():
    g = _golden("bf16_codec.json")
    for hexbits, val in g["decode"]:
        b = np.array([int(hexbits, 16)], dtype=np.uint16)
        assert _dec(b)[0] == val, hexbits


def test_bf16_round_golden():
    g = _golden("bf16_codec.json")
    for case in g["round"]:
        got = oracle.f64_to_bf16_bits(np.array([case["value"]]))[0]
        assert got == int(case["bits"], 16), case["why"]


def test_bf16_round_matches_torch_on_float32_inputs():
    # torch rounds float32 -> bfloat16 to nearest even; for inputs that are
    # already float32 there is no double rounding, so the two must agree.
    import torch
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormals
        np.float32(1.0) + np.arange(0, 512, dtype=np.float32) * np.float32(2 ** -15),
    ])
    ours = oracle.f64_to_bf16_bits(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_trip_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = _dec(bits)
    finite = np.isfinite(vals)
    back = oracle.f64_to_bf16_bits(vals[finite])
    # -0 and +0 both encode to their own sign; every finite pattern maps back to itself
    assert np.array_equal(back, bits[finite])


# ------------------------------------------------------------------ projection
def test_linear_golden():
    g = _golden("linear_hand.json")
    for c in g["cases"]:
        y, A = oracle.linear(_bits(c["x"]), _bits(c["W"]))
        assert np.array_equal(y, np.array(c["y"], dtype=np.float64))
        assert np.array_equal(A, np.array(c["absref"], dtype=np.float64))


def test_linear_matches_numpy_matmul():
    x = wl.normal_bf16((3, 200), 1.0, "pin", "lin", "x")
    W = wl.normal_bf16((37, 200), 0.02, "pin", "lin", "W")
    y, A = oracle.linear(x, W)
    ref = _dec(x) @ _dec(W).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(A, np.abs(_dec(x)) @ np.abs(_dec(W)).T, rtol=1e-12)


def test_linear_one_hot_rows_reproduce_x_exactly():
    x = wl.normal_bf16((4, 96), 1.0, "pin", "onehot", "x")
    W, perm = wl.one_hot_rows(50, 96, "pin", "onehot", "W")
    y, _ = oracle.linear(x, W)
    assert np.array_equal(y, _dec(x)[:, perm])


def test_linear_integer_inputs_exact():
    x = wl.integer_bf16((5, 64), -2, 2, "pin", "int", "x")
    W = wl.integer_bf16((33, 64), -2, 2, "pin", "int", "W")
    y, _ = oracle.linear(x, W)
    ref = _dec(x).astype(np.int64) @ _dec(W).astype(np.int64).T
    assert np.array_equal(y, ref.astype(np.float64))


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 8, 12, 16])
def test_linear_splitk_equals_unsplit(S):
    xi = wl.integer_bf16((3, 160), -2, 2, "pin", "sk", "x")
    Wi = wl.integer_bf16((17, 160), -2, 2, "pin", "sk", "W")
    assert np.array_equal(oracle.linear_splitk(xi, Wi, S), oracle.linear(xi, Wi)[0])
    xr = wl.normal_bf16((3, 160), 1.0, "pin", "sk", "xr")
    Wr = wl.normal_bf16((17, 160), 0.02, "pin", "sk", "Wr")
    np.testing.assert_allclose(oracle.linear_splitk(xr, Wr, S), oracle.linear(xr, Wr)[0],
                               rtol=1e-12, atol=1e-15)


def test_absref_bounds_result():
    x = wl.normal_bf16((2, 300), 1.0, "pin", "abs", "x")
    W = wl.normal_bf16((9, 300), 0.02, "pin", "abs", "W")
    y, A = oracle.linear(x, W)
    assert np.all(np.abs(y) <= A)
    # sum |x W| equals the product of the absolute values, term by term
    xa = oracle.f64_to_bf16_bits(np.abs(_dec(x)))
    Wa = oracle.f64_to_bf16_bits(np.abs(_dec(W)))
    assert np.array_equal(oracle.linear(xa, Wa)[0], A)


# ------------------------------------------------------------------ top-k + gates
def test_topk_golden():
    g = _golden("topk_hand.json")
    logits = np.array([g["logits"]])
    for c in g["cases"]:
        idx, gates = oracle.topk(logits, c["k"])
        assert idx[0].tolist() == c["idx"]
        if c["gates"] is not None:
            np.testing.assert_allclose(gates[0], c["gates"], rtol=1e-15, atol=1e-16)


def test_topk_is_prefix_of_full_sort():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((40, 384))
    logits[3, [5, 9, 11]] = logits[3].max() + 1.0   # a three-way tie at the top
    idx, _ = oracle.topk(logits, 8)
    for m in range(logits.shape[0]):
        order = np.lexsort((np.arange(384), -logits[m]))
        assert idx[m].tolist() == order[:8].tolist()
    assert idx[3, :3].tolist() == [5, 9, 11]


def test_topk_matches_torch_topk_on_separated_scores():
    import torch
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((64, 384))
    gaps = oracle.sorted_gaps(logits, 9)
    keep = np.all(gaps >= 1e-3, axis=1)
    idx, _ = oracle.topk(logits[keep], 8)
    ref = torch.topk(torch.from_numpy(logits[keep]), 8, dim=1, sorted=True).indices.numpy()
    assert np.array_equal(idx, ref.astype(np.int32))


def test_gates_equal_full_softmax_then_renormalise():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((16, 384))
    idx, gates = oracle.topk(logits, 8)
    p = scipy.special.softmax(logits, axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gates, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=1e-14)
    l = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gates[:, 0] / gates[:, 1], np.exp(l[:, 0] - l[:, 1]), rtol=1e-12)
    assert np.all(np.diff(gates, axis=1) <= 0)
    _, g1 = oracle.topk(logits, 1)
    assert np.all(g1 == 1.0)


# ------------------------------------------------------------------ SwiGLU expert
def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    for z in [0.1, 0.5, 1.0, 2.5, 7.0]:
        # silu(z) - silu(-z) = z, and silu(z) = z * expit(z)
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-15 * max(1, z)
        assert abs(oracle.silu(z) - z * scipy.special.expit(z)) < 1e-15 * max(1, z)
        assert abs(oracle.silu(-z) - (-z) * scipy.special.expit(-z)) < 1e-15 * max(1, z)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert -1e-15 < oracle.silu(-40.0) <= 0.0


def test_swiglu_golden():
    g = _golden("swiglu_hand.json")
    h = oracle.swiglu_hidden(_bits(g["x"]), _bits(g["W13"]), 1)
    np.testing.assert_allclose(h, g["h"], rtol=1e-15)
    o, _ = oracle.expert_mlp(_bits(g["x"]), _bits(g["W13"]), _bits(g["W2"]), 1)
    np.testing.assert_allclose(o, g["o"], rtol=1e-15)
    assert abs(h[0, 0] - g["h_if_gate_up_swapped"]) > 0.1


def test_swiglu_matches_numpy_and_expit():
    H, I, c = 96, 40, 3
    x = wl.normal_bf16((c, H), 1.0, "pin", "sw", "x")
    W13 = wl.normal_bf16((2 * I, H), 0.1, "pin", "sw", "W13")
    W2 = wl.normal_bf16((H, I), 0.1, "pin", "sw", "W2")
    a = _dec(x) @ _dec(W13)[:I].T
    b = _dec(x) @ _dec(W13)[I:].T
    h_ref = a * scipy.special.expit(a) * b
    np.testing.assert_allclose(oracle.swiglu_hidden(x, W13, I), h_ref, rtol=1e-11, atol=1e-13)
    o, A = oracle.expert_mlp(x, W13, W2, I)
    np.testing.assert_allclose(o, h_ref @ _dec(W2).T, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(A, np.abs(h_ref) @ np.abs(_dec(W2)).T, rtol=1e-10)
    hr = oracle.swiglu_hidden(x, W13, I, round_h=True)
    assert np.array_equal(hr, oracle.round_bf16(oracle.swiglu_hidden(x, W13, I)))


# ------------------------------------------------------------------ MoE block
def _bank_fetch(W13, W2):
    return lambda e: (W13[e], W2[e])


def test_moe_golden():
    g = _golden("moe_hand.json")
    W13 = np.stack([_bits(w) for w in g["W13"]])
    W2 = np.stack([_bits(w) for w in g["W2"]])
    r = oracle.moe(_bits(g["x"]), _bits(g["Wr"]), _bank_fetch(W13, W2), g["k"], 1,
                   shared=(_bits(g["Ws13"]), _bits(g["Ws2"])))
    assert r["idx"].tolist() == g["idx"]
    np.testing.assert_allclose(r["gates"], g["gates"], rtol=1e-15)
    np.testing.assert_allclose(r["out"], g["out"], rtol=1e-14)
    np.testing.assert_allclose(r["absref"], g["absref"], rtol=1e-14)


def _small_moe(E, H=64, I=24, M=5, key="moe"):
    x = wl.normal_bf16((M, H), 1.0, "pin", key, "x")
    Wr = wl.normal_bf16((E, H), 1.0 / math.sqrt(H), "pin", key, "Wr")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.1, "pin", key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.1, "pin", key, "W2", e) for e in range(E)])
    Ws13 = wl.normal_bf16((2 * I, H), 0.1, "pin", key, "Ws13")
    Ws2 = wl.normal_bf16((H, I), 0.1, "pin", key, "Ws2")
    return x, Wr, W13, W2, Ws13, Ws2, I


def _dense_swiglu(x, W13, W2, I):
    xv = _dec(x)
    a = xv @ _dec(W13)[:I].T
    b = xv @ _dec(W13)[I:].T
    return (a * scipy.special.expit(a) * b) @ _dec(W2).T


def test_moe_all_experts_uniform_gates_is_dense_mean():
    E = 6
    x, Wr, W13, W2, _, _, I = _small_moe(E, key="uni")
    Wr0 = np.zeros_like(Wr)                       # all scores 0 -> gates 1/E
    r = oracle.moe(x, Wr0, _bank_fetch(W13, W2), E, I, shared=None)
    assert np.all(r["idx"] == np.arange(E))       # ties resolve to index order
    np.testing.assert_allclose(r["gates"], 1.0 / E, rtol=1e-15)
    dense = sum(_dense_swiglu(x, W13[e], W2[e], I) for e in range(E)) / E
    np.testing.assert_allclose(r["out"], dense, rtol=1e-10, atol=1e-12)


def test_moe_single_expert_is_textbook_swiglu_mlp():
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(1, key="one")
    r = oracle.moe(x, Wr, _bank_fetch(W13, W2), 1, I, shared=(Ws13, Ws2))
    ref = _dense_swiglu(x, W13[0], W2[0], I) + _dense_swiglu(x, Ws13, Ws2, I)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-12)


def test_moe_zero_routed_down_projection_leaves_shared_expert():
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(8, key="zero")
    r = oracle.moe(x, Wr, _bank_fetch(W13, np.zeros_like(W2)), 3, I, shared=(Ws13, Ws2))
    np.testing.assert_allclose(r["out"], _dense_swiglu(x, Ws13, Ws2, I), rtol=1e-10, atol=1e-12)


def test_moe_matches_independent_dense_composition():
    # the gate-weighted sum written with numpy/scipy for every token
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(8, key="comp")
    k = 3
    r = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=(Ws13, Ws2))
    logits = _dec(x) @ _dec(Wr).T
    ref = _dense_swiglu(x, Ws13, Ws2, I)
    for m in range(x.shape[0]):
        order = np.lexsort((np.arange(8), -logits[m]))[:k]
        w = np.exp(logits[m, order] - logits[m, order[0]])
        w /= w.sum()
        for j, e in enumerate(order):
            ref[m] += w[j] * _dense_swiglu(x[m:m + 1], W13[e], W2[e], I)[0]
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-12)


def test_moe_is_linear_in_down_projections():
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(8, key="lin")
    r1 = oracle.moe(x, Wr, _bank_fetch(W13, W2), 3, I, shared=(Ws13, Ws2))
    dbl = lambda w: oracle.f64_to_bf16_bits(2.0 * _dec(w))  # exact: power of two
    r2 = oracle.moe(x, Wr, _bank_fetch(W13, dbl(W2)), 3, I, shared=(Ws13, dbl(Ws2)))
    assert np.array_equal(r2["out"], 2.0 * r1["out"])


def test_moe_invariant_under_expert_relabelling():
    E = 8
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(E, key="perm")
    perm = np.random.default_rng(5).permutation(E)
    r1 = oracle.moe(x, Wr, _bank_fetch(W13, W2), 3, I, shared=(Ws13, Ws2))
    r2 = oracle.moe(x, Wr[perm], _bank_fetch(W13[perm], W2[perm]), 3, I, shared=(Ws13, Ws2))
    np.testing.assert_allclose(r2["out"], r1["out"], rtol=1e-13, atol=1e-15)
    assert np.array_equal(perm[r2["idx"]], r1["idx"])


def test_moe_tokens_are_independent():
    x, Wr, W13, W2, Ws13, Ws2, I = _small_moe(8, key="tok")
    full = oracle.moe(x, Wr, _bank_fetch(W13, W2), 3, I, shared=(Ws13, Ws2))
    part = oracle.moe(x, Wr, _bank_fetch(W13, W2), 3, I, shared=(Ws13, Ws2), tokens=[1, 3])
    np.testing.assert_array_equal(part["out"][[1, 3]], full["out"][[1, 3]])
    assert np.all(np.isnan(part["out"][[0, 2, 4]]))
    solo = oracle.moe(x[3:4], Wr, _bank_fetch(W13, W2), 3, I, shared=(Ws13, Ws2))
    np.testing.assert_allclose(solo["out"][0], full["out"][3], rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------ decode layer
def test_decoder_layer_identity_and_doubling():
    H, I, E, M = 32, 8, 4, 3
    x = wl.normal_bf16((M, H), 1.0, "pin", "layer", "x")
    Wr = wl.normal_bf16((E, H), 0.2, "pin", "layer", "Wr")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.1, "pin", "layer", "W13", e) for e in range(E)])
    zW2 = np.zeros((E, H, I), dtype=np.uint16)
    Wkv = wl.normal_bf16((16, H), 0.1, "pin", "layer", "Wkv")
    zero = np.zeros((H, H), dtype=np.uint16)
    eye = _bits(np.eye(H))
    # Wq = Wo = 0 and zero expert outputs: the layer is the identity
    r = oracle.decoder_layer(x, zero, Wkv, zero, Wr, _bank_fetch(W13, zW2), 2, I, None)
    assert np.array_equal(r["out"], x)
    assert np.array_equal(r["kv"], oracle.f64_to_bf16_bits(oracle.linear(x, Wkv)[0]))
    # Wq = Wo = I: q = x and r = x + x = 2x, exactly
    r = oracle.decoder_layer(x, eye, Wkv, eye, Wr, _bank_fetch(W13, zW2), 2, I, None)
    assert np.array_equal(r["q"], x)
    assert np.array_equal(_dec(r["out"]), 2.0 * _dec(x))


def test_decoder_layer_o_projection_reads_q_not_x():
    # Wq = 2I, Wo = I: q = 2x and r = bf16(x + 2x) = bf16(3x). An o projection
    # wired to x would give 2x; one that skipped the residual would give 2x too.
    H, I, E, M = 32, 8, 4, 3
    x = wl.normal_bf16((M, H), 1.0, "pin", "layer-q", "x")
    Wr = wl.normal_bf16((E, H), 0.2, "pin", "layer-q", "Wr")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.1, "pin", "layer-q", "W13", e) for e in range(E)])
    zW2 = np.zeros((E, H, I), dtype=np.uint16)
    Wkv = wl.normal_bf16((16, H), 0.1, "pin", "layer-q", "Wkv")
    r = oracle.decoder_layer(x, _bits(2 * np.eye(H)), Wkv, _bits(np.eye(H)), Wr,
                             _bank_fetch(W13, zW2), 2, I, None)
    three_x = wl.f32_to_bf16_bits(np.float32(3) * _dec(x).astype(np.float32))  # exact in fp32
    assert np.array_equal(r["q"], _bits(2 * _dec(x)))
    assert np.array_equal(r["r"], three_x)
    assert np.array_equal(r["out"], three_x)          # zero expert outputs: x' = r
    # A permutation for Wq (row n picks column perm[n]) and Wo = 2I:
    # r = bf16(x + 2 x[:, perm]); a transposed Wq would pick the inverse permutation.
    perm = np.random.default_rng(5).permutation(H)
    P = np.zeros((H, H))
    P[np.arange(H), perm] = 1.0
    assert not np.array_equal(perm, np.argsort(perm))
    r = oracle.decoder_layer(x, _bits(P), Wkv, _bits(2 * np.eye(H)), Wr,
                             _bank_fetch(W13, zW2), 2, I, None)
    xv = _dec(x).astype(np.float32)
    assert np.array_equal(r["q"], x[:, perm])
    assert np.array_equal(r["r"], wl.f32_to_bf16_bits(xv + np.float32(2) * xv[:, perm]))


def test_decoder_layer_moe_reads_r_and_adds_r():
    # With r = bf16(3x) != x and nonzero experts, the block's input and its
    # residual must both be r: x' = bf16(r + moe(r)), routed on r's scores.
    H, I, E, M, k = 32, 8, 6, 4, 2
    x = wl.normal_bf16((M, H), 1.0, "pin", "layer-m", "x")
    Wr = wl.normal_bf16((E, H), 0.3, "pin", "layer-m", "Wr")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.2, "pin", "layer-m", "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.2, "pin", "layer-m", "W2", e) for e in range(E)])
    Ws = (wl.normal_bf16((2 * I, H), 0.2, "pin", "layer-m", "Ws13"),
          wl.normal_bf16((H, I), 0.2, "pin", "layer-m", "Ws2"))
    Wkv = wl.normal_bf16((16, H), 0.1, "pin", "layer-m", "Wkv")
    lay = oracle.decoder_layer(x, _bits(2 * np.eye(H)), Wkv, _bits(np.eye(H)), Wr,
                               _bank_fetch(W13, W2), k, I, Ws)
    r = wl.f32_to_bf16_bits(np.float32(3) * _dec(x).astype(np.float32))
    on_r = oracle.moe(r, Wr, _bank_fetch(W13, W2), k, I, shared=Ws)
    on_x = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=Ws)
    assert np.array_equal(lay["idx"], on_r["idx"])
    want = oracle.f64_to_bf16_bits(_dec(r) + on_r["out"])
    assert np.array_equal(lay["out"], want)
    # the pin has teeth: feeding x to the block, or adding x, changes the result
    assert not np.array_equal(want, oracle.f64_to_bf16_bits(_dec(r) + on_x["out"]))
    assert not np.array_equal(want, oracle.f64_to_bf16_bits(_dec(x) + on_r["out"]))


# ------------------------------------------------------------------ generators
def test_generators_are_deterministic_and_scaled():
    a = wl.normal_bf16((64, 512), 0.02, "gen", 1)
    b = wl.normal_bf16((64, 512), 0.02, "gen", 1)
    c = wl.normal_bf16((64, 512), 0.02, "gen", 2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    v = _dec(a)
    assert abs(v.std() - 0.02) < 0.001 and abs(v.mean()) < 0.001
    xr = wl.token_rows(3, 128, "gen", "x", attempts=[0, 1, 0])
    assert np.array_equal(xr[0], wl.token_rows(1, 128, "gen", "x")[0])
    assert not np.array_equal(xr[1], wl.token_rows(2, 128, "gen", "x")[1])


def test_skewed_router_scales():
    c = wl.router_scales(384, 1.0)
    assert abs(c.mean() - 1.0) < 1e-12 and np.all(np.diff(c) < 0)
    assert np.allclose(wl.router_scales(16, 0.0), 1.0)
    W = _dec(wl.skewed_router_bf16(8, 4096, 1.0, "gen", "Wr"))
    sd = W.std(axis=1) / wl.ROUTER_STD
    assert np.allclose(sd, wl.router_scales(8, 1.0), rtol=0.05)


def test_gates_for_a_given_choice():
    # the gates of the oracle's own choice equal the top-k routine's, and a
    # given route reproduces the unrouted block exactly when it is that choice
    l = oracle.bf16_to_f64(wl.normal_bf16((5, 24), 1.0, "pin", "gates-for"))
    idx, g = oracle.topk(l, 4)
    np.testing.assert_allclose(oracle.gates_for(l, idx), g, rtol=1e-14)
    # a permuted choice permutes the gates; sum is 1; ratio is exp(l_a - l_b)
    gp = oracle.gates_for(l, idx[:, ::-1])
    np.testing.assert_allclose(gp, g[:, ::-1], rtol=1e-14)
    H, I, E, M, k = 16, 8, 6, 3, 2
    x = wl.normal_bf16((M, H), 1.0, "pin", "route", "x")
    Wr = wl.normal_bf16((E, H), 0.3, "pin", "route", "Wr")
    W13 = np.stack([wl.normal_bf16((2 * I, H), 0.2, "pin", "route", "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((H, I), 0.2, "pin", "route", "W2", e) for e in range(E)])
    a = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I)
    b = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, route=a["idx"])
    assert np.array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-13, atol=1e-15)
    # another choice: each token's output is the gate-weighted sum of exactly
    # the experts named, with gates from the given scores
    alt = np.array([[0, 1], [2, 3], [5, 4]], dtype=np.int32)
    c = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, route=alt)
    gl = oracle.gates_for(c["logits"], alt)
    for m in range(M):
        want = sum(gl[m, j] * oracle.expert_mlp(x[m:m + 1], W13[alt[m, j]], W2[alt[m, j]], I)[0][0]
                   for j in range(k))
        np.testing.assert_allclose(c["out"][m], want, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ latent block
def _latent_case(H, L, E, I, M, key):
    x = wl.normal_bf16((M, H), 1.0, "pin", key, "x")
    Wr = wl.normal_bf16((E, H), 0.3, "pin", key, "Wr")
    Ws = (wl.normal_bf16((2 * I, H), 0.2, "pin", key, "Ws13"),
          wl.normal_bf16((H, I), 0.2, "pin", key, "Ws2"))
    W13 = np.stack([wl.normal_bf16((2 * I, L), 0.2, "pin", key, "W13", e) for e in range(E)])
    W2 = np.stack([wl.normal_bf16((L, I), 0.2, "pin", key, "W2", e) for e in range(E)])
    return x, Wr, Ws, W13, W2


def test_latent_with_identity_projections_is_the_plain_block():
    # L = H, latent rows = I, Wup = I: lat = x and z·Iᵀ = z exactly, so the
    # block is the plain block; with the diagnostic rounding of lat, h and z,
    # z is the plain block's routed sum (h rounded) rounded once more
    H, I, E, M, k = 24, 8, 6, 4, 2
    x, Wr, Ws, W13, W2 = _latent_case(H, H, E, I, M, "lat-id")
    eye = _bits(np.eye(H))
    Wrl = np.concatenate([Wr, eye])
    r = oracle.moe_latent(x, Wrl, E, _bank_fetch(W13, W2), k, I, eye, shared=Ws)
    plain = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=Ws)
    routed = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=None)
    assert np.array_equal(r["idx"], plain["idx"])
    assert np.array_equal(r["lat"], _dec(x))
    np.testing.assert_allclose(r["z"], routed["out"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["out"], plain["out"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["absref"], plain["absref"], rtol=1e-14, atol=1e-15)
    rr = oracle.moe_latent(x, Wrl, E, _bank_fetch(W13, W2), k, I, eye, shared=Ws,
                           round_inter=True)
    routed_h = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=None, round_h=True)
    s_h, _ = oracle.expert_mlp(x, Ws[0], Ws[1], I, round_h=True)
    np.testing.assert_allclose(rr["out"], oracle.round_bf16(routed_h["out"]) + s_h, rtol=1e-14,
                               atol=1e-15)
    assert not np.allclose(rr["out"], r["out"], rtol=1e-9, atol=0)


def test_expert_on_fp64_activations_matches_bf16_expert():
    H, I = 40, 16
    x = wl.normal_bf16((3, H), 1.0, "pin", "f64act", "x")
    W13 = wl.normal_bf16((2 * I, H), 0.2, "pin", "f64act", "W13")
    W2 = wl.normal_bf16((H, I), 0.2, "pin", "f64act", "W2")
    for rh in (False, True):
        a, aA = oracle.expert_mlp(x, W13, W2, I, round_h=rh)
        b, bA = oracle.expert_mlp_f64act(_dec(x), W13, W2, I, round_h=rh)
        np.testing.assert_allclose(b, a, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(bA, aA, rtol=1e-13, atol=1e-15)


def test_latent_input_is_projected_and_output_projected_back():
    # latent rows 2I (lat = 2x exactly) and Wup = I/2: the block equals the
    # plain routed block on 2x, routed on x's scores, rounded, halved, plus the
    # shared expert. lat = x, or an ignored Wup, would give another result.
    H, I, E, M, k = 24, 8, 6, 4, 2
    x, Wr, Ws, W13, W2 = _latent_case(H, H, E, I, M, "lat-scale")
    r = oracle.moe_latent(x, np.concatenate([Wr, _bits(2 * np.eye(H))]), E,
                          _bank_fetch(W13, W2), k, I, _bits(0.5 * np.eye(H)), shared=Ws)
    x2 = _bits(2 * _dec(x))
    half_Wr = _bits(0.5 * _dec(Wr))                    # (2x)·(Wr/2)ᵀ = x·Wrᵀ exactly
    on2x = oracle.moe(x2, half_Wr, _bank_fetch(W13, W2), k, I, shared=None, route=r["idx"])
    s, _ = oracle.expert_mlp(x, Ws[0], Ws[1], I)
    np.testing.assert_allclose(on2x["gates"], r["gates"], rtol=1e-14)
    want = 0.5 * on2x["out"] + s
    np.testing.assert_allclose(r["out"], want, rtol=1e-14, atol=1e-15)
    on1x = oracle.moe(x, Wr, _bank_fetch(W13, W2), k, I, shared=None, route=r["idx"])
    assert not np.allclose(r["out"], 0.5 * on1x["out"] + s, rtol=1e-6)


def test_latent_special_cases():
    H, L, I, E, M, k = 32, 12, 8, 5, 3, 2
    x, Wr, Ws, W13, W2 = _latent_case(H, L, E, I, M, "lat-special")
    Wd = wl.normal_bf16((L, H), 0.2, "pin", "lat-special", "Wd")
    Wup = wl.normal_bf16((H, L), 0.2, "pin", "lat-special", "Wup")
    f = _bank_fetch(W13, W2)
    base = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E, f, k, I, Wup, shared=Ws)
    assert base["out"].shape == (M, H) and base["lat"].shape == (M, L)
    s, sA = oracle.expert_mlp(x, Ws[0], Ws[1], I)
    # routing comes from the router rows alone
    other = oracle.moe_latent(x, np.concatenate([Wr, np.zeros_like(Wd)]), E, f, k, I, Wup,
                              shared=Ws)
    assert np.array_equal(other["idx"], base["idx"])
    assert np.array_equal(other["idx"], oracle.topk(oracle.linear(x, Wr)[0], k)[0])
    np.testing.assert_array_equal(other["gates"], base["gates"])
    # the latent input is the latent projection of x
    assert np.array_equal(base["lat"], oracle.linear(x, Wd)[0])
    # Wup = 0: the shared expert alone
    z0 = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E, f, k, I, np.zeros_like(Wup),
                           shared=Ws)
    assert np.array_equal(z0["out"], s) and np.array_equal(z0["absref"], sA)
    # no shared expert: the up-projection of z, and linear in Wup
    a = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E, f, k, I, Wup, shared=None)
    b = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E, f, k, I, _bits(2 * _dec(Wup)),
                          shared=None)
    assert np.array_equal(b["out"], 2 * a["out"])
    assert np.array_equal(b["absref"], 2 * a["absref"])
    assert np.all(a["absref"] >= np.abs(a["out"]) * (1 - 1e-12))
    # the scale is the whole expression in absolute values: with every weight
    # and activation replaced by its magnitude the block's value equals it
    absb = lambda w: w & np.uint16(0x7FFF)
    pos = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E,
                            lambda e: (W13[e], absb(W2[e])), k, I, absb(Wup), shared=None,
                            route=a["idx"])
    np.testing.assert_allclose(pos["absref"], a["absref"], rtol=1e-12)
    np.testing.assert_allclose(base["out"], a["out"] + s, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(a["out"], a["z"] @ _dec(Wup).T, rtol=1e-12, atol=1e-14)
    # token independence
    t = oracle.moe_latent(x, np.concatenate([Wr, Wd]), E, f, k, I, Wup, shared=Ws, tokens=[1])
    assert np.array_equal(t["out"][1], base["out"][1]) and np.isnan(t["out"][0]).all()
