"""GPU checks of the helper entry points: L2 prefetch, residual add, the
bounded-wait failure detection, launch accounting and the timing probe."""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_decode_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"


import moe_decode_gemm_gb300 as dg  # noqa: E402


def test_l2_prefetch_runs_and_changes_nothing():
    t = torch.randn(1 << 22, device="cuda").to(torch.bfloat16)
    before = t.clone()
    n0 = dg.launch_count()
    dg.l2_prefetch(t)
    dg.l2_prefetch(t.data_ptr(), 1 << 30)          # capped at half of L2
    assert dg.sync_check() == dg.DEC_OK
    assert dg.launch_count() == n0 + 2
    assert torch.equal(t, before)


def test_add_matches_oracle_rounding():
    a = wl.normal_bf16((4097,), 3.0, "add", "a")
    b = wl.normal_bf16((4097,), 3.0, "add", "b")
    out = dg.dec_add(wl.bits_to_torch(a), wl.bits_to_torch(b))
    assert dg.sync_check() == dg.DEC_OK
    # the exact sum of two bf16 values is representable in fp32, so both
    # sides round the same exact value
    ref = oracle.f64_to_bf16_bits(oracle.bf16_to_f64(a) + oracle.bf16_to_f64(b))
    assert np.array_equal(wl.torch_to_bits(out), ref)


def test_bounded_wait_reports_timeout_and_library_recovers():
    dg.selftest_timeout(2_000_000)                  # 2 ms on a barrier nobody completes
    assert dg.sync_check() == dg.DEC_ETIMEOUT
    assert dg.sync_check() == dg.DEC_OK             # status cleared
    x = wl.normal_bf16((2, 256), 1.0, "after", "x")
    W = wl.normal_bf16((64, 256), 0.02, "after", "W")
    y = dg.dec_linear(wl.bits_to_torch(x), wl.bits_to_torch(W))
    assert dg.sync_check() == dg.DEC_OK
    ref, A = oracle.linear(x, W)
    err = np.abs(y.float().cpu().numpy() - ref)
    assert np.all(err <= 8e-3 * np.abs(ref) + 1e-3 * A)


def test_probe_times_projection_launches():
    x = wl.bits_to_torch(wl.normal_bf16((1, 4096), 1.0, "probe", "x"))
    W = wl.bits_to_torch(wl.normal_bf16((4096, 4096), 0.02, "probe", "W"))
    dg.probe_begin(dg.PROBE_LINEAR, 8)
    for _ in range(5):
        dg.dec_linear(x, W)
    ms, n = dg.probe_end()
    assert n == 5 and ms > 0.0


def test_kernels_per_moe_block_and_per_layer():
    # the MoE block with a shared expert is seven launches: the shared
    # expert's gate/up and down (side stream), the router with the top-k,
    # schedule + gather, the routed gate/up and down projections, and the
    # combine; five without a shared expert. A decode layer adds the fused
    # q|kv and the o projection and the L2 prefetch: ten.
    import math
    from moe_decode_gemm_gb300.stack import decode_layer

    M, H, KV, E, I, k = 4, 256, 64, 32, 128, 4
    t = wl.bits_to_torch
    g = lambda *s, std=0.02, key="": t(wl.normal_bf16(s, std, "count", key, *s))
    x = g(M, H, std=1.0, key="x")
    Wr = g(E, H, std=1.0 / math.sqrt(H), key="Wr")
    W13, W2 = g(E, 2 * I, H, key="W13"), g(E, H, I, key="W2")
    Ws13, Ws2 = g(2 * I, H, key="Ws13"), g(H, I, key="Ws2")
    dg.moe_decode(x, Wr, W13, W2, Ws13, Ws2, k)        # workspace set up
    assert dg.sync_check() == dg.DEC_OK
    n0 = dg.launch_count()
    dg.moe_decode(x, Wr, W13, W2, Ws13, Ws2, k)
    assert dg.launch_count() - n0 == 7
    n0 = dg.launch_count()
    dg.moe_decode(x, Wr, W13, W2, None, None, k)
    assert dg.launch_count() - n0 == 5

    class L:
        pass
    L.Wqkv, L.Wo, L.Wr, L.W13, L.W2, L.Ws13, L.Ws2 = g(H + KV, H, key="qkv"), g(H, H, key="o"), \
        Wr, W13, W2, Ws13, Ws2
    bufs = [torch.empty((M, n), dtype=torch.bfloat16, device="cuda") for n in (H + KV, H, H)]
    side, ev = torch.cuda.Stream(), torch.cuda.Event()
    decode_layer(L, x, *bufs, k, prefetch=(side, ev, L.Wqkv.data_ptr(), 1 << 20))
    torch.cuda.synchronize()
    n0 = dg.launch_count()
    decode_layer(L, x, *bufs, k, prefetch=(side, ev, L.Wqkv.data_ptr(), 1 << 20))
    torch.cuda.synchronize()
    assert dg.launch_count() - n0 == 10
    assert dg.sync_check() == dg.DEC_OK
