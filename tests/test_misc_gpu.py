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
