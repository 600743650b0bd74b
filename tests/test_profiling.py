"""The ncu summary tool (moe_decode_gemm_gb300/profiling.py) on the host: kernel
labels from demangled names, and the launch-list aggregation."""
import io

from moe_decode_gemm_gb300 import profiling as pf

SA = "(CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, dg::StreamArgs)"


def test_labels_of_every_kernel_family():
    cases = {
        "void dg::wstream_kernel<8, 3, 0, false, false, false, 0, 2, true, 1>" + SA:
            "projection [wstream XR=8 S=3 bf16 128-row 2/SM cluster CUDA cores]",
        "void dg::wstream_kernel<16, 3, 1, false, false, true, 0, 1, false, 0>" + SA:
            "projection [wstream XR=16 S=3 bf16+residual 256-row]",
        "void dg::wstream_kernel<32, 3, 3, true, true, false, 2, 1, false, 0>" + SA:
            "routed expert gate/up [wstream XR=32 S=3 SwiGLU 128-row]",
        "void dg::wstream_kernel<16, 3, 2, false, true, true, 2, 1, false, 0>" + SA:
            "routed expert down [wstream XR=16 S=3 fp32 256-row]",
        "void dg::wstream_kernel<8, 6, 2, false, false, false, 1, 1, true, 0>" + SA:
            "router + top-k [wstream XR=8 S=6 fp32 128-row cluster]",
        "void dg::wstream_kernel<64, 2, 3, true, false, false, 3, 1, false, 0>" + SA:
            "shared expert gate/up [wstream XR=64 S=2 SwiGLU 128-row]",
        "void dg::tc_linear_kernel<1>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "projection [tcgen05 bf16+residual]",
        "void dg::tc_cluster_kernel<0>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "projection [tcgen05 bf16 cluster]",
        "void dg::tc_cluster_kernel<1, 1>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "projection [tcgen05 bf16+residual cluster, 64 k per stage]",
        "void dg::tc_cluster_kernel<2, 1, true>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "router + top-k [tcgen05 cluster, 64 k per stage]",
        "void dg::tc_cluster_kernel<0, 2, false>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "projection [tcgen05 bf16 cluster, 128 k per stage]",
        "void dg::tc_linear_kernel<3, true>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "shared expert gate/up [tcgen05 SwiGLU]",
        "void dg::tc_linear_kernel<2, false>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs, int, unsigned int)":
            "shared expert down [tcgen05 fp32]",
        "void dg::gemv_slab_kernel<8, 0>(CUtensorMap_st, const unsigned short *, long long, dg::StreamArgs)":
            "projection [slab 8 rows/CTA bf16, CUDA cores]",
        "void dg::gemv_mma_kernel<32, 4, 4, 2, 1>(CUtensorMap_st, CUtensorMap_st, dg::StreamArgs)":
            "projection [slab 32 rows/CTA XR=4 bf16+residual, mma.sync, 2/SM]",
        "void dg::gemv_mma_kernel<64, 16, 2, 1, 0>(CUtensorMap_st, CU":
            "projection [slab 64 rows/CTA XR=16 bf16, mma.sync]",
        "dg::schedule_gather_kernel(const uint4 *, const int *, int, int, int, int, uint4 *, int *)":
            "schedule + gather",
        "dg::combine_kernel(const float *, const float *, const float *)": "combine",
        "dg::prefetch_kernel(const unsigned char *, long long)": "l2_prefetch",
    }
    for name, want in cases.items():
        assert pf.kernel_label(name) == want, name


def test_labels_accept_shorter_template_lists():
    # names with fewer template arguments (defaults not printed) still parse
    assert pf.kernel_label("void dg::wstream_kernel<16, 3, 0, false, false, false>" + SA) == \
        "projection [wstream XR=16 S=3 bf16 128-row]"


def test_launch_list_aggregates_by_label(tmp_path):
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = [
        (0, "void dg::wstream_kernel<8, 6, 2, false, false, false, 1, 1, true, 0>" + SA, "usecond", "10.0"),
        (1, "void dg::wstream_kernel<32, 3, 3, true, true, false, 2, 1, false, 0>" + SA, "msecond", "2.5"),
        (2, "void dg::wstream_kernel<32, 3, 3, true, true, false, 2, 1, false, 0>" + SA, "usecond", "1,500.0"),
        (3, "dg::combine_kernel(const float *)", "nsecond", "4000"),
    ]
    p = tmp_path / "launches.csv"
    p.write_text(hdr + "".join('"%d","%s","gpu__time_duration.sum","%s","%s"\n' % r for r in rows))
    out = io.StringIO()
    pf.launches(str(p), out=out)
    text = out.getvalue()
    lines = [ln for ln in text.splitlines() if ln.startswith("| ") and "kernel" not in ln]
    # sorted by total time: the gate/up kernel (2 launches, 4000 us) first
    assert lines[0] == "| routed expert gate/up [wstream XR=32 S=3 SwiGLU 128-row] | 2 | 4000.0 | 99.7% | 2000.0 |"
    assert "| router + top-k [wstream XR=8 S=6 fp32 128-row cluster] | 1 | 10.0 |" in text
    assert "| combine | 1 | 4.0 |" in text
    assert "total 4014.0 us over 4 launches" in text
