"""Summaries of Nsight Compute output for this library's kernels.

    python -m moe_decode_gemm_gb300.profiling launches LAUNCHES.csv
        Per kernel: launches, total device time, share of the total and the
        average, from a launch list taken with
        `ncu --metrics gpu__time_duration.sum --csv --log-file LAUNCHES.csv`.
        Kernels of the input generators (torch's random-number kernels) are
        left out: they run before the timed region.

    python -m moe_decode_gemm_gb300.profiling raw RAW.csv
        The DRAM, tensor-pipe, occupancy and stall counters of each captured
        launch, from `ncu -i REPORT --page raw --csv`.

    python -m moe_decode_gemm_gb300.profiling case moe TOKENS EXPERTS [CALLS]
    python -m moe_decode_gemm_gb300.profiling case linear M N K [CALLS]
    python -m moe_decode_gemm_gb300.profiling case router TOKENS [CALLS]
    python -m moe_decode_gemm_gb300.profiling case shared TOKENS [CALLS]
    python -m moe_decode_gemm_gb300.profiling case prefetch M ON [CALLS]
        A small case to run under `ncu --set full` (needs a GPU): CALLS
        (default 3) MoE blocks of TOKENS tokens over a bank of EXPERTS routed
        experts (hidden 7168, intermediate 2048, top-8, no shared expert),
        or CALLS projections alternating over two weight matrices, or CALLS
        MoE blocks with the full router (384 experts x 7168) and tiny experts
        (intermediate 16), to profile routing alone, or CALLS MoE blocks with
        the full-size shared expert over a bank of 48 routed experts (4.2 GB;
        the shared expert's kernels), or CALLS 7168 x 7168 projections of M
        tokens, each after a write of 256 MB that evicts L2 and -- with ON = 1
        -- an l2_prefetch of the weight's first half-L2 bytes (for the L2 hit
        rate of the projection under `ncu --cache-control none`). Inputs are
        seeded and synthetic; each expert is 88 MB, so a bank of 32 (2.8 GB)
        is far larger than L2 and its DRAM counters mean what they say.

Kernel names are mapped to the step of the decode layer they run: the weight
streaming kernel's template arguments say which (token rows per stage, ring
depth, epilogue, paired gate/up tiles, grouped experts, 256-row tiles, role).
"""
import collections
import csv
import re
import sys

_EPI = {"0": "bf16", "1": "bf16+residual", "2": "fp32", "3": "SwiGLU"}
_ROLE = {"0": "projection", "1": "router + top-k", "2": "routed expert", "3": "shared expert"}
_TRUE = ("true", "1")


def kernel_label(name):
    """Readable label for one (demangled) kernel name."""
    m = re.search(r"wstream_kernel<([^>]*)>", name)
    if m:
        p = [v.strip() for v in m.group(1).split(",")]
        # defaults: projection role, 1 CTA per SM, no cluster, consumer chosen per group
        p += ["0"] * (10 - len(p))
        xr, st, epi, paired, grouped, wide, role, minb, cluster, path = p[:10]
        role = _ROLE.get(role, role)
        part = ""
        if role in ("routed expert", "shared expert"):
            part = " gate/up" if paired in _TRUE else " down"
        tile = "256-row" if wide in _TRUE else "128-row"
        extra = (" 2/SM" if minb == "2" else "") + (" cluster" if cluster in _TRUE else "")
        extra += " CUDA cores" if path == "1" else ""
        return "%s%s [wstream XR=%s S=%s %s %s%s]" % (role, part, xr, st, _EPI.get(epi, epi), tile,
                                                     extra)
    m = re.search(r"tc_linear_kernel<(\d+)(?:,\s*(\w+))?>", name)
    if m:
        if m.group(2) in _TRUE:
            return "shared expert gate/up [tcgen05 SwiGLU]"
        if m.group(1) == "2":  # the fp32-output instance runs the shared expert's down projection
            return "shared expert down [tcgen05 fp32]"
        return "projection [tcgen05 %s]" % _EPI.get(m.group(1), m.group(1))
    # <rows, token rows, k blocks per stage, CTAs per SM, epilogue>
    m = re.search(r"gemv_mma_kernel<(\d+),\s*(\d+),\s*\d+,\s*(\d+),\s*(\d+)>", name)
    if m:
        return "projection [slab %s rows/CTA XR=%s %s, mma.sync%s]" % (
            m.group(1), m.group(2), _EPI.get(m.group(4), m.group(4)),
            ", 2/SM" if m.group(3) == "2" else "")
    m = re.search(r"gemv_slab_kernel<(\d+),\s*(\d+)>", name)
    if m:
        return "projection [slab %s rows/CTA %s, CUDA cores]" % (m.group(1),
                                                                _EPI.get(m.group(2), m.group(2)))
    # <epilogue, k boxes per stage, router>
    m = re.search(r"tc_cluster_kernel<(\d+)(?:,\s*(\d+))?(?:,\s*(\w+))?>", name)
    if m:
        stage = "" if m.group(2) is None else ", %d k per stage" % (64 * int(m.group(2)))
        if m.group(3) in _TRUE:
            return "router + top-k [tcgen05 cluster%s]" % stage
        return "projection [tcgen05 %s cluster%s]" % (_EPI.get(m.group(1), m.group(1)), stage)
    for k, lab in (("schedule_gather_kernel", "schedule + gather"),
                   ("combine_kernel", "combine"), ("add_kernel", "residual add"),
                   ("prefetch_kernel", "l2_prefetch")):
        if k in name:
            return lab
    return name[:60]


_UNIT_US = {"ns": 1e-3, "nsecond": 1e-3, "usecond": 1.0, "us": 1.0, "ms": 1e3, "msecond": 1e3}


def _rows(path):
    rows = list(csv.reader(open(path, newline="")))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    return rows[hi], rows[hi + 1:]


def launches(path, out=sys.stdout):
    hdr, rows = _rows(path)
    ki, mi, ui, vi = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Unit",
                                             "Metric Value"))
    agg = collections.OrderedDict()
    for r in rows:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum" or "distribution_" in r[ki]:
            continue
        us = float(r[vi].replace(",", "")) * _UNIT_US[r[ui]]
        a = agg.setdefault(kernel_label(r[ki]), [0, 0.0])
        a[0] += 1
        a[1] += us
    tot = sum(a[1] for a in agg.values())
    print("| kernel | launches | total us | share | avg us |", file=out)
    print("|---|---:|---:|---:|---:|", file=out)
    for k, (n, us) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        print("| %s | %d | %.1f | %.1f%% | %.1f |" % (k, n, us, 100 * us / tot, us / n), file=out)
    print("\ntotal %.1f us over %d launches" % (tot, sum(a[0] for a in agg.values())), file=out)


_RAW = re.compile(r"^(dram__bytes_(read|write)\.sum|"
                  r"gpu__dram_throughput\.avg\.pct_of_peak_sustained_elapsed|"
                  r"gpu__time_duration\.sum|"
                  r"sm__pipe_tensor_cycles_active\.avg\.pct_of_peak_sustained_active|"
                  r"sm__warps_active\.avg\.pct_of_peak_sustained_active|"
                  r"launch__registers_per_thread|launch__grid_size|"
                  r"launch__shared_mem_per_block_dynamic|lts__t_sector_hit_rate\.pct|"
                  r"smsp__average_warps_issue_stalled_(long_scoreboard|barrier|wait|"
                  r"short_scoreboard|no_instruction|membar|sleeping|math_pipe_throttle)"
                  r"_per_issue_active\.ratio)$")


def raw(path, out=sys.stdout):
    rows = list(csv.reader(open(path, newline="")))
    hdr, units = rows[0], rows[1]
    ki = hdr.index("Kernel Name")
    for r in rows[2:]:
        print("## %s" % kernel_label(r[ki]), file=out)
        for i, h in enumerate(hdr):
            if _RAW.search(h):
                print("- %s = %s %s" % (h, r[i], units[i]), file=out)
        print(file=out)


def case(kind, *args):
    import os

    import torch

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import moe_decode_gemm_gb300 as dg
    from workloads import (HIDDEN, INTER, ROUTER_STD, TOPK, WEIGHT_STD, normal_bf16_cuda)

    if kind == "moe":
        M, E = int(args[0]), int(args[1])
        calls = int(args[2]) if len(args) > 2 else 3
        H, I = HIDDEN, INTER
        W13 = normal_bf16_cuda((E, 2 * I, H), WEIGHT_STD, "profile", "W13")
        W2 = normal_bf16_cuda((E, H, I), WEIGHT_STD, "profile", "W2")
        Wr = normal_bf16_cuda((E, H), ROUTER_STD, "profile", "Wr")
        x = normal_bf16_cuda((M, H), 1.0, "profile", "x", M)
        idx = torch.empty((M, TOPK), dtype=torch.int32, device="cuda")
        for _ in range(calls):
            dg.moe_decode(x, Wr, W13, W2, None, None, TOPK, topk_idx=idx)
        torch.cuda.synchronize()
        active = len(set(idx.cpu().numpy().ravel().tolist()))
        print("moe tokens=%d experts=%d active=%d calls=%d" % (M, E, active, calls))
    elif kind == "router":
        M = int(args[0])
        calls = int(args[1]) if len(args) > 1 else 3
        E, H, I = 384, HIDDEN, 16
        W13 = normal_bf16_cuda((E, 2 * I, H), WEIGHT_STD, "profile", "W13r")
        W2 = normal_bf16_cuda((E, H, I), WEIGHT_STD, "profile", "W2r")
        Wr = normal_bf16_cuda((E, H), ROUTER_STD, "profile", "Wr")
        x = normal_bf16_cuda((M, H), 1.0, "profile", "xr", M)
        for _ in range(calls):
            dg.moe_decode(x, Wr, W13, W2, None, None, TOPK)
        torch.cuda.synchronize()
        print("router tokens=%d experts=%d calls=%d" % (M, E, calls))
    elif kind == "linear":
        M, N, K = int(args[0]), int(args[1]), int(args[2])
        calls = int(args[3]) if len(args) > 3 else 3
        Ws = [normal_bf16_cuda((N, K), WEIGHT_STD, "profile", "W", i) for i in range(2)]
        x = normal_bf16_cuda((M, K), 1.0, "profile", "x", M)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for i in range(calls):
            dg.dec_linear(x, Ws[i % 2], y)
        torch.cuda.synchronize()
        print("linear M=%d N=%d K=%d regime=%s calls=%d" % (M, N, K, dg.last_choice(), calls))
    elif kind == "shared":
        M = int(args[0])
        calls = int(args[1]) if len(args) > 1 else 3
        E, H, I = 48, HIDDEN, INTER   # enough distinct experts that the shared expert is not
        #                               given dedicated SMs, as at 16-64 tokens over 384 experts
        W13 = normal_bf16_cuda((E, 2 * I, H), WEIGHT_STD, "profile", "W13s")
        W2 = normal_bf16_cuda((E, H, I), WEIGHT_STD, "profile", "W2s")
        Wr = normal_bf16_cuda((E, H), ROUTER_STD, "profile", "Wrs")
        Ws13 = normal_bf16_cuda((2 * I, H), WEIGHT_STD, "profile", "Ws13")
        Ws2 = normal_bf16_cuda((H, I), WEIGHT_STD, "profile", "Ws2")
        x = normal_bf16_cuda((M, H), 1.0, "profile", "xs", M)
        for _ in range(calls):
            dg.moe_decode(x, Wr, W13, W2, Ws13, Ws2, TOPK)
        torch.cuda.synchronize()
        print("shared expert tokens=%d calls=%d" % (M, calls))
    elif kind == "prefetch":
        M, on = int(args[0]), int(args[1])
        calls = int(args[2]) if len(args) > 2 else 3
        H = HIDDEN
        W = normal_bf16_cuda((H, H), WEIGHT_STD, "profile", "Wq")
        x = normal_bf16_cuda((M, H), 1.0, "profile", "xq", M)
        y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        half_l2 = torch.cuda.get_device_properties(0).L2_cache_size // 2
        for _ in range(calls):
            flush.fill_(1)                    # evicts L2
            if on:
                dg.l2_prefetch(W.data_ptr(), min(half_l2, W.numel() * 2))
            torch.cuda.synchronize()
            dg.dec_linear(x, W, y)
            torch.cuda.synchronize()
        print("prefetch M=%d on=%d calls=%d regime=%s" % (M, on, calls, dg.last_choice()))
    else:
        sys.exit(__doc__)
    if dg.sync_check() != 0:
        sys.exit("device status not clean")


if __name__ == "__main__":
    if len(sys.argv) >= 3 and sys.argv[1] == "case":
        case(*sys.argv[2:])
    elif len(sys.argv) == 3 and sys.argv[1] in ("launches", "raw"):
        {"launches": launches, "raw": raw}[sys.argv[1]](sys.argv[2])
    else:
        sys.exit(__doc__)
