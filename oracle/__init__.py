"""Plain fp64 CPU oracle for the decode projection GEMM and the MoE decode block.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` import this package. The CUDA path
never imports it, and it imports nothing from the CUDA path: the two share
only the seeded input generators in ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C loops in double precision, one
function per definition). This module loads it with ctypes and composes the
MoE block and the decode layer from those functions with numpy float64.

Sources, all of them prose (the pages print no formula or worked example):
  * "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 "针对工作负载调优形状":
    projections y = x·Wᵀ, a small-matrix kernel at batch 1-2 and split-K at
    larger batch, both computing the same product.
  * same page, Part 1 §3 "改进 MoE 调度与重叠": router scoring, the routed
    experts, and a shared expert on its own stream whose output is added.
  * same page, Part 1 §4 "将即将使用的权重预取到缓存": weight prefetch (no
    arithmetic, so nothing here).
Shapes, dtypes, top-k with renormalised softmax gates and the SwiGLU expert
come from the workload definitions that accompany the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc and OpenMP."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _configure(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.orc_bf16_to_f64.restype = ctypes.c_double
    lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f64_array.argtypes = [P, I64, P]
    lib.orc_f64_to_bf16_bits.restype = ctypes.c_uint16
    lib.orc_f64_to_bf16_bits.argtypes = [ctypes.c_double]
    lib.orc_f64_to_bf16_array.argtypes = [P, I64, P]
    lib.orc_round_bf16.restype = ctypes.c_double
    lib.orc_round_bf16.argtypes = [ctypes.c_double]
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_linear.argtypes = [P, P, I64, I64, I64, P, P]
    lib.orc_linear_f64act.argtypes = [P, P, I64, I64, I64, P, P]
    lib.orc_linear_splitk.argtypes = [P, P, I64, I64, I64, I64, P]
    lib.orc_topk.restype = ctypes.c_int
    lib.orc_topk.argtypes = [P, I64, I64, I64, P, P]
    lib.orc_swiglu_hidden.argtypes = [P, P, I64, I64, I64, ctypes.c_int, P]
    lib.orc_silu.restype = ctypes.c_double
    lib.orc_silu.argtypes = [ctypes.c_double]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def swap_library(path):
    """Load another build of oracle.c in place of the default one and return
    the previous handle (or None). Used only by the mutation tests, which
    check that the pins reject deliberately broken copies of the oracle."""
    global _lib
    with _lock:
        old = _lib
        _lib = None if path is None else _configure(ctypes.CDLL(path))
    return old


def restore_library(handle):
    """Undo ``swap_library``."""
    global _lib
    with _lock:
        _lib = handle


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle's loops use."""
    return int(_load().orc_num_threads())


# ---------------------------------------------------------------- bf16 codec
def bf16_to_f64(bits) -> np.ndarray:
    """Exact decode of bf16 bit patterns."""
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_bf16_to_f64_array(_ptr(b), b.size, _ptr(out))
    return out


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round doubles to bf16 (nearest, ties to even); returns uint16 bits."""
    a = _f64(v)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_f64_to_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


def round_bf16(v) -> np.ndarray:
    """Round doubles to the nearest bf16 value, returned as doubles."""
    return bf16_to_f64(f64_to_bf16_bits(v))


def silu(z: float) -> float:
    """silu(z) = z / (1 + e^-z)."""
    return float(_load().orc_silu(float(z)))


# ---------------------------------------------------------------- GEMM
def linear(x_bits, W_bits):
    """y = x·Wᵀ in fp64 and its reference scale sum_k |x_k W_nk|.

    x_bits: [M,K] bf16 bits, W_bits: [N,K] bf16 bits -> (y, absref), [M,N] each.
    """
    x = _u16(x_bits)
    W = _u16(W_bits)
    M, K = x.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError("K mismatch")
    y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _load().orc_linear(_ptr(x), _ptr(W), M, N, K, _ptr(y), _ptr(A))
    return y, A


def linear_f64act(a, W_bits):
    """y = a·Wᵀ with fp64 activations a [M,K] and bf16 weights W [N,K]."""
    a = _f64(a)
    W = _u16(W_bits)
    M, K = a.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError("K mismatch")
    y = np.empty((M, N), dtype=np.float64)
    A = np.empty((M, N), dtype=np.float64)
    _load().orc_linear_f64act(_ptr(a), _ptr(W), M, N, K, _ptr(y), _ptr(A))
    return y, A


def linear_splitk(x_bits, W_bits, S: int):
    """Split-K form: S contiguous K chunks, partials summed s = 0..S-1."""
    x = _u16(x_bits)
    W = _u16(W_bits)
    M, K = x.shape
    N = W.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _load().orc_linear_splitk(_ptr(x), _ptr(W), M, N, K, int(S), _ptr(y))
    return y


# ---------------------------------------------------------------- routing
def topk(logits, k: int):
    """Full-sort top-k: (value desc, index asc); gates renormalised softmax.

    Returns (idx int32 [M,k], gates float64 [M,k]).
    """
    l = _f64(logits)
    M, E = l.shape
    idx = np.empty((M, k), dtype=np.int32)
    g = np.empty((M, k), dtype=np.float64)
    rc = _load().orc_topk(_ptr(l), M, E, int(k), _ptr(idx), _ptr(g))
    if rc != 0:
        raise ValueError("orc_topk failed (%d)" % rc)
    return idx, g


def sorted_gaps(logits, count: int) -> np.ndarray:
    """Adjacent gaps among the ``count`` largest logits of each row, [M, count-1]."""
    l = _f64(logits)
    top = -np.sort(-l, axis=1)[:, :count]
    return top[:, :-1] - top[:, 1:]


# ---------------------------------------------------------------- experts
def swiglu_hidden(x_bits, W13_bits, I: int, round_h: bool = False):
    """h = silu(x·W1ᵀ) * (x·W3ᵀ); W13 rows 0..I-1 = W1 (gate), I..2I-1 = W3 (up)."""
    x = _u16(x_bits)
    W13 = _u16(W13_bits)
    c, H = x.shape
    if W13.shape != (2 * I, H):
        raise ValueError("W13 must be [2I, H]")
    h = np.empty((c, I), dtype=np.float64)
    _load().orc_swiglu_hidden(_ptr(x), _ptr(W13), c, H, I, int(bool(round_h)), _ptr(h))
    return h


def expert_mlp(x_bits, W13_bits, W2_bits, I: int, round_h: bool = False):
    """One SwiGLU expert: o = h·W2ᵀ. Returns (o, absref) with absref_n = sum_i |h_i W2_ni|."""
    h = swiglu_hidden(x_bits, W13_bits, I, round_h)
    return linear_f64act(h, W2_bits)


def expert_mlp_f64act(a, W13_bits, W2_bits, I: int, round_h: bool = False):
    """One SwiGLU expert on fp64 activations a [c, L]: g = a·W1ᵀ, u = a·W3ᵀ,
    h = silu(g) * u with silu(z) = z / (1 + e^-z), o = h·W2ᵀ; the same
    definition as ``expert_mlp``, for an input that is not a bf16 tensor.
    Returns (o, absref) with absref_n = sum_i |h_i W2_ni|."""
    W13 = _u16(W13_bits)
    if W13.shape[0] != 2 * I:
        raise ValueError("W13 must be [2I, L]")
    g, _ = linear_f64act(a, W13[:I])
    u, _ = linear_f64act(a, W13[I:])
    h = g / (1.0 + np.exp(-g)) * u
    if round_h:
        h = round_bf16(h)
    return linear_f64act(h, W2_bits)


def gates_for(logits, idx) -> np.ndarray:
    """Renormalised softmax gates of a given choice of experts, in fp64:
    g[m,j] = exp(l[m,idx[m,j]] - l_max) / sum_j' exp(l[m,idx[m,j']] - l_max),
    l_max the largest chosen score of token m (the same closed form the top-k
    routine returns for its own choice)."""
    l = _f64(logits)
    idx = np.asarray(idx)
    chosen = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    w = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    return w / w.sum(axis=1, keepdims=True)


def _routed_sum(rows_in, rows, idx, gates, fetch_expert, topk_k: int, I: int, round_h: bool):
    """acc[r] = sum_{j=0..k-1} g[m,j] * expert_{idx[m,j]}(rows_in[m]) for m = rows[r],
    summed in the order j = 0..k-1, and accabs[r] = sum_j g[m,j] * absref of
    that expert's output. rows_in: bf16 bits, or fp64 activations. Only the
    experts the given rows chose are fetched."""
    width = None
    o, oabs = {}, {}
    needed = sorted(set(int(e) for m in rows for e in idx[m]))
    for e in needed:
        W13_e, W2_e = fetch_expert(e)
        pairs = [(m, j) for m in rows for j in range(topk_k) if idx[m, j] == e]
        xs = rows_in[[m for m, _ in pairs]]
        if xs.dtype == np.uint16:
            oe, ae = expert_mlp(xs, W13_e, W2_e, I, round_h)
        else:
            oe, ae = expert_mlp_f64act(xs, W13_e, W2_e, I, round_h)
        width = oe.shape[1]
        for r, (m, j) in enumerate(pairs):
            o[(m, j)] = oe[r]
            oabs[(m, j)] = ae[r]
    acc = np.zeros((len(rows), width or 0))
    accabs = np.zeros((len(rows), width or 0))
    for r, m in enumerate(rows):
        a = np.zeros(width)
        aa = np.zeros(width)
        for j in range(topk_k):
            a = a + gates[m, j] * o[(m, j)]
            aa = aa + gates[m, j] * oabs[(m, j)]
        acc[r] = a
        accabs[r] = aa
    return acc, accabs


def _route(logits, topk_k, route):
    if route is None:
        return topk(logits, topk_k)
    idx = np.ascontiguousarray(route, dtype=np.int32)
    if idx.shape != (logits.shape[0], topk_k) or idx.min() < 0 or idx.max() >= logits.shape[1]:
        raise ValueError("route must be [M, k] expert indices")
    return idx, gates_for(logits, idx)


def moe(x_bits, Wr_bits, fetch_expert, topk_k: int, I: int, shared=None,
        round_h: bool = False, tokens=None, route=None):
    """MoE decode block, "vLLM 如何用智能体辅助优化 Kimi K3 解码性能" Part 1 §3.

    logits = x·Wrᵀ (fp64); (idx, g) = top-k with renormalised softmax gates;
    out[m] = sum_{j=0..k-1} g[m,j] * expert_{idx[m,j]}(x[m]) + shared(x[m]),
    the sum taken in the order j = 0..k-1, then the shared term.

    fetch_expert(e) -> (W13_e [2I,H] bits, W2_e [H,I] bits); only the experts
    that the oracle itself selects are fetched. shared is (Ws13, Ws2) or None.
    tokens: optional list of token rows to compute (the others stay NaN).
    route: optional [M,k] choice of experts to use instead of the oracle's own
    top-k (gates from ``gates_for`` on the oracle's scores). Where two scores
    are closer than fp32 can separate, an implementation that scores in fp32
    may legitimately choose the other expert; its output is then checked for
    the choice it made.

    Returns dict(out, absref, idx, gates, logits), where
    absref[m,n] = sum_j g_j sum_i |h_ji W2[e_j,n,i]| + sum_i |hs_i Ws2[n,i]|.
    """
    x = _u16(x_bits)
    M, H = x.shape
    logits, _ = linear(x, Wr_bits)
    idx, gates = _route(logits, topk_k, route)
    rows = list(range(M)) if tokens is None else sorted(set(int(t) for t in tokens))
    acc, accabs = _routed_sum(x, rows, idx, gates, fetch_expert, topk_k, I, round_h)
    out = np.full((M, H), np.nan)
    absref = np.full((M, H), np.nan)
    if shared is not None:
        Ws13, Ws2 = shared
        s, sabs = expert_mlp(x[rows], Ws13, Ws2, I, round_h)
        acc = acc + s
        accabs = accabs + sabs
    out[rows] = acc
    absref[rows] = accabs
    return dict(out=out, absref=absref, idx=idx, gates=gates, logits=logits)


def moe_latent(x_bits, Wrl_bits, E: int, fetch_expert, topk_k: int, I: int, Wup_bits,
               shared=None, round_inter: bool = False, tokens=None, route=None):
    """MoE decode block whose routed experts work on a latent width L.

    "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §3: the router scores and
    the latent input projection are computed as one matrix product. The
    reading taken here (the pages name the two projections and nothing else):
      sc     = x·Wrlᵀ in fp64, Wrl [E + L, H] = the router's E rows stacked on
               the latent input projection's L rows;
      logits = sc[:, :E] (the router scores);
      lat    = sc[:, E:] (the latent input);
      (idx, g) = top-k of logits with renormalised softmax gates;
      z      = sum_{j=0..k-1} g_j * expert_{idx_j}(lat) -- experts map
               L -> I -> L (W13_e [2I, L], W2_e [L, I]);
      out    = z·Wupᵀ + shared(x), Wup [H, L] the up-projection back to the
               hidden width, the shared expert on x as in ``moe``.
    Everything stays in fp64, as in the plain block: an implementation rounds
    lat, h and z to bf16 where they become a product's operand, and the
    tolerance absorbs those roundings. round_inter rounds lat and z to bf16
    here too (a diagnostic, to tell rounding-point effects from bugs).
    Returns dict(out, absref, idx, gates, logits, lat, z), with the reference
    scale carried through the block's linear steps after the experts:
      absref[m,n] = sum_l |Wup[n,l]| * Az[m,l] + sum_i |hs_i Ws2[n,i]|,
      Az[m,l]     = sum_j g_j sum_i |h_ji W2[e_j,l,i]|
    (the plain block's scale, in the latent space, expanded through the
    up-projection: every product of the expression taken in absolute value).
    lat and z are fp64 ([M, L], rows not computed are NaN in z).
    """
    x = _u16(x_bits)
    Wrl = _u16(Wrl_bits)
    M, H = x.shape
    L = Wrl.shape[0] - E
    if L < 1:
        raise ValueError("Wrl must stack E router rows on L >= 1 latent rows")
    sc, _ = linear(x, Wrl)
    logits = np.ascontiguousarray(sc[:, :E])
    lat = np.ascontiguousarray(sc[:, E:])
    if round_inter:
        lat = round_bf16(lat)
    idx, gates = _route(logits, topk_k, route)
    rows = list(range(M)) if tokens is None else sorted(set(int(t) for t in tokens))
    acc, acc_abs = _routed_sum(lat, rows, idx, gates, fetch_expert, topk_k, I, round_inter)
    if round_inter:
        acc = round_bf16(acc)
    z = np.full((M, L), np.nan)
    z[rows] = acc
    u, _ = linear_f64act(acc, Wup_bits)
    Wup_abs = _u16(Wup_bits) & np.uint16(0x7FFF)       # |w| of a bf16 value: its sign bit cleared
    uabs, _ = linear_f64act(acc_abs, Wup_abs)
    out = np.full((M, H), np.nan)
    absref = np.full((M, H), np.nan)
    if shared is not None:
        Ws13, Ws2 = shared
        s, sabs = expert_mlp(x[rows], Ws13, Ws2, I, round_inter)
        u = u + s
        uabs = uabs + sabs
    out[rows] = u
    absref[rows] = uabs
    return dict(out=out, absref=absref, idx=idx, gates=gates, logits=logits, lat=lat, z=z)


def residual(x_bits, f, f_absref):
    """Residual add r = x + f in fp64, with reference scale |x| + absref(f)."""
    xv = bf16_to_f64(x_bits)
    return xv + f, np.abs(xv) + f_absref


def decoder_layer(x_bits, Wq, Wkv, Wo, Wr, fetch_expert, topk_k, I, shared,
                  round_h: bool = False):
    """One synthetic decode layer as a composition of the library's operations.

    Each operation's result is rounded to bf16 where the operation's interface
    hands bf16 to the next one:
      q  = bf16(x·Wqᵀ);  kv = bf16(x·Wkvᵀ)  (computed, unused: attention excluded)
      r  = bf16(x + q·Woᵀ)                  (o-proj stands in for attention output)
      x' = bf16(r + moe(r))
    Returns dict with bf16 bits and fp64 values/scales of q, kv, r, x', plus
    the MoE routing of r.
    """
    qv, qA = linear(x_bits, Wq)
    q = f64_to_bf16_bits(qv)
    kvv, kvA = linear(x_bits, Wkv)
    kv = f64_to_bf16_bits(kvv)
    ov, oA = linear(q, Wo)
    rv, rA = residual(x_bits, ov, oA)
    r = f64_to_bf16_bits(rv)
    mo = moe(r, Wr, fetch_expert, topk_k, I, shared, round_h)
    xv, xA = residual(r, mo["out"], mo["absref"])
    xn = f64_to_bf16_bits(xv)
    return dict(q=q, q_val=qv, q_abs=qA, kv=kv, kv_val=kvv, kv_abs=kvA,
                r=r, r_val=rv, r_abs=rA, out=xn, out_val=xv, out_abs=xA,
                idx=mo["idx"], gates=mo["gates"], logits=mo["logits"])
