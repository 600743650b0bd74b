"""GB300-native decode projection GEMM + MoE decode block.

Thin ctypes binding over ``libdecgemm.so`` (the C ABI in include/decgemm.h).
The functions below only marshal arguments: torch tensors give device
pointers and sizes, the current torch stream gives the CUDA stream. Every
step of the computation runs in the library's CUDA kernels; there is no
fallback path. If the library is missing, importing the binding's functions
raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdecgemm.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libdecgemm_debug.so")

DEC_OK = 0
DEC_EINVAL = -1
DEC_EUNSUPPORTED = -2
DEC_ECUDA = -3
DEC_ETIMEOUT = -4
DEC_ENOMEM = -5
DEC_ENODEV = -6
DEC_EBOUNDS = -7

REGIME_NONE, REGIME_SMALLM, REGIME_MMA, REGIME_TC = 0, 1, 2, 3
REGIME_NAMES = {0: "none", 1: "smallm", 2: "mma", 3: "tc"}

# Names the header declares; the ABI tests check every one is exported.
EXPORTS = [
    "dec_linear", "dec_linear_residual", "dec_linear_ex", "dec_linear_splitk", "moe_decode",
    "moe_decode_residual", "moe_decode_latent", "l2_prefetch", "dec_add", "dec_last_choice", "dec_last_grid",
    "dec_strerror", "dec_sync_check", "dec_set_wait_timeout_ns", "dec_selftest_timeout",
    "dec_launch_count", "dec_probe_begin", "dec_probe_end", "dec_shutdown", "dec_version",
    "dec_linear_noalloc", "dec_debug_build", "dec_debug_check_site",
]

_lib = None


class DecError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, strerror(code), code))


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run `python -m moe_decode_gemm_gb300.build` "
                           "(no fallback exists)" % os.path.basename(path))
    return _configure(ctypes.CDLL(path))


def lib():
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


def use_library(path):
    """Route every call of this binding to another build of the library (the
    index-checking one, DEBUG_LIB_PATH) and return the previous handle; give
    the handle back to restore it."""
    global _lib
    old = _lib
    _lib = path if not isinstance(path, str) else _load(path)
    return old


def _configure(L):
    """Declare the C signatures of every exported function on a loaded library."""
    P, I, SZ, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
    sig = {
        "dec_linear": (I, [P, P, P, I, I, I, P]),
        "dec_linear_residual": (I, [P, P, P, P, I, I, I, P]),
        "dec_linear_ex": (I, [P, I, P, P, P, I, I, I, P]),
        "dec_linear_splitk": (I, [P, P, P, I, I, I, I, P]),
        "moe_decode": (I, [P, P, P, P, P, P, P, I, I, I, I, I, P, P, P]),
        "moe_decode_residual": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P]),
        "moe_decode_latent": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]),
        "l2_prefetch": (I, [P, SZ, P]),
        "dec_add": (I, [P, P, P, SZ, P]),
        "dec_last_choice": (I, []),
        "dec_last_grid": (I, []),
        "dec_strerror": (ctypes.c_char_p, [I]),
        "dec_sync_check": (I, [P]),
        "dec_set_wait_timeout_ns": (LL, [LL]),
        "dec_selftest_timeout": (I, [LL, P]),
        "dec_launch_count": (LL, []),
        "dec_probe_begin": (I, [I, I]),
        "dec_probe_end": (I, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
        "dec_shutdown": (None, []),
        "dec_version": (I, []),
        "dec_linear_noalloc": (I, [P, P, P, I, I, I, P]),
        "dec_debug_build": (I, []),
        "dec_debug_check_site": (I, [ctypes.POINTER(ctypes.c_int),
                                     ctypes.POINTER(ctypes.c_longlong)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def check_site():
    """(line, index) of the first failed index check of the debug build, as
    read by the last sync_check that returned DEC_EBOUNDS, or None."""
    line, idx = ctypes.c_int(0), ctypes.c_longlong(0)
    if lib().dec_debug_check_site(ctypes.byref(line), ctypes.byref(idx)):
        return line.value, idx.value
    return None


def strerror(code: int) -> str:
    return lib().dec_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != DEC_OK:
        raise DecError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, shape=None, dtype="bf16", contiguous=True):
    """Reject a tensor the C ABI would misread: the ABI sees only pointers
    and sizes, so dtype, shape and layout are checked here (the device by
    ``_on_one_gpu`` once every operand has passed)."""
    import torch

    want = {"bf16": torch.bfloat16, "i32": torch.int32, "f32": torch.float32}[dtype]
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s: expected a torch tensor, got %s" % (name, type(t).__name__))
    if t.dtype != want:
        raise TypeError("%s: expected %s, got %s" % (name, want, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s: expected shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if contiguous and not t.is_contiguous():
        raise ValueError("%s: must be contiguous (row-major)" % name)
    return t


def _on_one_gpu(**tensors):
    """Every given tensor (None entries skipped) lives on one CUDA device."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError("%s: expected a CUDA tensor, got one on %s" % (name, t.device))
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("%s: on %s, the other operands on %s" % (name, t.device, dev))


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------- the hot path
def dec_linear(x, W, y=None, stream=None, residual=None):
    """y = x·Wᵀ (bf16), or y = residual + x·Wᵀ when ``residual`` is given.

    x: [M,K] bf16 with unit column stride; its rows may be further apart than
    K (a column slice of a wider tensor, read in place through dec_linear_ex).
    W: [N,K] bf16, y: [M,N] bf16 (allocated if None).
    """
    import torch

    _need(x, "x", contiguous=False)
    if x.dim() != 2:
        raise ValueError("x: expected [M, K], got shape %s" % (tuple(x.shape),))
    M, K = x.shape
    _need(W, "W")
    if W.dim() != 2 or W.shape[1] != K:
        raise ValueError("W: expected [N, %d], got shape %s" % (K, tuple(W.shape)))
    N = W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", shape=(M, N))
    if residual is not None:
        _need(residual, "residual", shape=(M, N))
    ldx = x.stride(0) if M > 1 else K
    if x.stride(1) != 1:
        raise ValueError("dec_linear: x needs unit column stride")
    _on_one_gpu(x=x, W=W, y=y, residual=residual)
    if ldx != K:
        rc = lib().dec_linear_ex(_ptr(x), ldx, _ptr(W), _ptr(residual), _ptr(y), M, N, K,
                                 _stream(stream))
    elif residual is None:
        rc = lib().dec_linear(_ptr(x), _ptr(W), _ptr(y), M, N, K, _stream(stream))
    else:
        rc = lib().dec_linear_residual(_ptr(x), _ptr(W), _ptr(residual), _ptr(y), M, N, K,
                                       _stream(stream))
    _check(rc, "dec_linear")
    return y


def dec_linear_noalloc(x, W, y, stream=None):
    """dec_linear that allocates nothing: its split-K scratch is a fixed array
    inside the library (for callers that cannot allocate device memory).
    ``y`` must be given. Calls that may overlap on the GPU race."""
    _need(x, "x")
    M, K = x.shape
    _need(W, "W")
    if W.dim() != 2 or W.shape[1] != K:
        raise ValueError("W: expected [N, %d], got shape %s" % (K, tuple(W.shape)))
    N = W.shape[0]
    _need(y, "y", shape=(M, N))
    _on_one_gpu(x=x, W=W, y=y)
    _check(lib().dec_linear_noalloc(_ptr(x), _ptr(W), _ptr(y), M, N, K, _stream(stream)),
           "dec_linear_noalloc")
    return y


def dec_linear_splitk(x, W, S, y=None, stream=None):
    """dec_linear with the split factor forced to S (test/tuning hook)."""
    import torch

    _need(x, "x")
    M, K = x.shape
    _need(W, "W")
    if W.dim() != 2 or W.shape[1] != K:
        raise ValueError("W: expected [N, %d], got shape %s" % (K, tuple(W.shape)))
    N = W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", shape=(M, N))
    _on_one_gpu(x=x, W=W, y=y)
    _check(lib().dec_linear_splitk(_ptr(x), _ptr(W), _ptr(y), M, N, K, int(S), _stream(stream)),
           "dec_linear_splitk")
    return y


def moe_decode(x, Wr, W13, W2, Ws13, Ws2, topk, out=None, topk_idx=None, topk_w=None,
               stream=None, residual=None):
    """MoE decode block. Shapes: x [M,H], Wr [E,H], W13 [E,2I,H], W2 [E,H,I],
    Ws13 [2I,H] / Ws2 [H,I] or both None. Returns out [M,H] bf16 (plus the
    residual when given)."""
    import torch

    _need(x, "x")
    if x.dim() != 2:
        raise ValueError("x: expected [M, H], got shape %s" % (tuple(x.shape),))
    M, H = x.shape
    _need(Wr, "Wr")
    if Wr.dim() != 2 or Wr.shape[1] != H:
        raise ValueError("Wr: expected [E, %d], got shape %s" % (H, tuple(Wr.shape)))
    E = Wr.shape[0]
    _need(W13, "W13")
    if W13.dim() != 3 or W13.shape[0] != E or W13.shape[2] != H or W13.shape[1] % 2:
        raise ValueError("W13: expected [%d, 2I, %d], got shape %s" % (E, H, tuple(W13.shape)))
    I = W13.shape[1] // 2
    _need(W2, "W2", shape=(E, H, I))
    if (Ws13 is None) != (Ws2 is None):
        raise ValueError("Ws13 and Ws2: give both or neither")
    if Ws13 is not None:
        _need(Ws13, "Ws13", shape=(2 * I, H))
        _need(Ws2, "Ws2", shape=(H, I))
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", shape=(M, H))
    if residual is not None:
        _need(residual, "residual", shape=(M, H))
    if topk_idx is not None:
        _need(topk_idx, "topk_idx", shape=(M, int(topk)), dtype="i32")
    if topk_w is not None:
        _need(topk_w, "topk_w", shape=(M, int(topk)), dtype="f32")
    _on_one_gpu(x=x, Wr=Wr, W13=W13, W2=W2, Ws13=Ws13, Ws2=Ws2, out=out, residual=residual,
                topk_idx=topk_idx, topk_w=topk_w)
    args = [_ptr(x), _ptr(Wr), _ptr(W13), _ptr(W2), _ptr(Ws13), _ptr(Ws2)]
    tail = [M, H, E, int(topk), I, _ptr(topk_idx), _ptr(topk_w), _stream(stream)]
    if residual is None:
        rc = lib().moe_decode(*args, _ptr(out), *tail)
    else:
        rc = lib().moe_decode_residual(*args, _ptr(residual), _ptr(out), *tail)
    _check(rc, "moe_decode")
    return out


def moe_decode_latent(x, Wrl, W13, W2, Wup, Ws13, Ws2, topk, out=None, topk_idx=None,
                      topk_w=None, stream=None, residual=None):
    """MoE block with the routed experts on a latent width L. Shapes: x [M,H],
    Wrl [E+L,H] (router rows, then the latent input projection), W13 [E,2I,L],
    W2 [E,L,I], Wup [H,L], Ws13 [2I,H] / Ws2 [H,I] or both None. Returns out
    [M,H] bf16 (plus the residual when given)."""
    import torch

    _need(x, "x")
    if x.dim() != 2:
        raise ValueError("x: expected [M, H], got shape %s" % (tuple(x.shape),))
    M, H = x.shape
    _need(W13, "W13")
    if W13.dim() != 3 or W13.shape[1] % 2:
        raise ValueError("W13: expected [E, 2I, L], got shape %s" % (tuple(W13.shape),))
    E, I, L = W13.shape[0], W13.shape[1] // 2, W13.shape[2]
    _need(Wrl, "Wrl", shape=(E + L, H))
    _need(W2, "W2", shape=(E, L, I))
    _need(Wup, "Wup", shape=(H, L))
    if (Ws13 is None) != (Ws2 is None):
        raise ValueError("Ws13 and Ws2: give both or neither")
    if Ws13 is not None:
        _need(Ws13, "Ws13", shape=(2 * I, H))
        _need(Ws2, "Ws2", shape=(H, I))
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", shape=(M, H))
    if residual is not None:
        _need(residual, "residual", shape=(M, H))
    if topk_idx is not None:
        _need(topk_idx, "topk_idx", shape=(M, int(topk)), dtype="i32")
    if topk_w is not None:
        _need(topk_w, "topk_w", shape=(M, int(topk)), dtype="f32")
    _on_one_gpu(x=x, Wrl=Wrl, W13=W13, W2=W2, Wup=Wup, Ws13=Ws13, Ws2=Ws2, out=out,
                residual=residual, topk_idx=topk_idx, topk_w=topk_w)
    rc = lib().moe_decode_latent(_ptr(x), _ptr(Wrl), _ptr(W13), _ptr(W2), _ptr(Wup), _ptr(Ws13),
                                 _ptr(Ws2), _ptr(residual), _ptr(out), M, H, L, E, int(topk), I,
                                 _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(rc, "moe_decode_latent")
    return out


def l2_prefetch(t_or_ptr, nbytes=None, stream=None):
    """Warm L2 with a tensor's bytes (or a raw device pointer and byte count)."""
    if nbytes is None:
        if t_or_ptr.device.type != "cuda":
            raise ValueError("l2_prefetch: expected a CUDA tensor")
        ptr, nbytes = t_or_ptr.data_ptr(), t_or_ptr.numel() * t_or_ptr.element_size()
    else:
        ptr = int(t_or_ptr)
    _check(lib().l2_prefetch(ctypes.c_void_p(ptr), int(nbytes), _stream(stream)), "l2_prefetch")


def dec_add(a, b, out=None, stream=None):
    """out = bf16(a + b) elementwise."""
    import torch

    _need(a, "a")
    _need(b, "b", shape=a.shape)
    if out is None:
        out = torch.empty_like(a)
    _need(out, "out", shape=a.shape)
    _on_one_gpu(a=a, b=b, out=out)
    _check(lib().dec_add(_ptr(a), _ptr(b), _ptr(out), a.numel(), _stream(stream)), "dec_add")
    return out


# ---------------------------------------------------------------- introspection
def last_choice():
    """(regime name, split factor) of this thread's last projection call."""
    v = lib().dec_last_choice()
    return REGIME_NAMES.get(v & 0xFF, "?"), (v >> 8) & 0xFF


def last_cluster() -> bool:
    """Whether this thread's last projection call used the cluster split."""
    return bool((lib().dec_last_choice() >> 16) & 1)


def last_wide() -> bool:
    """Whether this thread's last projection call used 256-row output tiles."""
    return bool((lib().dec_last_choice() >> 17) & 1)


def last_slab() -> bool:
    """Whether this thread's last projection call gave each CTA whole weight
    rows (1-16 tokens, no split over K)."""
    return bool((lib().dec_last_choice() >> 18) & 1)


def last_grid() -> int:
    return lib().dec_last_grid()


def sync_check(stream=None) -> int:
    return lib().dec_sync_check(_stream(stream))


def set_wait_timeout_ns(ns: int) -> int:
    return lib().dec_set_wait_timeout_ns(int(ns))


def selftest_timeout(ns: int, stream=None):
    _check(lib().dec_selftest_timeout(int(ns), _stream(stream)), "dec_selftest_timeout")


def launch_count() -> int:
    return lib().dec_launch_count()


def probe_begin(kind: int, capacity: int):
    _check(lib().dec_probe_begin(int(kind), int(capacity)), "dec_probe_begin")


def probe_end():
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int(0)
    _check(lib().dec_probe_end(ctypes.byref(ms), ctypes.byref(n)), "dec_probe_end")
    return ms.value, n.value


def shutdown():
    lib().dec_shutdown()


PROBE_EXPERT_W13, PROBE_EXPERT_W2, PROBE_LINEAR, PROBE_ROUTER, PROBE_COMBINE = 0, 1, 2, 3, 4
