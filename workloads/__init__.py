"""Seeded synthetic input generators.

This module draws random numbers and encodes them as bf16; it holds none of
the arithmetic of the decode GEMM or the MoE block. It is the one module that
both the fp64 oracle's tests and the CUDA path's tests and benchmark use.

Two back ends:
  * CPU: numpy's Philox counter-based generator, deterministic on any host.
    Used for everything small (activations, router weights, test-size
    weights) so that the oracle and the GPU see identical bits.
  * CUDA: torch's Philox generator on the device, for the multi-GB expert
    banks and projection weights of the full-size workloads. The oracle gets
    those bits by copying the slices it needs to the host.

Every tensor has its own key: ``seed_for(base, name, layer, index, ...)``
hashes the parts, so any single expert of any layer can be regenerated alone.
"""
from __future__ import annotations

import hashlib
import math

import numpy as np

# ----------------------------------------------------------------- shapes
# Decode shapes of the MoE model the workloads describe.
HIDDEN = 7168
EXPERTS = 384
TOPK = 8
INTER = 2048
KV_WIDTH = 1024
WEIGHT_STD = 0.02
ROUTER_STD = 1.0 / math.sqrt(HIDDEN)  # makes the router logits ~N(0,1) for x ~N(0,1)


def seed_for(*parts) -> int:
    """Stable 63-bit seed from any tuple of str/int parts."""
    h = hashlib.blake2b(repr(tuple(parts)).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Encode float32 values as bf16 bit patterns, round to nearest even."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed_for(*key)))


def normal_bf16(shape, std, *key) -> np.ndarray:
    """bf16 bits of std * N(0,1) drawn in float32 (CPU, Philox)."""
    z = _rng(*key).standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(z * np.float32(std))


def integer_bf16(shape, lo, hi, *key) -> np.ndarray:
    """bf16 bits of integers uniform in [lo, hi] (exactly representable)."""
    z = _rng(*key).integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(z)


def one_hot_rows(N, K, *key):
    """W[n,:] = e_{perm[n]} with a random column per row; returns (bits, perm)."""
    perm = _rng(*key).integers(0, K, size=N)
    W = np.zeros((N, K), dtype=np.float32)
    W[np.arange(N), perm] = 1.0
    return f32_to_bf16_bits(W), perm


def router_scales(E, s) -> np.ndarray:
    """Per-expert scale of the router rows for a skewed-routing workload.

    Row e of the router is drawn with standard deviation ROUTER_STD * c_e,
    c_e = (e + 1)^-s normalised to mean 1: a token's score for expert e is
    then ~N(0, c_e^2), so low-index experts win the top-k far more often
    (popularity falls off roughly like a power law), tokens share experts and
    fewer distinct experts are read. s = 0 is the uniform workload.
    """
    c = (np.arange(E, dtype=np.float64) + 1.0) ** (-float(s))
    return c / c.mean()


def skewed_router_bf16(E, H, s, *key) -> np.ndarray:
    """[E, H] router weights of the skewed-routing workload, as bf16 bits."""
    c = router_scales(E, s)
    return np.stack([normal_bf16((H,), ROUTER_STD * c[e], *key, "row", e) for e in range(E)])


def token_rows(M, H, *key, attempts=None) -> np.ndarray:
    """x rows ~N(0,1) as bf16 bits; row m is drawn from key (+m, attempt).

    ``attempts[m]`` (default 0) selects a redraw of row m; callers that need a
    property of the rows (a gap between router scores, say) redraw a row by
    raising its attempt number.
    """
    att = [0] * M if attempts is None else list(attempts)
    rows = [normal_bf16((H,), 1.0, *key, "row", m, att[m]) for m in range(M)]
    return np.stack(rows) if rows else np.zeros((0, H), dtype=np.uint16)


# ----------------------------------------------------------------- CUDA side
def normal_bf16_cuda(shape, std, *key, device="cuda", out=None):
    """N(0, std) drawn on the device straight into a bf16 tensor.

    torch's normal_ on a bf16 tensor draws in float32, scales and rounds once
    to bf16, writing 2 bytes per element; it writes into ``out`` (a bf16
    tensor of ``shape``) when given.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed_for(*key))
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    out.normal_(0.0, float(std), generator=g)
    return out


def bits_to_torch(bits, device="cuda"):
    """uint16 bf16 bits (numpy) -> torch bf16 tensor on ``device``."""
    import torch

    b = np.ascontiguousarray(bits, dtype=np.uint16)
    t = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(device)


def torch_to_bits(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> uint16 bits on the host."""
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ----------------------------------------------------------------- layer stack
class LayerWeights:
    """Seeded weights of one synthetic decode layer, on the device.

    Wqkv [H + KV, H] holds Wq (rows 0..H-1) and Wkv (rows H..H+KV-1) as one
    matrix, so q and kv are one fused projection; Wq and Wkv are views of it.
    Wo [H, H]; router Wr [E, H] ~N(0, 1/sqrt(H)) (row e scaled by c_e for a
    skewed-routing workload, ``router_scales``); routed experts W13 [E, 2I, H]
    and W2 [E, H, I]; shared expert Ws13 [2I, H] and Ws2 [H, I]; all other
    weights ~N(0, 0.02).
    """

    def __init__(self, l, device="cuda", skew=0.0, H=HIDDEN, KV=KV_WIDTH, E=EXPERTS, I=INTER):
        import torch

        g = lambda shape, *key: normal_bf16_cuda(shape, WEIGHT_STD, "stack", l, *key,
                                                 device=device)
        self.Wqkv = torch.empty((H + KV, H), dtype=torch.bfloat16, device=device)
        normal_bf16_cuda((H, H), WEIGHT_STD, "stack", l, "Wq", device=device, out=self.Wqkv[:H])
        normal_bf16_cuda((KV, H), WEIGHT_STD, "stack", l, "Wkv", device=device,
                         out=self.Wqkv[H:])
        self.Wq, self.Wkv = self.Wqkv[:H], self.Wqkv[H:]
        self.Wo = g((H, H), "Wo")
        self.Wr = normal_bf16_cuda((E, H), ROUTER_STD, "stack", l, "Wr", device=device)
        if skew > 0:
            c = torch.tensor(router_scales(E, skew), dtype=torch.float32, device=device)
            self.Wr.copy_((self.Wr.float() * c[:, None]).to(torch.bfloat16))
        self.W13 = g((E, 2 * I, H), "W13")
        self.W2 = g((E, H, I), "W2")
        self.Ws13 = g((2 * I, H), "Ws13")
        self.Ws2 = g((H, I), "Ws2")
        self.H, self.KV, self.E, self.I = H, KV, E, I
