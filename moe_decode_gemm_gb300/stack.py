"""The synthetic decode layer, composed from the library's C ABI.

One layer of the layer-stack workload (attention core excluded):
  [q | kv] = x·[Wq; Wkv]ᵀ          one fused projection (dec_linear)
  r        = bf16(x + q·Woᵀ)        o projection reading q in place from the
                                    fused output, residual fused (dec_linear_ex)
  x'       = bf16(r + MoE(r))       the MoE decode block with its shared expert
                                    and the residual fused (moe_decode_residual)
and, on a side stream, an L2 prefetch of the next layer's weights. The o
projection consuming q stands in for the attention output; kv is computed and
not consumed. The benchmark and the full-size parity tests both run this
function, so what is timed is what is checked.

Sources: "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 (projections),
§3 (MoE block, shared expert on its own stream) and §4 (prefetch of upcoming
weights on a side stream); "vLLM 宣布 Kimi K3 在 GB300 NVL72 上实现 batch 1 解码
842 tokens/s", the per-layer kernel trace (a layer as the unit of work).
"""
from __future__ import annotations

from . import dec_linear, l2_prefetch, moe_decode


def decode_layer(L, x, qkv, r, out, topk, idx=None, stream=None, prefetch=None):
    """Enqueue one decode layer on ``stream``; returns ``out``.

    L: weights with Wqkv [H+KV, H], Wo [H, H], Wr, W13, W2, Ws13, Ws2 (bf16,
    on the device). x [M, H] bf16 input; qkv [M, H+KV], r [M, H] and out
    [M, H] bf16 buffers the caller owns (out may alias x). idx: optional
    [M, topk] int32 for the chosen experts. prefetch: optional
    (side_stream, event, ptr, nbytes) -- the range is pulled into L2 on the
    side stream once the o projection has been enqueued.
    """
    H = x.shape[1]
    dec_linear(x, L.Wqkv, qkv, stream=stream)
    dec_linear(qkv[:, :H], L.Wo, r, stream=stream, residual=x)
    if prefetch is not None:
        side, ev, ptr, nbytes = prefetch
        ev.record(stream)
        side.wait_event(ev)
        l2_prefetch(ptr, nbytes, stream=side)
    moe_decode(r, L.Wr, L.W13, L.W2, L.Ws13, L.Ws2, topk, out=out, topk_idx=idx, stream=stream,
               residual=r)
    return out
