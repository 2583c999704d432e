"""Work accounting for the throughput metrics (FLOPs and algorithmic bytes).

Prefill FLOPs follow the convention the gpu-inference blog (section 02, "Why
there is no throughput table here") spells out: full attention costs
4*b*h*n^2*d FLOPs (two matmuls of 2*n^2*d each per head) and causal attention
is credited half of that.  The inference-kernel-cookbook README's recipe 01
output (N=2048, d=64: 12.28 ms -> 0.087 TFLOPS, 996.18 ms -> 0.001 TFLOPS)
is consistent with 4*N^2*d, which the tests check.

Algorithmic bytes count every input read once and every output written once.
"""
from __future__ import annotations


def prefill_flops(B: int, H: int, Nq: int, Nkv: int, d: int, causal: bool) -> float:
    """Metric FLOPs: 4*B*H*Nq*Nkv*d, halved when causal."""
    f = 4.0 * B * H * Nq * Nkv * d
    return f / 2.0 if causal else f


def backward_flops(B: int, H: int, Nq: int, Nkv: int, d: int, causal: bool) -> float:
    """Backward FLOPs by the usual accounting: five Nq x Nkv x d products (S, dP, dV, dK, dQ)
    against the forward's two, i.e. 2.5 x prefill_flops.  The dQ kernel recomputes S and dP,
    so the tensor cores execute 3.5 x prefill_flops (backward_flops_executed)."""
    return 2.5 * prefill_flops(B, H, Nq, Nkv, d, causal)


def backward_flops_executed(B: int, H: int, Nq: int, Nkv: int, d: int, causal: bool) -> float:
    return 3.5 * prefill_flops(B, H, Nq, Nkv, d, causal)


def prefill_flops_kvlen(H: int, Nq: int, d: int, kv_lens) -> float:
    """FLOPs actually required with key padding: 4*H*Nq*d*sum_b(kv_len_b) (non-causal)."""
    return 4.0 * H * Nq * d * float(sum(int(x) for x in kv_lens))


def prefill_bytes(B: int, H: int, Nq: int, Nkv: int, d: int, elem: int = 2, lse: bool = True,
                  kv_lens=None) -> float:
    """Q and O once, K and V once (only the valid prefix when key lengths are given), LSE fp32."""
    qo = 2.0 * B * H * Nq * d * elem
    if kv_lens is None:
        kv = 2.0 * B * H * Nkv * d * elem
    else:
        kv = 2.0 * H * d * elem * float(sum(min(int(x), Nkv) for x in kv_lens))
    return qo + kv + (4.0 * B * H * Nq if lse else 0.0)


def decode_bytes(H: int, d: int, ctx_lens, page_size: int, elem: int = 2, lse: bool = True,
                 kv_heads: int | None = None, kv_elem: int | None = None) -> float:
    """K and V of every cached token once (kv_heads cache heads, default H; kv_elem bytes per
    cached element, default elem: 1 for an e4m3 cache), q and o once (elem bytes), LSE fp32,
    page-table entries used."""
    ctx = [int(x) for x in ctx_lens]
    B = len(ctx)
    Hkv = H if kv_heads is None else kv_heads
    kv = 2.0 * Hkv * d * (elem if kv_elem is None else kv_elem) * float(sum(ctx))
    qo = 2.0 * B * H * d * elem
    pt = 4.0 * float(sum(-(-c // page_size) for c in ctx))
    return kv + qo + pt + (4.0 * B * H if lse else 0.0)


def paged_prefill_bytes(H: int, Nq: int, d: int, ctx_lens, page_size: int, kv_heads: int | None = None,
                        elem: int = 2, lse: bool = True) -> float:
    """Chunked prefill over the paged cache: K and V of every cached token once (kv_heads cache
    heads, default H), the Nq queries and their outputs once, LSE fp32, page-table entries used."""
    ctx = [int(x) for x in ctx_lens]
    B = len(ctx)
    Hkv = H if kv_heads is None else kv_heads
    kv = 2.0 * Hkv * d * elem * float(sum(ctx))
    qo = 2.0 * B * H * Nq * d * elem
    pt = 4.0 * float(sum(-(-c // page_size) for c in ctx))
    return kv + qo + pt + (4.0 * B * H * Nq if lse else 0.0)


def paged_prefill_flops(H: int, Nq: int, d: int, ctx_lens, causal: bool = True) -> float:
    """FLOPs of a chunked prefill whose Nq queries are the last Nq of ctx_b cached tokens:
    4*d per (query, visible key); with the bottom-right causal mask query i sees
    ctx_b - Nq + i + 1 keys, else ctx_b."""
    total = 0.0
    for c in (int(x) for x in ctx_lens):
        if causal:
            # sum over i of (c - Nq + i + 1), counting only positive terms
            first = c - Nq + 1
            keys = sum(max(0, first + i) for i in range(Nq))
        else:
            keys = Nq * c
        total += 4.0 * H * d * keys
    return total
