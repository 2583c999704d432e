"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws random tensors with a
torch CPU generator and lays them out.  Both the CUDA path and the fp64 oracle
consume what it returns, so neither depends on the other.

Recipe (all draws from ``torch.Generator().manual_seed(seed)``, in this order):
  prefill: q, k, v = randn(shape, fp32) * value_scale  -> bf16 (round to nearest even);
           kv_lens  = randint(lo, hi + 1, (B,)) if a key-padding range is given.
  decode:  ctx_lens = randint(lo, hi + 1, (B,));
           q        = randn(B, H, d) -> bf16;
           pages    = randperm(total pages used) gives each logical page a physical slot;
           k, v     = randn(num_pages, H, page_size, d) -> bf16;
           one extra "poison" page (every element 3.0e4) is the target of every unused
           page-table slot, and the unused tail slots of each sequence's last page hold
           the same value, so an over-read changes the result instead of faulting.

The named workloads follow the benchmark shapes: a single 128x64 tile, a
BERT-large-like encoder with key padding, a GPT-2-small-like causal decoder, a
long-context causal head-dim-128 case, and paged decode over 16-token pages.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    H: int
    Nq: int
    Nkv: int
    d: int
    causal: bool
    value_scale: float = 1.0
    kv_len_range: tuple[int, int] | None = None  # inclusive [lo, hi]; None = all keys valid
    seed: int = 0
    softmax_scale: float | None = None  # None = 1/sqrt(d)
    kv_heads: int | None = None  # None = H (multi-head); fewer = grouped-query attention

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def Hkv(self) -> int:
        return self.H if self.kv_heads is None else self.kv_heads


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    H: int
    d: int
    ctx_range: tuple[int, int]  # inclusive [lo, hi]
    page_size: int = 16
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def max_pages(self) -> int:
        return -(-self.ctx_range[1] // self.page_size)


# The five benchmark workloads (seed 1000 + k for the k-th).
TILE_128x64 = PrefillShape("single-tile B1 H1 N128 d64 non-causal", 1, 1, 128, 128, 64, False, seed=1001)
ENCODER_PAD = PrefillShape("encoder B8 H16 N512 d64 non-causal key-padding U[256,512]",
                           8, 16, 512, 512, 64, False, kv_len_range=(256, 512), seed=1002)
DECODER_CAUSAL = PrefillShape("causal decoder B8 H12 N1024 d64", 8, 12, 1024, 1024, 64, True, seed=1003)
LONG_CAUSAL = PrefillShape("long-context causal B2 H32 N8192 d128 inputs x0.5",
                           2, 32, 8192, 8192, 128, True, value_scale=0.5, seed=1004)
PAGED_DECODE = DecodeShape("paged decode B32 H32 d128 ctx U[512,8192] page16",
                           32, 32, 128, (512, 8192), 16, seed=1005)

# Grouped-query paged decode (32 query heads over 8 cache heads) on the same lengths.
PAGED_DECODE_GQA = DecodeShape("paged decode GQA B32 Hq32 Hkv8 d128 ctx U[512,8192] page16",
                               32, 32, 128, (512, 8192), 16, seed=1007)
PAGED_DECODE_GQA_KV_HEADS = 8

# Chunked prefill over the paged cache: 1024 new tokens per sequence on top of a cache of
# 1024..8192 tokens (the chunk included), 32 query heads over 8 cache heads.
PAGED_PREFILL = DecodeShape("chunked prefill B8 Hq32 Hkv8 d128 Nq1024 ctx U[1024,8192] page16",
                            8, 32, 128, (1024, 8192), 16, seed=1008)
PAGED_PREFILL_KV_HEADS = 8
PAGED_PREFILL_NQ = 1024
# The same chunked prefill at the other head dims (same seed: the same context lengths and table).
PAGED_PREFILL_BY_DIM = {d: DecodeShape(f"chunked prefill B8 Hq32 Hkv8 d{d} Nq1024 ctx U[1024,8192] page16",
                                       8, 32, d, (1024, 8192), 16, seed=1008) for d in (32, 64, 80, 96)}

# The paged decode at the other head dims the Kernel-Inference-Engine README instantiates (same
# seed, so the same context lengths and page table as the d = 128 workload).
PAGED_DECODE_BY_DIM = {d: DecodeShape(f"paged decode B32 H32 d{d} ctx U[512,8192] page16", 32, 32, d, (512, 8192), 16,
                                      seed=1005) for d in (32, 64, 80, 96)}

# A quarter-size paged decode (same lengths distribution) for multi-pass profiler captures.
PAGED_DECODE_SMALL = DecodeShape("paged decode B8 H32 d128 ctx U[512,8192] page16",
                                 8, 32, 128, (512, 8192), 16, seed=1006)

PREFILL_WORKLOADS = (TILE_128x64, ENCODER_PAD, DECODER_CAUSAL, LONG_CAUSAL)


def prefill_inputs(shape: PrefillShape):
    """Return dict(q, k, v, kv_lens) as CPU tensors (bf16 / int32 or None).
    K and V have shape.kv_heads heads (grouped-query attention) when it is set."""
    g = torch.Generator().manual_seed(shape.seed)
    B, H, Nq, Nkv, d = shape.B, shape.H, shape.Nq, shape.Nkv, shape.d
    Hkv = shape.Hkv
    q = (torch.randn(B, H, Nq, d, generator=g) * shape.value_scale).to(torch.bfloat16)
    k = (torch.randn(B, Hkv, Nkv, d, generator=g) * shape.value_scale).to(torch.bfloat16)
    v = (torch.randn(B, Hkv, Nkv, d, generator=g) * shape.value_scale).to(torch.bfloat16)
    kv_lens = None
    if shape.kv_len_range is not None:
        lo, hi = shape.kv_len_range
        kv_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return dict(q=q, k=k, v=v, kv_lens=kv_lens)


def backward_upstream(shape: PrefillShape):
    """Seeded upstream gradient dO [B, H, Nq, d] (bf16, standard normal) for the backward of a
    prefill workload; its own seed (shape.seed + 500), so the forward's inputs are unchanged."""
    g = torch.Generator().manual_seed(shape.seed + 500)
    return torch.randn(shape.B, shape.H, shape.Nq, shape.d, generator=g).to(torch.bfloat16)


POISON_VALUE = 3.0e4


def decode_inputs(shape: DecodeShape, ctx_lens=None, kv_heads=None):
    """Return dict(q, k_pages, v_pages, page_table, ctx_lens) as CPU tensors.

    ``ctx_lens`` (optional list) overrides the drawn context lengths (for edge cases).
    ``kv_heads`` (optional) gives the cache fewer heads than the query (grouped-query
    attention; shape.H must be a multiple of it).  The poison page is the last physical page."""
    g = torch.Generator().manual_seed(shape.seed)
    B, H, d, ps = shape.B, shape.H, shape.d, shape.page_size
    Hkv = H if kv_heads is None else kv_heads
    if H % Hkv:
        raise ValueError("query heads must be a multiple of the cache heads")
    lo, hi = shape.ctx_range
    drawn = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    cl = drawn if ctx_lens is None else torch.tensor(list(ctx_lens), dtype=torch.int64)
    max_pages = max(shape.max_pages, int((cl.max().item() + ps - 1) // ps) if B else 1, 1)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16)
    pages_per_seq = [(int(c) + ps - 1) // ps for c in cl.tolist()]
    used = sum(pages_per_seq)
    perm = torch.randperm(used, generator=g).to(torch.int32)
    poison = used  # physical id of the poison page
    table = torch.full((B, max_pages), poison, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    num_pages = used + 1
    k = torch.randn(num_pages, Hkv, ps, d, generator=g).to(torch.bfloat16)
    v = torch.randn(num_pages, Hkv, ps, d, generator=g).to(torch.bfloat16)
    k[poison] = POISON_VALUE
    v[poison] = POISON_VALUE
    for b, c in enumerate(cl.tolist()):
        tail = int(c) % ps
        if tail:
            last = int(table[b, pages_per_seq[b] - 1])
            k[last, :, tail:, :] = POISON_VALUE
            v[last, :, tail:, :] = POISON_VALUE
    return dict(q=q, k_pages=k, v_pages=v, page_table=table, ctx_lens=cl.to(torch.int32))
