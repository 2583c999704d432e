"""GPU parity for grouped-query / multi-query attention (query heads sharing key/value
heads) against the fp64 oracle: prefill and paged decode, same tolerances as the
multi-head tests."""
import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads

pytestmark = pytest.mark.gpu
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    return binding


def check(o, lse, o_ref, lse_ref, what):
    o = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (what, err.max(), err.mean())
    l = lse.cpu().numpy().astype(np.float64)
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), inf), what
    if (~inf).any():
        assert np.abs(l[~inf] - lse_ref[~inf]).max() <= LSE_MAX, what


PREFILL = [
    workloads.PrefillShape("GQA 8/2 N300 d128 causal", 2, 8, 300, 300, 128, True, seed=70, kv_heads=2),
    workloads.PrefillShape("GQA 6/3 N260 d64", 1, 6, 260, 260, 64, False, seed=71, kv_heads=3),
    workloads.PrefillShape("MQA 4/1 N384 d64 causal padded", 3, 4, 384, 384, 64, True, seed=72, kv_heads=1,
                           kv_len_range=(1, 384)),
    workloads.PrefillShape("GQA 4/2 Nq<Nkv causal d128", 1, 4, 150, 400, 128, True, seed=73, kv_heads=2),
]


@pytest.mark.parametrize("shape", PREFILL, ids=lambda s: s.name)
def test_gqa_prefill_vs_oracle(lib, oracle_mod, shape):
    inp = workloads.prefill_inputs(shape)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kl = inp["kv_lens"]
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    lib.attn_fwd_gqa(q, k, v, shape.causal, shape.scale, kv_lens=None if kl is None else kl.cuda(), out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.attn_fwd_gqa(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=kl)
    check(o, lse, o_ref, lse_ref, shape.name)


def test_gqa_prefill_equals_mha_with_hkv_equal_h(lib):
    shape = workloads.PrefillShape("GQA with Hkv = H", 1, 4, 200, 200, 128, True, seed=74)
    inp = workloads.prefill_inputs(shape)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = lib.attn_fwd_gqa(q, k, v, True, shape.scale)
    o2, l2 = lib.attn_fwd(q, k, v, True, shape.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


DECODE = [
    (workloads.DecodeShape("GQA 32/8 decode d128", 4, 32, 128, (1, 3000), seed=75), 8, [3000, 1, 700, 1500]),
    (workloads.DecodeShape("GQA 12/6 decode d64", 3, 12, 64, (1, 600), seed=76), 6, [600, 17, 0]),
    (workloads.DecodeShape("MQA 16/1 decode d128", 2, 16, 128, (1, 2100), seed=77), 1, [2100, 513]),
    (workloads.DecodeShape("GQA 24/2 decode d128", 2, 24, 128, (1, 900), seed=78), 2, [900, 33]),
]


@pytest.mark.parametrize("shape,hkv,ctx", DECODE, ids=[d[0].name for d in DECODE])
def test_gqa_decode_vs_oracle(lib, oracle_mod, shape, hkv, ctx):
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=hkv)
    d = {k: v.cuda() for k, v in inp.items()}
    o = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), device="cuda")
    lib.paged_attn_decode_gqa(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"], shape.scale,
                              out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                                 inp["ctx_lens"], shape.scale)
    check(o, lse, o_ref, lse_ref, shape.name)


def test_gqa_decode_full_size_vs_oracle(lib, oracle_mod):
    # the grouped-query decode workload (B=32, 32 query heads over 8 cache heads, ctx U[512,8192])
    shape = workloads.PAGED_DECODE_GQA
    inp = workloads.decode_inputs(shape, kv_heads=workloads.PAGED_DECODE_GQA_KV_HEADS)
    d = {k: v.cuda() for k, v in inp.items()}
    o, lse = lib.paged_attn_decode_gqa(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"],
                                       shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                                 inp["ctx_lens"], shape.scale)
    check(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("hkv", [8, 2])
def test_gqa_decode_ignores_nan_past_the_context(lib, oracle_mod, hkv):
    # cache slots past each sequence's end hold NaN (memory nobody wrote): they must not reach O
    shape = workloads.DecodeShape("GQA NaN tail", 3, 16, 128, (1, 700), seed=79)
    ctx = [700, 33, 129]
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=hkv)
    for b, n in enumerate(ctx):
        if n % 16:
            last = int(inp["page_table"][b, n // 16])
            inp["k_pages"][last, :, n % 16:] = float("nan")
            inp["v_pages"][last, :, n % 16:] = float("nan")
    d = {k: v.cuda() for k, v in inp.items()}
    o, lse = lib.paged_attn_decode_gqa(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"],
                                       shape.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                                 inp["ctx_lens"], shape.scale)
    check(o, lse, o_ref, lse_ref, shape.name)
