"""GPU parity for the FP8 (E4M3) KV cache: conversion bit-exact against the oracle's code table
(every finite bf16 value, several scales), the FP8 KV append bit-exact against the oracle's
quantisation and a direct scatter, and decode over e4m3 pages against the fp64 oracle (same
tolerances as the bf16 decode: O max-abs <= 1e-2, mean-abs <= 1e-3, LSE abs <= 1e-3; the
oracle dequantises the codes exactly, the kernel widens them exactly, so only fp32 arithmetic
and the bf16 output separate the two)."""
import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads

pytestmark = pytest.mark.gpu
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
KV_SCALE = 6.0 / 448  # N(0,1) data: values beyond +-6 saturate


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    return binding


def all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    return torch.from_numpy(bits[finite].view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("scale", [1.0, KV_SCALE, 0.37, 1e-3, 250.0])
def test_quantize_every_finite_bf16_bit_exact(lib, oracle_mod, scale):
    x = all_finite_bf16()
    x = x[: x.numel() // 8 * 8].contiguous()
    got = lib.kv_quantize_fp8(x.cuda(), scale)
    torch.cuda.synchronize()
    want = oracle_mod.e4m3_quantize(x, scale)
    g = got.cpu().numpy()
    bad = np.nonzero(g != want)[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. x={x[bad[0]].item()} got {g[bad[0]]:#x} want {want[bad[0]]:#x}"


def test_append_fp8_bit_exact(lib, oracle_mod):
    B, Hkv, d, Nnew = 3, 2, 128, 37
    shape = workloads.DecodeShape("fp8 append", B, 4, d, (1, 400), seed=700)
    inp = workloads.decode_inputs(shape, ctx_lens=[400, 100, 250], kv_heads=Hkv)
    start = torch.tensor([363, 0, 213], dtype=torch.int32)
    g = torch.Generator().manual_seed(701)
    kn = torch.randn(B, Hkv, Nnew, d, generator=g).to(torch.bfloat16)
    vn = (torch.randn(B, Hkv, Nnew, d, generator=g) * 3).to(torch.bfloat16)
    ks, vs = KV_SCALE, 2 * KV_SCALE
    kp = torch.from_numpy(oracle_mod.e4m3_quantize(inp["k_pages"], ks))
    vp = torch.from_numpy(oracle_mod.e4m3_quantize(inp["v_pages"], vs))
    kq = torch.from_numpy(oracle_mod.e4m3_quantize(kn, ks))
    vq = torch.from_numpy(oracle_mod.e4m3_quantize(vn, vs))
    kd, vd = kp.cuda(), vp.cuda()
    for b in range(B):
        for t in range(Nnew):
            pos = int(start[b]) + t
            pg = int(inp["page_table"][b, pos // 16])
            kp[pg, :, pos % 16] = kq[b, :, t]
            vp[pg, :, pos % 16] = vq[b, :, t]
    lib.paged_kv_append_fp8(kn.cuda(), vn.cuda(), kd, vd, ks, vs, inp["page_table"].cuda(), start.cuda())
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kp) and torch.equal(vd.cpu(), vp)


def run_fp8_decode(lib, oracle_mod, shape, ctx=None, kv_heads=None, ks=KV_SCALE, vs=KV_SCALE):
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=kv_heads)
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], ks)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], vs)
    o = torch.full(inp["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(inp["q"].shape[:2], float("nan"), device="cuda")
    lib.paged_attn_decode_fp8(inp["q"].cuda(), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), ks, vs,
                              inp["page_table"].cuda(), inp["ctx_lens"].cuda(), shape.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc, vc, ks, vs, inp["page_table"], inp["ctx_lens"],
                                                     shape.scale)
    og = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    assert np.isfinite(og).all() and err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.abs(lg - lse_ref).max() <= LSE_MAX
    return err.max(), err.mean()


CASES = [
    # name, B, H, Hkv, d, ctx
    ("d128 MHA ragged", 4, 4, 4, 128, [1, 17, 513, 2000]),
    ("d64 MHA", 3, 2, 2, 64, [16, 1024, 777]),
    ("d128 GQA 4", 3, 8, 2, 128, [5, 600, 1500]),
    ("d64 MQA 8", 2, 8, 1, 64, [300, 1025]),
    ("d128 GQA chunk edges", 2, 4, 1, 128, [512, 1536]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fp8_decode_vs_oracle(lib, oracle_mod, case):
    name, B, H, Hkv, d, ctx = case
    shape = workloads.DecodeShape(name, B, H, d, (1, max(ctx)), seed=710 + len(name))
    run_fp8_decode(lib, oracle_mod, shape, ctx=ctx, kv_heads=Hkv)


def test_fp8_decode_unequal_scales(lib, oracle_mod):
    shape = workloads.DecodeShape("scales", 2, 4, 128, (1, 900), seed=720)
    run_fp8_decode(lib, oracle_mod, shape, ctx=[900, 33], ks=0.02, vs=0.5)


def test_fp8_decode_full_size(lib, oracle_mod):
    # the paged-decode workload (B=32, H=32, d=128, ctx U[512,8192]) with its cache in e4m3
    run_fp8_decode(lib, oracle_mod, workloads.PAGED_DECODE)


def test_fp8_gqa_decode_full_size(lib, oracle_mod):
    # the grouped-query decode workload (32 query heads over 8 cache heads) with its cache in e4m3
    run_fp8_decode(lib, oracle_mod, workloads.PAGED_DECODE_GQA, kv_heads=workloads.PAGED_DECODE_GQA_KV_HEADS)


# every decode form: grouped-query tensor-core kernel, multi-head lane groups (d = 32, 64), the split
# dim layout (d = 80), a token per warp (d = 128), multi-head on the tensor-core kernel (d = 96)
NAN_TAIL_FORMS = [(128, 16, 4), (32, 4, 4), (64, 4, 4), (80, 4, 4), (128, 4, 4), (96, 4, 4), (32, 8, 2)]


@pytest.mark.parametrize("d,H,Hkv", NAN_TAIL_FORMS, ids=[f"d{d}-{h}/{k}" for d, h, k in NAN_TAIL_FORMS])
def test_fp8_decode_ignores_nan_codes_past_the_context(lib, oracle_mod, d, H, Hkv):
    # e4m3 NaN codes (0x7F) in cache slots past each sequence's end must not reach O
    shape = workloads.DecodeShape("fp8 NaN tail", 3, H, d, (1, 700), seed=730 + d + H)
    ctx = [700, 33, 129]
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], KV_SCALE)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], KV_SCALE)
    for b, n in enumerate(ctx):
        if n % 16:
            last = int(inp["page_table"][b, n // 16])
            kc[last, :, n % 16:] = 0x7F
            vc[last, :, n % 16:] = 0x7F
    o, lse = lib.paged_attn_decode_fp8(inp["q"].cuda(), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                                       KV_SCALE, KV_SCALE, inp["page_table"].cuda(), inp["ctx_lens"].cuda(),
                                       shape.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc, vc, KV_SCALE, KV_SCALE, inp["page_table"],
                                                     inp["ctx_lens"], shape.scale)
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(og).all()
    assert np.abs(og - o_ref).max() <= O_MAX
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_MAX


def test_fp8_gqa_decode_query_beyond_fp16_range(lib, oracle_mod):
    # the grouped-query e4m3 path multiplies q in fp16; a query of magnitude ~1e5 (past fp16's
    # 65504) with a correspondingly smaller softmax scale must give the same attention
    shape = workloads.DecodeShape("fp8 big q", 2, 8, 128, (1, 800), seed=740)
    inp = workloads.decode_inputs(shape, ctx_lens=[800, 77], kv_heads=2)
    big = 3.0e4
    q = (inp["q"].float() * big).to(torch.bfloat16)
    scale = shape.scale / big
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], KV_SCALE)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], KV_SCALE)
    o, lse = lib.paged_attn_decode_fp8(q.cuda(), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(), KV_SCALE,
                                       KV_SCALE, inp["page_table"].cuda(), inp["ctx_lens"].cuda(), scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_mod.paged_decode_fp8_gqa(q, kc, vc, KV_SCALE, KV_SCALE, inp["page_table"],
                                                     inp["ctx_lens"], scale)
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(og).all()
    assert np.abs(og - o_ref).max() <= O_MAX and np.abs(og - o_ref).mean() <= O_MEAN
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_MAX


# ----------------------------------------------------------------------------- chunked prefill over e4m3

PREFILL_FP8_CASES = [
    # (name, B, H, Hkv, d, Nq, ctx lengths, causal)
    ("d128 GQA causal ragged", 3, 8, 2, 128, 200, [200, 777, 345], True),
    ("d128 MHA non-causal", 2, 2, 2, 128, 64, [64, 1500], False),
    ("d64 MQA causal", 2, 4, 1, 64, 130, [1000, 130], True),
    ("d32 causal short", 4, 4, 2, 32, 17, [17, 33, 300, 2049], True),
    ("d80 GQA causal", 2, 6, 3, 80, 150, [600, 150], True),
    ("d96 causal Nq>ctx (rows without keys)", 2, 4, 4, 96, 100, [60, 400], True),
]


@pytest.mark.parametrize("case", PREFILL_FP8_CASES, ids=[c[0] for c in PREFILL_FP8_CASES])
def test_paged_prefill_fp8_vs_oracle(lib, oracle_mod, case):
    name, B, H, Hkv, d, Nq, ctx, causal = case
    shape = workloads.DecodeShape(name, B, H, d, (1, max(ctx)), seed=750 + len(name))
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    g = torch.Generator().manual_seed(751)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    dv = {k: v.cuda() for k, v in inp.items()}
    ks, vs = KV_SCALE, 2 * KV_SCALE
    kc = lib.kv_quantize_fp8(dv["k_pages"], ks)
    vc = lib.kv_quantize_fp8(dv["v_pages"], vs)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), device="cuda")
    lib.paged_attn_prefill_fp8(q.cuda(), kc, vc, ks, vs, dv["page_table"], dv["ctx_lens"], causal, shape.scale,
                               out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_prefill_fp8_gqa(q, kc.cpu(), vc.cpu(), ks, vs, inp["page_table"],
                                                      inp["ctx_lens"], causal, shape.scale)
    og = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    assert np.isfinite(og).all() and err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lg = lse.cpu().numpy().astype(np.float64)
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), inf)
    assert np.abs(lg[~inf] - lse_ref[~inf]).max() <= LSE_MAX
    assert not og[inf].any()


@pytest.mark.parametrize("d", [128, 64])
def test_paged_prefill_fp8_query_beyond_fp16_range(lib, oracle_mod, d):
    # over e4m3 pages the products run in fp16 with each query row brought below 2^15 by a power of
    # two: rows of magnitude ~1e5 (past fp16's 65504) next to rows of ordinary size, with a softmax
    # scale that keeps the large rows' scores O(1), must give the oracle's attention
    B, H, Hkv, Nq, ctx = 2, 4, 2, 150, [150, 900]
    shape = workloads.DecodeShape("fp8 prefill big q", B, H, d, (1, max(ctx)), seed=770 + d)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    g = torch.Generator().manual_seed(771)
    big = 3.0e4
    rows = torch.where(torch.rand(B, H, Nq, 1, generator=g) < 0.5, big, 1.0)
    q = (torch.randn(B, H, Nq, d, generator=g) * rows).to(torch.bfloat16)
    scale = shape.scale / big
    kc = torch.from_numpy(oracle_mod.e4m3_quantize(inp["k_pages"], KV_SCALE))
    vc = torch.from_numpy(oracle_mod.e4m3_quantize(inp["v_pages"], KV_SCALE))
    o, lse = lib.paged_attn_prefill_fp8(q.cuda(), kc.cuda(), vc.cuda(), KV_SCALE, KV_SCALE,
                                        inp["page_table"].cuda(), inp["ctx_lens"].cuda(), True, scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_prefill_fp8_gqa(q, kc, vc, KV_SCALE, KV_SCALE, inp["page_table"],
                                                      inp["ctx_lens"], True, scale)
    og = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    assert np.isfinite(og).all() and err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_MAX


def test_append_fp8_then_paged_prefill_fp8_with_unmapped_pages(lib, oracle_mod):
    # a serving step over an e4m3 cache: append the chunk's K/V (converted), then attend; one page
    # of the table is unmapped (its positions hold no token), as on every paged entry point
    B, H, Hkv, d, Nq, old = 2, 8, 2, 128, 96, [700, 40]
    ctx = [o + Nq for o in old]
    shape = workloads.DecodeShape("fp8 step", B, H, d, (1, max(ctx)), seed=760)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    inp["page_table"][0, 5] = -1
    g = torch.Generator().manual_seed(761)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, Nq, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, Nq, d, generator=g).to(torch.bfloat16)
    dv = {k: v.cuda() for k, v in inp.items()}
    ks, vs = KV_SCALE, KV_SCALE
    kc = lib.kv_quantize_fp8(dv["k_pages"], ks)
    vc = lib.kv_quantize_fp8(dv["v_pages"], vs)
    lib.paged_kv_append_fp8(kn.cuda(), vn.cuda(), kc, vc, ks, vs, dv["page_table"],
                            torch.tensor(old, dtype=torch.int32).cuda())
    o, lse = lib.paged_attn_prefill_fp8(q.cuda(), kc, vc, ks, vs, dv["page_table"], dv["ctx_lens"], True,
                                        shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_prefill_fp8_gqa(q, kc.cpu(), vc.cpu(), ks, vs, inp["page_table"],
                                                      inp["ctx_lens"], True, shape.scale, skip_bad_pages=True)
    err = np.abs(o.float().cpu().numpy() - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_MAX
