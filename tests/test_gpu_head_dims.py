"""GPU parity at head dims 32, 80 and 96 (the other dims the Kernel-Inference-Engine README
instantiates its attention kernel for, besides 64 and 128): contiguous prefill (causal, key
padding, ragged, Nq != Nkv), grouped-query heads, chunked prefill over pages and the KV append;
paged decode (multi-head, grouped-query, over an e4m3 cache) and the e4m3 KV append; against the
fp64 oracle.  Same tolerances as the other
forward tests: O max-abs <= 1e-2, mean-abs <= 1e-3, LSE abs <= 1e-3."""
import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads

from test_gpu_parity import compare, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    return binding


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


SHAPES = []
for d in (32, 80, 96):
    SHAPES += [
        workloads.PrefillShape(f"d{d} one tile", 1, 1, 128, 128, d, False, seed=400 + d),
        workloads.PrefillShape(f"d{d} ragged causal", 2, 3, 300, 300, d, True, seed=401 + d),
        workloads.PrefillShape(f"d{d} ragged non-causal", 2, 2, 260, 260, d, False, seed=402 + d),
        workloads.PrefillShape(f"d{d} Nq<Nkv causal", 1, 2, 200, 457, d, True, seed=403 + d),
        workloads.PrefillShape(f"d{d} Nq>Nkv causal (masked rows)", 1, 2, 333, 150, d, True, seed=404 + d),
        workloads.PrefillShape(f"d{d} key padding causal", 3, 2, 384, 384, d, True, kv_len_range=(1, 384),
                               seed=405 + d),
        workloads.PrefillShape(f"d{d} several tiles", 2, 4, 1024, 1024, d, True, seed=406 + d),
    ]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_prefill_head_dim_vs_oracle(lib, oracle_mod, shape):
    inp, kl, o, lse = run_prefill(lib, shape)
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=kl)
    compare(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("d,Hq,Hkv", [(32, 8, 2), (80, 4, 1), (96, 6, 3)])
def test_gqa_prefill_head_dim_vs_oracle(lib, oracle_mod, d, Hq, Hkv):
    shape = workloads.PrefillShape(f"gqa d{d}", 2, Hq, 270, 390, d, True, seed=500 + d, kv_heads=Hkv)
    inp = workloads.prefill_inputs(shape)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = lib.attn_fwd_gqa(q, k, v, True, shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.attn_fwd_gqa(inp["q"], inp["k"], inp["v"], True, shape.scale)
    compare(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("d", [32, 80, 96])
def test_append_then_paged_prefill_head_dim_vs_oracle(lib, oracle_mod, d):
    # a prefill step at this head dim: append the chunk's K/V into the pages (checked bit-exact
    # against a direct scatter), then attend over the pages; compared with the oracle
    B, H, Hkv, Nq, old = 3, 4, 2, 120, [300, 0, 77]
    ctx = [o + Nq for o in old]
    shape = workloads.DecodeShape(f"paged d{d}", B, H, d, (1, max(ctx)), seed=600 + d)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    kn, vn = rand_bf16((B, Hkv, Nq, d), 601 + d), rand_bf16((B, Hkv, Nq, d), 602 + d)
    q = rand_bf16((B, H, Nq, d), 603 + d)
    kp, vp = inp["k_pages"].clone(), inp["v_pages"].clone()
    for b in range(B):
        for t in range(Nq):
            pos = old[b] + t
            pg = int(inp["page_table"][b, pos // 16])
            kp[pg, :, pos % 16] = kn[b, :, t]
            vp[pg, :, pos % 16] = vn[b, :, t]
    dv = {k: v.cuda() for k, v in inp.items()}
    lib.paged_kv_append(kn.cuda(), vn.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"],
                        torch.tensor(old, dtype=torch.int32).cuda())
    o, lse = lib.paged_attn_prefill(q.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"], True,
                                    shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    assert torch.equal(dv["k_pages"].cpu(), kp) and torch.equal(dv["v_pages"].cpu(), vp)
    o_ref, lse_ref = oracle_mod.paged_prefill_gqa(q, kp, vp, inp["page_table"], inp["ctx_lens"], True, shape.scale)
    compare(o, lse, o_ref, lse_ref, f"paged d{d}")


# ----------------------------------------------------------------------------- decode at d = 32, 80, 96

DECODE_CTX = [1, 16, 17, 700, 1500, 0, 513]  # one token, a full page, a page plus one, several splits, empty


def _compare_decode(o, lse, o_ref, lse_ref, what):
    compare(o, lse, o_ref, lse_ref, what)


@pytest.mark.parametrize("d", [32, 80, 96])
def test_paged_decode_head_dim_vs_oracle(lib, oracle_mod, d):
    shape = workloads.DecodeShape(f"decode d{d}", len(DECODE_CTX), 3, d, (1, max(DECODE_CTX)), seed=700 + d)
    inp = workloads.decode_inputs(shape, ctx_lens=DECODE_CTX)
    dv = {k: v.cuda() for k, v in inp.items()}
    o = torch.full_like(dv["q"], float("nan"))
    lse = torch.full(dv["q"].shape[:2], float("nan"), device="cuda")
    lib.paged_attn_decode(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"], shape.scale,
                          out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                             inp["ctx_lens"], shape.scale)
    _compare_decode(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("d,H,Hkv", [(32, 16, 2), (80, 8, 2), (96, 4, 2), (80, 6, 2), (96, 12, 4)])
def test_paged_decode_gqa_head_dim_vs_oracle(lib, oracle_mod, d, H, Hkv):
    # groups of 8, 4 and 2 query heads (tensor-core kernel) and of 3 (one query head per CTA)
    shape = workloads.DecodeShape(f"gqa decode d{d} {H}/{Hkv}", len(DECODE_CTX), H, d, (1, max(DECODE_CTX)),
                                  seed=710 + d + H)
    inp = workloads.decode_inputs(shape, ctx_lens=DECODE_CTX, kv_heads=Hkv)
    dv = {k: v.cuda() for k, v in inp.items()}
    o, lse = lib.paged_attn_decode_gqa(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"],
                                       shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                                 inp["ctx_lens"], shape.scale)
    _compare_decode(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("d,H,Hkv", [(32, 4, 4), (80, 4, 4), (96, 4, 4), (80, 8, 2), (96, 8, 1), (32, 6, 2)])
def test_paged_decode_fp8_head_dim_vs_oracle(lib, oracle_mod, d, H, Hkv):
    scale_kv = 6.0 / 448
    shape = workloads.DecodeShape(f"fp8 decode d{d} {H}/{Hkv}", len(DECODE_CTX), H, d, (1, max(DECODE_CTX)),
                                  seed=720 + d + H)
    inp = workloads.decode_inputs(shape, ctx_lens=DECODE_CTX, kv_heads=Hkv)
    dv = {k: v.cuda() for k, v in inp.items()}
    kc = lib.kv_quantize_fp8(dv["k_pages"], scale_kv)
    vc = lib.kv_quantize_fp8(dv["v_pages"], scale_kv)
    o, lse = lib.paged_attn_decode_fp8(dv["q"], kc, vc, scale_kv, scale_kv, dv["page_table"], dv["ctx_lens"],
                                       shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc.cpu(), vc.cpu(), scale_kv, scale_kv,
                                                     inp["page_table"], inp["ctx_lens"], shape.scale)
    _compare_decode(o, lse, o_ref, lse_ref, shape.name)


@pytest.mark.parametrize("d", [32, 80, 96])
def test_append_fp8_head_dim_bit_exact(lib, oracle_mod, d):
    B, Hkv, Nnew = 3, 2, 29
    ks, vs = 6.0 / 448, 12.0 / 448
    shape = workloads.DecodeShape(f"fp8 append d{d}", B, 4, d, (1, 300), seed=730 + d)
    inp = workloads.decode_inputs(shape, ctx_lens=[300, 29, 100], kv_heads=Hkv)
    start = torch.tensor([271, 0, 71], dtype=torch.int32)
    kn, vn = rand_bf16((B, Hkv, Nnew, d), 731 + d), rand_bf16((B, Hkv, Nnew, d), 732 + d)
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
    assert lib.attn_check_device_status() == 0
    assert torch.equal(kd.cpu(), kp) and torch.equal(vd.cpu(), vp)


# every decode form over bf16 pages: multi-head lane groups (d = 32), multi-head on the tensor-core
# kernel (d = 64), the split dim layout (d = 80, 96), a token per warp (d = 128), grouped-query
BF16_NAN_TAIL_FORMS = [(32, 4, 4), (64, 4, 4), (80, 4, 4), (96, 4, 4), (128, 4, 4), (128, 8, 2), (32, 8, 2)]


@pytest.mark.parametrize("d,H,Hkv", BF16_NAN_TAIL_FORMS, ids=[f"d{d}-{h}/{k}" for d, h, k in BF16_NAN_TAIL_FORMS])
def test_decode_ignores_nan_past_the_context(lib, oracle_mod, d, H, Hkv):
    # NaN in the cache slots past each sequence's end (K and V) must not reach O or LSE
    ctx = [700, 33, 129, 16]
    shape = workloads.DecodeShape(f"nan tail d{d}", len(ctx), H, d, (1, max(ctx)), seed=740 + d + H)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    kp, vp = inp["k_pages"].clone(), inp["v_pages"].clone()
    for b, n in enumerate(ctx):
        if n % 16:
            last = int(inp["page_table"][b, n // 16])
            kp[last, :, n % 16:] = float("nan")
            vp[last, :, n % 16:] = float("nan")
    dv = {k: v.cuda() for k, v in inp.items()}
    if Hkv == H:
        o, lse = lib.paged_attn_decode(dv["q"], kp.cuda(), vp.cuda(), dv["page_table"], dv["ctx_lens"], shape.scale)
    else:
        o, lse = lib.paged_attn_decode_gqa(dv["q"], kp.cuda(), vp.cuda(), dv["page_table"], dv["ctx_lens"],
                                           shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], kp, vp, inp["page_table"], inp["ctx_lens"], shape.scale)
    assert np.isfinite(o.float().cpu().numpy()).all()
    _compare_decode(o, lse, o_ref, lse_ref, shape.name)
