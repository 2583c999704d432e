"""GPU parity for chunked prefill over the paged KV cache (queries = the last Nq cached
positions of each sequence, bottom-right causal) and for appending new tokens' K/V to
the pages, against the fp64 oracle and a direct scatter."""
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


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


CASES = [
    # (name, B, H, Hkv, d, Nq, ctx lengths, causal)
    ("d128 causal ragged", 3, 4, 4, 128, 200, [200, 777, 345], True),
    ("d64 GQA causal", 2, 8, 2, 64, 130, [1000, 130], True),
    ("d128 non-causal", 2, 2, 2, 128, 64, [64, 1500], False),
    ("d128 MQA causal short", 4, 4, 1, 128, 17, [17, 33, 300, 2049], True),
    ("d64 Nq 300 causal", 1, 2, 2, 64, 300, [3000], True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_paged_prefill_vs_oracle(lib, oracle_mod, case):
    name, B, H, Hkv, d, Nq, ctx, causal = case
    shape = workloads.DecodeShape(name, B, H, d, (1, max(ctx)), seed=80 + len(name))
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    q = rand_bf16((B, H, Nq, d), 81)
    dv = {k: v.cuda() for k, v in inp.items()}
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), device="cuda")
    lib.paged_attn_prefill(q.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"], causal,
                           shape.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_prefill_gqa(q, inp["k_pages"], inp["v_pages"], inp["page_table"],
                                                  inp["ctx_lens"], causal, shape.scale)
    og = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    assert np.isfinite(og).all() and err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lg = lse.cpu().numpy().astype(np.float64)
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), inf)
    assert np.abs(lg[~inf] - lse_ref[~inf]).max() <= LSE_MAX


def test_kv_append_scatters_bit_exact(lib):
    # append 37 new tokens after start_pos, compare with a direct scatter through the page table
    shape = workloads.DecodeShape("append", 3, 4, 128, (1, 400), seed=90)
    inp = workloads.decode_inputs(shape, ctx_lens=[400, 100, 250], kv_heads=2)
    start = torch.tensor([363, 0, 213], dtype=torch.int32)  # last 37 positions of each sequence
    kn = rand_bf16((3, 2, 37, 128), 91)
    vn = rand_bf16((3, 2, 37, 128), 92)
    kp, vp = inp["k_pages"].clone(), inp["v_pages"].clone()
    for b in range(3):
        for t in range(37):
            pos = int(start[b]) + t
            pg = int(inp["page_table"][b, pos // 16])
            kp[pg, :, pos % 16] = kn[b, :, t]
            vp[pg, :, pos % 16] = vn[b, :, t]
    kd, vd = inp["k_pages"].cuda(), inp["v_pages"].cuda()
    lib.paged_kv_append(kn.cuda(), vn.cuda(), kd, vd, inp["page_table"].cuda(), start.cuda())
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kp) and torch.equal(vd.cpu(), vp)


def test_append_then_paged_prefill_matches_contiguous(lib):
    # prefill step: append the chunk's K/V, then attend with its queries (causal) == contiguous attn_fwd
    B, H, d, Nq, old = 2, 4, 128, 96, [160, 40]
    shape = workloads.DecodeShape("chunk", B, H, d, (1, 400), seed=93)
    ctx = [o + Nq for o in old]
    inp = workloads.decode_inputs(shape, ctx_lens=ctx)
    q = rand_bf16((B, H, Nq, d), 94)
    kn, vn = rand_bf16((B, H, Nq, d), 95), rand_bf16((B, H, Nq, d), 96)
    dv = {k: v.cuda() for k, v in inp.items()}
    lib.paged_kv_append(kn.cuda(), vn.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"],
                        torch.tensor(old, dtype=torch.int32).cuda())
    o, lse = lib.paged_attn_prefill(q.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"], True,
                                    shape.scale)
    torch.cuda.synchronize()
    for b in range(B):
        n = ctx[b]
        pages = dv["page_table"][b, :(n + 15) // 16].long()
        kc = dv["k_pages"][pages].permute(1, 0, 2, 3).reshape(H, -1, d)[:, :n][None].contiguous()
        vc = dv["v_pages"][pages].permute(1, 0, 2, 3).reshape(H, -1, d)[:, :n][None].contiguous()
        assert torch.equal(kc[0, :, old[b]:], kn[b].cuda())  # the appended rows are in place
        oc, lc = lib.attn_fwd(q[b:b + 1].cuda(), kc, vc, True, shape.scale)
        torch.cuda.synchronize()
        assert (oc[0].float() - o[b].float()).abs().max().item() <= 1e-2
        assert (lc[0] - lse[b]).abs().max().item() <= 1e-3


def _check(o, lse, o_ref, lse_ref):
    og = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    assert np.isfinite(og).all() and err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lg = lse.cpu().numpy().astype(np.float64)
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), inf)
    if (~inf).any():
        assert np.abs(lg[~inf] - lse_ref[~inf]).max() <= LSE_MAX
    assert not og[inf].any()  # rows without a key are exactly zero


def test_unmapped_pages_mean_the_same_on_every_paged_entry_point(lib, oracle_mod):
    """A page id outside the pool is an unmapped page holding no token, on the chunked prefill
    and on every decode entry point alike; compared with the oracle's reading of it."""
    B, H, Hkv, d = 3, 8, 2, 128
    ctx = [1000, 300, 40]
    shape = workloads.DecodeShape("unmapped", B, H, d, (1, max(ctx)), seed=97)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=Hkv)
    pt = inp["page_table"]
    pt[0, 3] = 1 << 24          # past the pool, inside a 128-key tile
    pt[0, 40] = -1              # negative, in a later tile
    pt[0, 8:16] = -5            # one whole 128-key tile unmapped
    pt[1, 0] = inp["k_pages"].shape[0]  # the first id past the end
    pt[2, :3] = -1              # every page of sequence 2: no key at all
    dv = {k: v.cuda() for k, v in inp.items()}
    for Nq, causal in ((64, True), (200, False), (1, True)):
        q = rand_bf16((B, H, Nq, d), 98 + Nq)
        o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, Nq), float("nan"), device="cuda")
        lib.paged_attn_prefill(q.cuda(), dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"], causal,
                               shape.scale, out=o, lse=lse)
        torch.cuda.synchronize()
        assert lib.attn_check_device_status() == 0
        o_ref, lse_ref = oracle_mod.paged_prefill_gqa(q, inp["k_pages"], inp["v_pages"], pt, inp["ctx_lens"], causal,
                                                      shape.scale, skip_bad_pages=True)
        _check(o, lse, o_ref, lse_ref)
    # decode over the same table: grouped-query, multi-head (the same heads repeated) and e4m3
    o_ref, lse_ref = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], pt, inp["ctx_lens"],
                                                 shape.scale, skip_bad_pages=True)
    o, lse = lib.paged_attn_decode_gqa(dv["q"], dv["k_pages"], dv["v_pages"], dv["page_table"], dv["ctx_lens"],
                                       shape.scale)
    torch.cuda.synchronize()
    _check(o, lse, o_ref, lse_ref)
    kmh = dv["k_pages"].repeat_interleave(H // Hkv, dim=1).contiguous()
    vmh = dv["v_pages"].repeat_interleave(H // Hkv, dim=1).contiguous()
    o, lse = lib.paged_attn_decode(dv["q"], kmh, vmh, dv["page_table"], dv["ctx_lens"], shape.scale)
    torch.cuda.synchronize()
    _check(o, lse, o_ref, lse_ref)
    kc = lib.kv_quantize_fp8(dv["k_pages"], 0.25)
    vc = lib.kv_quantize_fp8(dv["v_pages"], 0.25)
    o, lse = lib.paged_attn_decode_fp8(dv["q"], kc, vc, 0.25, 0.25, dv["page_table"], dv["ctx_lens"], shape.scale)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc.cpu(), vc.cpu(), 0.25, 0.25, pt, inp["ctx_lens"],
                                                     shape.scale, skip_bad_pages=True)
    _check(o, lse, o_ref, lse_ref)
