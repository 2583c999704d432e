"""Pins for the fp64 oracle: closed forms, invariants, a hand-worked example and a
library special case.  None of these re-types the oracle's own formula; each is a
fact the definition of exact attention fixes independently of how it is computed.
Every test here runs on the CPU."""
import json
import math
import os

import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads
from attn_fwd_02_gb300.metrics import prefill_flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


# ----------------------------------------------------------------------------- hand-worked

def test_hand_worked_tiny_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "tiny_hand.json")))
    q = bf(g["q"]).reshape(1, 1, 2, 2)
    k = bf(g["k"]).reshape(1, 1, 2, 2)
    v = bf(g["v"]).reshape(1, 1, 2, 2)
    for key, causal, kl in (("noncausal", False, None), ("causal", True, None),
                            ("kvlen1", False, [1])):
        o, lse = oracle_mod.attn_fwd(q, k, v, causal, g["scale"],
                                     kv_lens=None if kl is None else np.array(kl, np.int32))
        np.testing.assert_allclose(o[0, 0], np.array(g[key]["o"]), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], np.array(g[key]["lse"]), rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_P_sum_to_one(oracle_mod, causal):
    # With V = identity (Nkv = d) the output row IS the probability row P_i.
    d = 16
    q = rand_bf16((2, 3, d, d), 1)
    k = rand_bf16((2, 3, d, d), 2)
    v = torch.eye(d).to(torch.bfloat16).expand(2, 3, d, d).contiguous()
    o, lse = oracle_mod.attn_fwd(q, k, v, causal, 0.25)
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (o >= 0).all()
    if causal:
        # key j > i has probability exactly 0
        iu = np.triu_indices(d, 1)
        assert np.all(o[:, :, iu[0], iu[1]] == 0.0)
    # P_ij = exp(s_ij - LSE_i): the LSE is the log-normaliser of these probabilities
    s = 0.25 * np.einsum("bhid,bhjd->bhij", f64(q), f64(k))
    p = np.exp(s - lse[..., None])
    if causal:
        p = np.tril(p)
    np.testing.assert_allclose(o, p, rtol=0, atol=1e-12)


def test_constant_V_returns_the_constant(oracle_mod):
    q = rand_bf16((2, 2, 37, 64), 3)
    k = rand_bf16((2, 2, 53, 64), 4)
    c = bf(np.linspace(-3, 3, 64)).reshape(1, 1, 1, 64).expand(2, 2, 53, 64).contiguous()
    for causal in (False, True):
        o, _ = oracle_mod.attn_fwd(q, k, c, causal, 0.125)
        np.testing.assert_allclose(o, np.broadcast_to(f64(c[:, :, :1]), o.shape), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_valid_values(oracle_mod):
    B, H, N, d = 2, 3, 40, 32
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    k = rand_bf16((B, H, N, d), 5)
    v = rand_bf16((B, H, N, d), 6)
    kl = np.array([17, 40], np.int32)
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 0.3, kv_lens=kl)
    for b in range(B):
        np.testing.assert_allclose(o[b], np.broadcast_to(f64(v[b, :, :kl[b]]).mean(1, keepdims=True),
                                                         o[b].shape), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], math.log(kl[b]), rtol=0, atol=1e-12)
    # causal: row i sees i+1 keys -> LSE = ln(i+1), O_i = mean of v_0..v_i
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.3)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape),
                               rtol=0, atol=1e-12)
    vv = f64(v)
    cm = np.cumsum(vv, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, cm, rtol=0, atol=1e-12)


def test_causal_query0_and_single_key(oracle_mod):
    q = rand_bf16((1, 2, 9, 16), 7)
    k = rand_bf16((1, 2, 9, 16), 8)
    v = rand_bf16((1, 2, 9, 16), 9)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.5)
    np.testing.assert_allclose(o[:, :, 0], f64(v[:, :, 0]), rtol=0, atol=1e-15)
    s00 = 0.5 * np.einsum("bhd,bhd->bh", f64(q[:, :, 0]), f64(k[:, :, 0]))
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-12)
    # a single key: every query returns that key's value row, LSE = its score
    o1, lse1 = oracle_mod.attn_fwd(q, k[:, :, :1].contiguous(), v[:, :, :1].contiguous(), False, 0.5)
    np.testing.assert_allclose(o1, np.broadcast_to(f64(v[:, :, :1]), o1.shape), rtol=0, atol=1e-15)
    s = 0.5 * np.einsum("bhid,bhd->bhi", f64(q), f64(k[:, :, 0]))
    np.testing.assert_allclose(lse1, s, rtol=0, atol=1e-12)


def test_fully_masked_row_is_zero_and_minus_inf(oracle_mod):
    q = rand_bf16((1, 1, 6, 8), 10)
    k = rand_bf16((1, 1, 4, 8), 11)
    v = rand_bf16((1, 1, 4, 8), 12)
    # causal, Nq > Nkv, bottom-right: row i sees keys j <= i - 2, rows 0,1 see nothing
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 1.0)
    assert np.all(o[0, 0, :2] == 0.0) and np.all(np.isneginf(lse[0, 0, :2]))
    assert np.all(np.isfinite(lse[0, 0, 2:]))
    np.testing.assert_allclose(o[0, 0, 2], f64(v[0, 0, 0]), rtol=0, atol=1e-15)
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 1.0, kv_lens=np.array([0], np.int32))
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------- invariants

def test_causal_row_equals_noncausal_on_prefix(oracle_mod):
    B, H, N, d = 1, 2, 23, 16
    q, k, v = rand_bf16((B, H, N, d), 13), rand_bf16((B, H, N, d), 14), rand_bf16((B, H, N, d), 15)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.25)
    for i in (0, 5, 11, 22):
        oi, li = oracle_mod.attn_fwd(q[:, :, i:i + 1].contiguous(), k[:, :, :i + 1].contiguous(),
                                     v[:, :, :i + 1].contiguous(), False, 0.25)
        np.testing.assert_allclose(o[:, :, i], oi[:, :, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], li[:, :, 0], rtol=0, atol=1e-13)


def test_bottom_right_causal_with_fewer_queries(oracle_mod):
    # Nq < Nkv: query i (of Nq) is the last Nq positions of the key sequence
    q, k, v = rand_bf16((1, 1, 4, 8), 16), rand_bf16((1, 1, 10, 8), 17), rand_bf16((1, 1, 10, 8), 18)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.5)
    for i in range(4):
        n = 10 - 4 + i + 1
        oi, li = oracle_mod.attn_fwd(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                                     v[:, :, :n].contiguous(), False, 0.5)
        np.testing.assert_allclose(o[0, 0, i], oi[0, 0, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], li[0, 0, 0], rtol=0, atol=1e-13)


def test_key_padding_equals_truncated_keys(oracle_mod):
    B, H, N, d = 3, 2, 30, 16
    q, k, v = rand_bf16((B, H, N, d), 19), rand_bf16((B, H, N, d), 20), rand_bf16((B, H, N, d), 21)
    kl = np.array([1, 17, 30], np.int32)
    for causal in (False, True):
        o, lse = oracle_mod.attn_fwd(q, k, v, causal, 0.25, kv_lens=kl)
        for b in range(B):
            n = int(kl[b])
            ob, lb = oracle_mod.attn_fwd(q[b:b + 1], k[b:b + 1, :, :n].contiguous(),
                                         v[b:b + 1, :, :n].contiguous(), False, 0.25)
            if not causal:
                np.testing.assert_allclose(o[b], ob[0], rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[b], lb[0], rtol=0, atol=1e-13)
            else:
                # AND of the masks: rows i < n see keys 0..i; rows i >= n see keys 0..n-1
                oc, lc = oracle_mod.attn_fwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], True, 0.25)
                np.testing.assert_allclose(o[b, :, :n], oc[0, :, :n], rtol=0, atol=1e-13)
                np.testing.assert_allclose(o[b, :, n:], ob[0, :, n:], rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[b, :, n:], lb[0, :, n:], rtol=0, atol=1e-13)


def test_permuting_keys_and_values_together(oracle_mod):
    q, k, v = rand_bf16((2, 2, 12, 16), 22), rand_bf16((2, 2, 31, 16), 23), rand_bf16((2, 2, 31, 16), 24)
    perm = torch.randperm(31, generator=torch.Generator().manual_seed(5))
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 0.25)
    op, lp = oracle_mod.attn_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.25)
    np.testing.assert_allclose(o, op, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lp, rtol=0, atol=1e-13)
    # permuting V alone must change the result (V rows are tied to their keys)
    ov, _ = oracle_mod.attn_fwd(q, k, v[:, :, perm].contiguous(), False, 0.25)
    assert np.abs(ov - o).max() > 1e-3


def test_large_score_shift_is_stable(oracle_mod):
    # k[..., 0] = 1 for every key; moving q[..., 0] from 0 to delta shifts every score by
    # scale*delta: O is unchanged and LSE moves by exactly scale*delta.
    d, delta, scale = 16, 8000.0, 0.125
    q, k, v = rand_bf16((1, 2, 7, d), 25), rand_bf16((1, 2, 11, d), 26), rand_bf16((1, 2, 11, d), 27)
    k[..., 0] = 1.0
    q0 = q.clone(); q0[..., 0] = 0.0
    q1 = q.clone(); q1[..., 0] = delta
    for causal in (False, True):
        o0, l0 = oracle_mod.attn_fwd(q0, k, v, causal, scale)
        o1, l1 = oracle_mod.attn_fwd(q1, k, v, causal, scale)
        assert np.isfinite(o1).all() and np.isfinite(l1).all()
        np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1 - l0, scale * delta, rtol=0, atol=1e-9)


def test_split_kv_merge_identity(oracle_mod):
    # attention over [0,n) == LSE-weighted merge of attention over [0,c) and [c,n)
    q, k, v = rand_bf16((2, 2, 5, 32), 28), rand_bf16((2, 2, 50, 32), 29), rand_bf16((2, 2, 50, 32), 30)
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 0.2)
    c = 19
    o1, l1 = oracle_mod.attn_fwd(q, k[:, :, :c].contiguous(), v[:, :, :c].contiguous(), False, 0.2)
    o2, l2 = oracle_mod.attn_fwd(q, k[:, :, c:].contiguous(), v[:, :, c:].contiguous(), False, 0.2)
    L = np.logaddexp(l1, l2)
    om = (np.exp(l1 - L)[..., None] * o1 + np.exp(l2 - L)[..., None] * o2)
    np.testing.assert_allclose(L, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)


def test_rows_api_matches_full(oracle_mod):
    q, k, v = rand_bf16((2, 3, 20, 16), 31), rand_bf16((2, 3, 26, 16), 32), rand_bf16((2, 3, 26, 16), 33)
    kl = np.array([26, 9], np.int32)
    o, lse = oracle_mod.attn_fwd(q, k, v, True, 0.25, kv_lens=kl)
    rows = [0, 7, 19, 20, 61, 119]
    orow, lrow = oracle_mod.attn_rows(q, k, v, True, 0.25, rows, kv_lens=kl)
    np.testing.assert_array_equal(orow, o.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(lrow, lse.reshape(-1)[rows])


# ----------------------------------------------------------------------------- library case

@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_fp64(oracle_mod, causal):
    # torch's CPU scaled_dot_product_attention in fp64 is an independent implementation
    # of the same definition (top-left causal alignment, equal to ours when Nq == Nkv).
    B, H, N, d = 2, 3, 37, 64
    q, k, v = rand_bf16((B, H, N, d), 34), rand_bf16((B, H, N, d), 35), rand_bf16((B, H, N, d), 36)
    kl = np.array([37, 21], np.int32)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_fwd(q, k, v, causal, scale, kv_lens=kl)
    mask = torch.arange(N)[None, :] < torch.as_tensor(kl, dtype=torch.int64)[:, None]  # [B, Nkv]
    mask = mask[:, None, None, :].expand(B, H, N, N)
    if causal:
        mask = mask & torch.ones(N, N, dtype=torch.bool).tril()
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = (qd @ kd.transpose(-1, -2)) * scale
    ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- paged gather

def test_paged_equals_contiguous(oracle_mod):
    shape = workloads.DecodeShape("t", 5, 3, 32, (1, 70), page_size=16, seed=7)
    inp = workloads.decode_inputs(shape, ctx_lens=[1, 16, 17, 70, 33])
    o, lse = oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                     inp["ctx_lens"], 0.17)
    ps = 16
    for b, n in enumerate(inp["ctx_lens"].tolist()):
        # build the contiguous cache by indexing pages with torch (independent of the oracle)
        pages = inp["page_table"][b, : (n + ps - 1) // ps].long()
        kc = inp["k_pages"][pages].permute(1, 0, 2, 3).reshape(3, -1, 32)[:, :n]
        vc = inp["v_pages"][pages].permute(1, 0, 2, 3).reshape(3, -1, 32)[:, :n]
        oc, lc = oracle_mod.attn_fwd(inp["q"][b][None, :, None].contiguous(), kc[None].contiguous(),
                                     vc[None].contiguous(), False, 0.17)
        np.testing.assert_array_equal(o[b], oc[0, :, 0])
        np.testing.assert_array_equal(lse[b], lc[0, :, 0])
        assert np.abs(o[b]).max() < 100.0  # no poison reached the result


def test_paged_rejects_bad_page_ids(oracle_mod):
    shape = workloads.DecodeShape("t", 2, 1, 8, (1, 20), seed=8)
    inp = workloads.decode_inputs(shape, ctx_lens=[20, 5])
    pt = inp["page_table"].clone()
    pt[0, 1] = 10_000
    with pytest.raises(RuntimeError):
        oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], pt, inp["ctx_lens"], 1.0)


def _torch_masked_attention(q, kc, vc, mask, scale):
    """fp64 attention of query rows q [n, d] over keys kc/vc [m, d] with a boolean mask [n, m],
    written with torch primitives (softmax, logsumexp); rows with no key give 0 and -inf."""
    s = (q.to(torch.float64) @ kc.to(torch.float64).T) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)
    return (p @ vc.to(torch.float64)).numpy(), lse.numpy()


def _unmapped_case(shape_seed, ctx, bad):
    """Decode-layout inputs whose page-table entries listed in ``bad`` ((b, logical page, id))
    point outside the pool."""
    shape = workloads.DecodeShape("t", len(ctx), 4, 32, (1, max(ctx)), seed=shape_seed)
    inp = workloads.decode_inputs(shape, ctx_lens=ctx, kv_heads=2)
    for b, lp, pid in bad:
        inp["page_table"][b, lp] = pid
    return inp


def _mapped_positions(inp, b, n, ps=16):
    P = inp["k_pages"].shape[0]
    ids = inp["page_table"][b].long()
    return torch.tensor([0 <= int(ids[t // ps]) < P for t in range(n)], dtype=torch.bool)


def _gather(pages, inp, b, n, kvh, ps=16):
    """Contiguous [n, d] cache of key/value head kvh by torch indexing; unmapped pages -> 0."""
    P = pages.shape[0]
    ids = inp["page_table"][b].long()
    rows = []
    for t in range(n):
        pid = int(ids[t // ps])
        rows.append(pages[pid, kvh, t % ps] if 0 <= pid < P else torch.zeros_like(pages[0, 0, 0]))
    return torch.stack(rows)


def test_paged_decode_skips_unmapped_pages(oracle_mod):
    # an id past the pool and a negative id inside the context, one at the very start; sequence 2
    # has every page unmapped (no key at all: 0 and -inf)
    ctx = [70, 33, 20]
    inp = _unmapped_case(9, ctx, [(0, 1, 10_000), (0, 3, -1), (1, 0, -7), (2, 0, -1), (2, 1, 999_999)])
    scale = 0.21
    o, lse = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                         inp["ctx_lens"], scale, skip_bad_pages=True)
    with pytest.raises(RuntimeError):
        oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                    scale)
    for b, n in enumerate(ctx):
        keep = _mapped_positions(inp, b, n)
        for h in range(4):
            kc = _gather(inp["k_pages"], inp, b, n, h // 2)
            vc = _gather(inp["v_pages"], inp, b, n, h // 2)
            ro, rl = _torch_masked_attention(inp["q"][b, h][None], kc, vc, keep[None], scale)
            np.testing.assert_allclose(o[b, h], ro[0], rtol=0, atol=1e-12)
            if np.isfinite(rl[0]):
                np.testing.assert_allclose(lse[b, h], rl[0], rtol=0, atol=1e-12)
            else:
                assert lse[b, h] == -np.inf and not o[b, h].any()
    assert lse[2].tolist() == [-np.inf] * 4


@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_skips_unmapped_pages(oracle_mod, causal):
    ctx, Nq = [70, 40], 24
    inp = _unmapped_case(10, ctx, [(0, 2, 55_555), (1, 0, -3)])
    scale = 0.19
    g = torch.Generator().manual_seed(11)
    q = torch.randn(2, 4, Nq, 32, generator=g).to(torch.bfloat16)
    o, lse = oracle_mod.paged_prefill_gqa(q, inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                          causal, scale, skip_bad_pages=True)
    for b, n in enumerate(ctx):
        keep = _mapped_positions(inp, b, n)
        i = torch.arange(Nq)[:, None]
        j = torch.arange(n)[None, :]
        mask = keep[None, :].expand(Nq, n)
        if causal:
            mask = mask & (j <= i + n - Nq)  # bottom-right: query i sits at position n - Nq + i
        for h in range(4):
            kc = _gather(inp["k_pages"], inp, b, n, h // 2)
            vc = _gather(inp["v_pages"], inp, b, n, h // 2)
            ro, rl = _torch_masked_attention(q[b, h], kc, vc, mask, scale)
            np.testing.assert_allclose(o[b, h], ro, rtol=0, atol=1e-12)
            fin = np.isfinite(rl)
            np.testing.assert_allclose(lse[b, h][fin], rl[fin], rtol=0, atol=1e-12)
            assert np.all(lse[b, h][~fin] == -np.inf) and not o[b, h][~fin].any()
    if causal:
        # sequence 1's first page (positions 0-15) is unmapped; its query 0 sits at position 16
        # and still sees the mapped key 16
        assert np.isfinite(lse[1, :, 0]).all()


def test_paged_decode_fp8_skips_unmapped_pages(oracle_mod):
    ctx = [50, 17]
    inp = _unmapped_case(12, ctx, [(0, 1, 1 << 20), (1, 1, -2)])
    kc8 = oracle_mod.e4m3_quantize(inp["k_pages"], 0.5)
    vc8 = oracle_mod.e4m3_quantize(inp["v_pages"], 0.25)
    vals = torch.from_numpy(oracle_mod.e4m3_values())
    scale = 0.3
    o, lse = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc8, vc8, 0.5, 0.25, inp["page_table"], inp["ctx_lens"], scale,
                                             skip_bad_pages=True)
    kd = vals[torch.from_numpy(kc8).long()] * 0.5
    vd = vals[torch.from_numpy(vc8).long()] * 0.25
    for b, n in enumerate(ctx):
        keep = _mapped_positions(inp, b, n)
        for h in range(4):
            kc = _gather(kd, inp, b, n, h // 2)
            vc = _gather(vd, inp, b, n, h // 2)
            ro, rl = _torch_masked_attention(inp["q"][b, h][None], kc, vc, keep[None], scale)
            np.testing.assert_allclose(o[b, h], ro[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], rl[0], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- accounting

def test_flop_formula_reproduces_printed_numbers():
    g = json.load(open(os.path.join(GOLDEN, "flop_accounting.json")))
    f = prefill_flops(1, 1, g["N"], g["N"], g["d"], causal=False)
    assert f == 4 * 2048 * 2048 * 64
    for c in g["cases"]:
        tflops = f / (c["ms"] * 1e-3) / 1e12
        assert round(tflops, 3) == c["tflops_printed"]
    assert prefill_flops(2, 3, 64, 64, 32, True) == 0.5 * prefill_flops(2, 3, 64, 64, 32, False)


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    """Mutation check: a plausible bug planted in a copy of the oracle C source
    (on the CPU) must fail at least one of the pins above."""
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "attn_oracle.c")).read()
    mutants = {
        "no_max_subtraction": ("l += exp(srow[j] - m);", "l += exp(srow[j]);"),
        "causal_off_by_one": ("(long)j > (long)i + (long)Nkv - (long)Nq", "(long)j >= (long)i + (long)Nkv - (long)Nq"),
        "lse_missing_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
        "transposed_v": ("bf16_to_f64(vb[(size_t)j * d + c])", "bf16_to_f64(vb[(size_t)c * d + j % d])"),
    }
    q = rand_bf16((1, 2, 16, 16), 40)
    k = rand_bf16((1, 2, 16, 16), 41)
    v = rand_bf16((1, 2, 16, 16), 42)
    good_o, good_l = oracle_mod.attn_fwd(q, k, v, True, 0.25)
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(a, b, 1))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"],
                       check=True)
        lib = ctypes.CDLL(str(so))
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.oracle_attn_fwd_f64.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, P, I]
        o = np.empty_like(good_o)
        l = np.empty_like(good_l)
        qb, kb, vb = (oracle_mod.bf16_bits(t) for t in (q, k, v))
        lib.oracle_attn_fwd_f64(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, None, 1, 2, 16, 16, 16, 1,
                                0.25, o.ctypes.data, l.ctypes.data, 1)
        # the same closed forms used above: causal query 0 returns v_0 and the torch fp64 reference
        qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True, scale=0.25)
        s = (qd @ kd.transpose(-1, -2)) * 0.25
        ref_l = torch.logsumexp(s.masked_fill(~torch.ones(16, 16, dtype=torch.bool).tril(), float("-inf")), -1)
        assert np.allclose(good_l, ref_l.numpy(), atol=1e-12)
        caught = (not np.allclose(o, ref.numpy(), atol=1e-9)) or (not np.allclose(l, ref_l.numpy(), atol=1e-9))
        assert caught, f"planted mistake {name} not caught"


# ----------------------------------------------------------------------------- grouped-query

@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 1), (4, 4)])
def test_gqa_equals_mha_on_repeated_kv(oracle_mod, Hq, Hkv):
    # grouped-query attention shares each K/V head among Hq/Hkv consecutive query heads:
    # it must equal multi-head attention on K/V repeated along the head axis
    B, N, d = 2, 33, 16
    q = rand_bf16((B, Hq, N, d), 50)
    k = rand_bf16((B, Hkv, N, d), 51)
    v = rand_bf16((B, Hkv, N, d), 52)
    kl = np.array([33, 20], np.int32)
    rep = Hq // Hkv
    for causal in (False, True):
        o, lse = oracle_mod.attn_fwd_gqa(q, k, v, causal, 0.25, kv_lens=kl)
        om, lm = oracle_mod.attn_fwd(q, k.repeat_interleave(rep, dim=1).contiguous(),
                                     v.repeat_interleave(rep, dim=1).contiguous(), causal, 0.25, kv_lens=kl)
        np.testing.assert_array_equal(o, om)
        np.testing.assert_array_equal(lse, lm)


def test_gqa_against_torch_sdpa_fp64(oracle_mod):
    B, Hq, Hkv, N, d = 2, 8, 2, 29, 32
    q, k, v = rand_bf16((B, Hq, N, d), 53), rand_bf16((B, Hkv, N, d), 54), rand_bf16((B, Hkv, N, d), 55)
    o, lse = oracle_mod.attn_fwd_gqa(q, k, v, True, 0.2)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True, scale=0.2, enable_gqa=True)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_paged_gqa_equals_contiguous_gqa(oracle_mod):
    shape = workloads.DecodeShape("t", 3, 8, 16, (1, 70), page_size=16, seed=9)
    inp = workloads.decode_inputs(shape, ctx_lens=[5, 70, 33], kv_heads=2)
    o, lse = oracle_mod.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                         inp["ctx_lens"], 0.3)
    ps = 16
    for b, n in enumerate(inp["ctx_lens"].tolist()):
        pages = inp["page_table"][b, : (n + ps - 1) // ps].long()
        kc = inp["k_pages"][pages].permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
        vc = inp["v_pages"][pages].permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
        oc, lc = oracle_mod.attn_fwd_gqa(inp["q"][b][None, :, None].contiguous(), kc[None].contiguous(),
                                         vc[None].contiguous(), False, 0.3)
        np.testing.assert_array_equal(o[b], oc[0, :, 0])
        np.testing.assert_array_equal(lse[b], lc[0, :, 0])


def test_planted_gqa_head_mapping_mistake_is_caught(oracle_mod, tmp_path):
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "attn_oracle.c")).read()
    a = "int64_t bhkv = (int64_t)b * Hkv + h / group;"
    assert a in src
    path = tmp_path / "m.c"
    path.write_text(src.replace(a, "int64_t bhkv = (int64_t)b * Hkv + h % Hkv;", 1))
    so = tmp_path / "m.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.oracle_attn_gqa_rows_f64.argtypes = [P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double, P, ctypes.c_int64,
                                             P, P, I]
    B, Hq, Hkv, N, d = 1, 8, 2, 12, 16
    q, k, v = rand_bf16((B, Hq, N, d), 56), rand_bf16((B, Hkv, N, d), 57), rand_bf16((B, Hkv, N, d), 58)
    rows = np.arange(B * Hq * N, dtype=np.int64)
    o = np.empty((len(rows), d))
    l = np.empty(len(rows))
    qb, kb, vb = (oracle_mod.bf16_bits(t) for t in (q, k, v))
    lib.oracle_attn_gqa_rows_f64(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, None, B, Hq, Hkv, N, N, d, 0,
                                 0.25, rows.ctypes.data, len(rows), o.ctypes.data, l.ctypes.data, 1)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=0.25, enable_gqa=True)
    assert not np.allclose(o.reshape(B, Hq, N, d), ref.numpy(), atol=1e-6)


# ----------------------------------------------------------------------------- paged prefill

def test_paged_prefill_equals_contiguous_bottom_right(oracle_mod):
    # chunked prefill over the paged cache == the contiguous prefill definition (bottom-right
    # causal, Nkv = ctx_len) run per sequence on the gathered cache
    shape = workloads.DecodeShape("t", 3, 4, 16, (1, 90), page_size=16, seed=11)
    inp = workloads.decode_inputs(shape, ctx_lens=[40, 90, 23], kv_heads=2)
    Nq = 20
    q = rand_bf16((3, 4, Nq, 16), 60)
    for causal in (False, True):
        o, lse = oracle_mod.paged_prefill_gqa(q, inp["k_pages"], inp["v_pages"], inp["page_table"],
                                              inp["ctx_lens"], causal, 0.3)
        ps = 16
        for b, n in enumerate(inp["ctx_lens"].tolist()):
            pages = inp["page_table"][b, : (n + ps - 1) // ps].long()
            kc = inp["k_pages"][pages].permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
            vc = inp["v_pages"][pages].permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
            oc, lc = oracle_mod.attn_fwd_gqa(q[b:b + 1], kc[None].contiguous(), vc[None].contiguous(), causal, 0.3)
            np.testing.assert_array_equal(o[b], oc[0])
            np.testing.assert_array_equal(lse[b], lc[0])


def test_paged_prefill_single_query_is_decode(oracle_mod):
    shape = workloads.DecodeShape("t", 4, 4, 32, (1, 64), page_size=16, seed=12)
    inp = workloads.decode_inputs(shape, ctx_lens=[1, 64, 17, 33])
    q1 = inp["q"][:, :, None].contiguous()
    o, lse = oracle_mod.paged_prefill_gqa(q1, inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                          True, 0.2)
    od, ld = oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                     0.2)
    np.testing.assert_array_equal(o[:, :, 0], od)
    np.testing.assert_array_equal(lse[:, :, 0], ld)


def test_paged_prefill_flop_count_closed_form():
    from attn_fwd_02_gb300.metrics import paged_prefill_flops
    # Nq == ctx (no earlier cache): query i sees i + 1 keys -> 4*d*H*N(N+1)/2
    assert paged_prefill_flops(3, 10, 8, [10]) == 4 * 8 * 3 * 55
    # Nq = 1 is one decode row over all ctx keys
    assert paged_prefill_flops(2, 1, 16, [7, 9]) == 4 * 16 * 2 * (7 + 9)
    # non-causal: every query sees every cached key
    assert paged_prefill_flops(1, 4, 2, [6], causal=False) == 4 * 2 * 4 * 6


def test_paged_prefill_byte_count():
    from attn_fwd_02_gb300.metrics import decode_bytes, paged_prefill_bytes
    # with one query per sequence it moves exactly what a decode step moves
    assert paged_prefill_bytes(4, 1, 64, [17, 300], 16, kv_heads=2) == decode_bytes(4, 64, [17, 300], 16, kv_heads=2)
    # by hand: 2 cache heads x 33 tokens of K and V (bf16), 4 heads x 5 queries of Q and O, LSE, 3 table entries
    assert paged_prefill_bytes(4, 5, 8, [33], 16, kv_heads=2) == 2 * 2 * 8 * 2 * 33 + 2 * 4 * 5 * 8 * 2 + 4 * 4 * 5 + 4 * 3
