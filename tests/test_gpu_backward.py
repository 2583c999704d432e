"""Backward parity on the GPU: attn_bwd (dQ, dK, dV and the row term D) against the fp64 oracle.

The backward's o and lse inputs are the oracle's forward output rounded to the kernel's storage
types (bf16, fp32), so the comparison isolates the backward; a second test chains the GPU
forward into the GPU backward.  Tolerances (per output tensor X, relative to the reference's
own magnitude): mean |X - ref| <= 2^-7 mean |ref| and max |X - ref| <= 2^-5 max |ref|.  Each
gradient is a sum of products in which one factor was rounded to bf16 (P or dS, unit roundoff
2^-9, RMS error 2^-9/sqrt(3) per term), plus the bf16 rounding of the output itself: the
expected mean relative error is about 1.5e-3, and 2^-7 leaves a factor 5.  Keys past a
sequence's length and rows that see no key must be exactly zero."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL_MEAN = 2.0 ** -7
TOL_MAX = 2.0 ** -5


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def compare(name, got, ref):
    got = got.float().cpu().double().numpy()
    err = np.abs(got - ref)
    mean_ref, max_ref = np.abs(ref).mean(), np.abs(ref).max()
    assert err.mean() <= TOL_MEAN * mean_ref + 1e-7, f"{name}: mean err {err.mean():.3e} vs mean |ref| {mean_ref:.3e}"
    assert err.max() <= TOL_MAX * max_ref + 1e-6, f"{name}: max err {err.max():.3e} vs max |ref| {max_ref:.3e}"
    return err.mean() / max(mean_ref, 1e-30), err.max() / max(max_ref, 1e-30)


def make_case(B, Hq, Hkv, Nq, Nkv, d, seed, value_scale=1.0):
    q = rand_bf16((B, Hq, Nq, d), seed, value_scale)
    k = rand_bf16((B, Hkv, Nkv, d), seed + 1, value_scale)
    v = rand_bf16((B, Hkv, Nkv, d), seed + 2)
    do = rand_bf16((B, Hq, Nq, d), seed + 3)
    return q, k, v, do


CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal, kv_lens
    (1, 2, 2, 128, 128, 128, False, None),          # one tile
    (1, 2, 2, 300, 300, 64, False, None),           # ragged tail
    (1, 2, 2, 300, 300, 128, True, None),
    (2, 4, 2, 200, 333, 128, True, None),           # GQA, bottom-right causal, Nq < Nkv
    (2, 2, 2, 256, 256, 64, True, [256, 100]),      # key padding
    (2, 2, 1, 260, 130, 64, True, None),            # Nq > Nkv: the first rows see no key
    (3, 2, 2, 140, 140, 128, False, [0, 140, 77]),  # a sequence with no keys at all
    (1, 4, 4, 1024, 1024, 128, True, None),         # several tiles each way
    (1, 8, 1, 384, 384, 64, True, None),            # multi-query
    # head dims 32, 80, 96: tiles padded to 64 / 128 columns, dQ split 16 / 16, 48 / 32, 48 / 48
    (1, 2, 2, 300, 300, 32, True, None),
    (2, 4, 2, 200, 333, 80, True, [333, 150]),
    (1, 2, 2, 260, 260, 96, False, None),
    (2, 3, 3, 384, 384, 80, True, None),
    (1, 4, 1, 256, 256, 32, False, [200]),
    (1, 2, 2, 140, 140, 96, True, [0]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}/{c[2]}N{c[3]}x{c[4]}d{c[5]}{'c' if c[6] else ''}"
                                             f"{'kl' if c[7] else ''}" for c in CASES])
def test_backward_matches_oracle(oracle_mod, case):
    import attn_fwd_02_gb300 as A
    B, Hq, Hkv, Nq, Nkv, d, causal, kl = case
    q, k, v, do = make_case(B, Hq, Hkv, Nq, Nkv, d, 7000 + Nq + d)
    scale = d ** -0.5
    kl_t = None if kl is None else torch.tensor(kl, dtype=torch.int32)
    ref = oracle_mod.attn_bwd_gqa(q, k, v, do, causal, scale, kv_lens=kl_t)
    o_in = torch.from_numpy(ref["o"]).to(torch.bfloat16)
    lse_in = torch.from_numpy(ref["lse"]).to(torch.float32)
    dev = lambda t: t.cuda()
    ws = torch.empty(max(A.attn_bwd_workspace_size(B, Hq, Nq), 16), dtype=torch.uint8, device="cuda")
    dq, dk, dv = A.attn_bwd(dev(q), dev(k), dev(v), dev(o_in), dev(lse_in), dev(do), causal, scale,
                            kv_lens=None if kl_t is None else dev(kl_t), workspace=ws)
    torch.cuda.synchronize()
    assert A.attn_check_device_status() == 0
    # the row term: D_i = dO_i . O_i over the bf16 output, fp32 accumulation of d products
    D_ref = oracle_mod.bwd_rowdot(o_in, do)
    D_gpu = ws[:B * Hq * Nq * 4].view(torch.float32).cpu().double().numpy().reshape(B, Hq, Nq)
    bound = 1e-5 * (np.abs(o_in.double().numpy()) * np.abs(do.double().numpy())).sum(-1) + 1e-6
    assert np.all(np.abs(D_gpu - D_ref) <= bound)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, got, ref[name])
    # exact zeros where nothing contributes
    if kl is not None:
        for b, n in enumerate(kl):
            assert torch.all(dk[b, :, n:] == 0) and torch.all(dv[b, :, n:] == 0)
            if n == 0:
                assert torch.all(dq[b] == 0)
    if causal and Nq > Nkv:
        assert torch.all(dq[:, :, :Nq - Nkv] == 0)


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False), (32, True), (80, True), (96, False)])
def test_forward_then_backward_matches_oracle(oracle_mod, d, causal):
    import attn_fwd_02_gb300 as A
    B, H, N = 2, 4, 520
    q, k, v, do = make_case(B, H, H, N, N, d, 8100 + d)
    scale = d ** -0.5
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = A.attn_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    assert A.attn_check_device_status() == 0
    ref = oracle_mod.attn_bwd_gqa(q, k, v, do, causal, scale)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, got, ref[name])


def test_backward_full_size_long_context_one_head(oracle_mod):
    """The long-context causal workload (B=2, H=32, N=8192, d=128, inputs x0.5) in the launch
    configuration the benchmark times; every gradient of one head checked against the oracle
    run on that head's slice (heads are independent)."""
    import attn_fwd_02_gb300 as A
    from attn_fwd_02_gb300 import workloads
    s = workloads.LONG_CAUSAL
    inp = workloads.prefill_inputs(s)
    q, k, v = inp["q"], inp["k"], inp["v"]
    do = workloads.backward_upstream(s)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = A.attn_fwd(qd, kd, vd, s.causal, s.scale)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, s.causal, s.scale)
    torch.cuda.synchronize()
    assert A.attn_check_device_status() == 0
    b, h = 1, 17
    sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
    ref = oracle_mod.attn_bwd_gqa(sl(q), sl(k), sl(v), sl(do), s.causal, s.scale)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, got[b:b + 1, h:h + 1], ref[name])
