"""Pins for the backward oracle (gradients of exact attention): a hand-worked example, central
finite differences of the oracle's own forward, fp64 autograd of plain attention written with
torch ops, invariants the softmax Jacobian fixes, and planted mistakes that the pins must catch.
Every test here runs on the CPU."""
import json
import os
import subprocess

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand64(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64) * scale


def rand_bf16(shape, seed, scale=1.0):
    return rand64(shape, seed, scale).to(torch.bfloat16)


def key_mask(B, Nq, Nkv, causal, kv_lens):
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nkv)[None, :]
    m = torch.ones(B, 1, Nq, Nkv, dtype=torch.bool)
    if causal:
        m = m & (j <= i + Nkv - Nq)
    if kv_lens is not None:
        m = m & (j[None, None] < torch.as_tensor(kv_lens)[:, None, None, None])
    return m


def torch_grads(q, k, v, do, causal, scale, kv_lens=None):
    """fp64 autograd through softmax(scale q k^T, masked) v; rows without a valid key give 0."""
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    qq, kk, vv = (t.detach().to(torch.float64).clone().requires_grad_() for t in (q, k, v))
    kr = kk.repeat_interleave(Hq // Hkv, 1)
    vr = vv.repeat_interleave(Hq // Hkv, 1)
    s = (qq @ kr.transpose(-1, -2)) * scale
    mask = key_mask(B, Nq, Nkv, causal, kv_lens)
    rows_ok = mask.any(-1, keepdim=True)
    s = torch.where(rows_ok, s.masked_fill(~mask, float("-inf")), torch.zeros_like(s))
    p = torch.softmax(s, -1) * rows_ok
    o = p @ vr
    o.backward(do.to(torch.float64))
    return qq.grad.numpy(), kk.grad.numpy(), vv.grad.numpy(), o.detach().numpy()


# ----------------------------------------------------------------------------- hand-worked

@pytest.mark.parametrize("key,causal", [("noncausal", False), ("causal", True)])
def test_hand_worked_gradients(oracle_mod, key, causal):
    g = json.load(open(os.path.join(GOLDEN, "tiny_hand_bwd.json")))
    t = lambda x: torch.tensor(x, dtype=torch.float64).reshape(1, 1, 2, 2)
    r = oracle_mod.attn_bwd_gqa(t(g["q"]).numpy(), t(g["k"]).numpy(), t(g["v"]).numpy(), t(g["do"]).numpy(),
                                causal, g["scale"])
    want = g[key]
    np.testing.assert_allclose(r["dq"][0, 0], np.array(want["dq_over_scale"]) * g["scale"], atol=1e-14)
    np.testing.assert_allclose(r["dk"][0, 0], np.array(want["dk_over_scale"]) * g["scale"], atol=1e-14)
    np.testing.assert_allclose(r["dv"][0, 0], np.array(want["dv"]), atol=1e-14)
    np.testing.assert_allclose(r["D"][0, 0], np.array(want["D"]), atol=1e-14)


def test_rowdot_hand_worked(oracle_mod):
    # D = dO . O: [1,2].[3,4] = 11 and [0.5,-1].[2,2] = -1 (exact in bf16)
    o = torch.tensor([[3.0, 4.0], [2.0, 2.0]]).to(torch.bfloat16)
    do = torch.tensor([[1.0, 2.0], [0.5, -1.0]]).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle_mod.bwd_rowdot(o, do), [11.0, -1.0])


# ----------------------------------------------------------------------------- finite differences

FD_CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal, kv_lens
    (1, 2, 2, 4, 4, 3, False, None),
    (1, 2, 2, 5, 5, 3, True, None),
    (2, 2, 1, 3, 6, 3, True, [6, 4]),      # bottom-right causal, key padding, GQA
    (1, 4, 2, 6, 4, 2, True, None),        # Nq > Nkv: the first two rows see no key
]


@pytest.mark.parametrize("case", FD_CASES)
def test_central_finite_differences(oracle_mod, case):
    """dL/dx for L = sum(dO * O(q, k, v)) by central differences of the oracle's forward output
    must equal the analytic gradients (h = 1e-6: truncation ~h^2, rounding ~1e-16/h)."""
    B, Hq, Hkv, Nq, Nkv, d, causal, kl = case
    q = rand64((B, Hq, Nq, d), 1).numpy()
    k = rand64((B, Hkv, Nkv, d), 2).numpy()
    v = rand64((B, Hkv, Nkv, d), 3).numpy()
    do = rand64((B, Hq, Nq, d), 4).numpy()
    kl_arr = None if kl is None else np.array(kl, np.int32)
    scale = 0.7
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, causal, scale, kv_lens=kl_arr)

    def loss(qx, kx, vx):
        return float((oracle_mod.attn_bwd_gqa(qx, kx, vx, do, causal, scale, kv_lens=kl_arr)["o"] * do).sum())

    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(x)
        flat = x.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + h
            lp = loss(q, k, v)
            flat[idx] = old - h
            lm = loss(q, k, v)
            flat[idx] = old
            num.reshape(-1)[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(r[name], num, atol=2e-8, rtol=1e-6, err_msg=name)


def test_oracle_forward_part_equals_forward_oracle(oracle_mod):
    # the o and lse the backward oracle recomputes are the pinned forward oracle's, on bf16 inputs
    q = rand_bf16((2, 4, 37, 16), 5)
    k = rand_bf16((2, 2, 45, 16), 6)
    v = rand_bf16((2, 2, 45, 16), 7)
    do = rand_bf16((2, 4, 37, 16), 8)
    kl = torch.tensor([45, 30], dtype=torch.int32)
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, True, 0.25, kv_lens=kl)
    o, lse = oracle_mod.attn_fwd_gqa(q, k, v, True, 0.25, kv_lens=kl)
    np.testing.assert_allclose(r["o"], o, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(r["lse"]), np.isinf(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(r["lse"][fin], lse[fin], atol=1e-13)


# ----------------------------------------------------------------------------- library special case

@pytest.mark.parametrize("causal,kl,Hq,Hkv", [(False, None, 4, 4), (True, None, 4, 4), (True, [70, 33], 4, 2),
                                              (False, [9, 70], 6, 1)])
def test_against_torch_autograd_fp64(oracle_mod, causal, kl, Hq, Hkv):
    B, Nq, Nkv, d = 2, 53, 70, 16
    q = rand_bf16((B, Hq, Nq, d), 10)
    k = rand_bf16((B, Hkv, Nkv, d), 11)
    v = rand_bf16((B, Hkv, Nkv, d), 12)
    do = rand_bf16((B, Hq, Nq, d), 13)
    kl_t = None if kl is None else torch.tensor(kl, dtype=torch.int32)
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, causal, 0.25, kv_lens=kl_t)
    gq, gk, gv, o = torch_grads(q, k, v, do, causal, 0.25, kv_lens=kl)
    np.testing.assert_allclose(r["dq"], gq, atol=1e-12)
    np.testing.assert_allclose(r["dk"], gk, atol=1e-12)
    np.testing.assert_allclose(r["dv"], gv, atol=1e-12)
    np.testing.assert_allclose(r["o"], o, atol=1e-12)


# ----------------------------------------------------------------------------- invariants

def test_softmax_jacobian_invariants(oracle_mod):
    """Rows of dS sum to zero, so the dK of one head sums to zero over keys; rows of P sum to
    one, so the dV of one head sums to the dO of the rows that see a key; D_i = dO_i . O_i."""
    B, Hq, Hkv, Nq, Nkv, d = 2, 4, 2, 40, 24, 8
    q, k, v, do = (rand_bf16(s, 20 + i) for i, s in enumerate(
        [(B, Hq, Nq, d), (B, Hkv, Nkv, d), (B, Hkv, Nkv, d), (B, Hq, Nq, d)]))
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, True, 0.3)  # Nq > Nkv: rows 0..15 see no key
    np.testing.assert_allclose(r["dk"].sum(axis=2), 0.0, atol=1e-12)
    dod = do.to(torch.float64).numpy()
    seen = dod[:, :, Nq - Nkv:, :].sum(axis=2)  # rows with at least one key, per query head
    want_dv = seen.reshape(B, Hkv, Hq // Hkv, d).sum(axis=2)
    np.testing.assert_allclose(r["dv"].sum(axis=2), want_dv, atol=1e-12)
    np.testing.assert_allclose(r["D"], (dod * r["o"]).sum(-1), atol=1e-12)
    assert np.all(r["dq"][:, :, :Nq - Nkv] == 0.0)


def test_constant_values_give_zero_score_gradients(oracle_mod):
    # every v_j equal: O does not depend on the scores, so dQ = dK = 0 and dV_j = sum_i P_ij dO_i
    B, H, N, d = 1, 2, 20, 8
    q, k, do = rand_bf16((B, H, N, d), 30), rand_bf16((B, H, N, d), 31), rand_bf16((B, H, N, d), 32)
    v = torch.full((B, H, N, d), 1.5).to(torch.bfloat16)
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, True, 0.5)
    assert np.abs(r["dq"]).max() < 1e-13 and np.abs(r["dk"]).max() < 1e-13


def test_fully_padded_sequence_has_zero_gradients(oracle_mod):
    B, H, N, d = 2, 2, 12, 4
    q, k, v, do = (rand_bf16((B, H, N, d), 40 + i) for i in range(4))
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, False, 0.5, kv_lens=np.array([0, 12], np.int32))
    for n in ("dq", "dk", "dv"):
        assert np.all(r[n][0] == 0.0)
        assert np.abs(r[n][1]).max() > 0


def test_rowdot_of_rounded_output_is_within_bf16_rounding(oracle_mod):
    # D computed from the bf16-rounded O differs from the exact D by at most 2^-8 sum |dO||O|
    q, k, v, do = (rand_bf16((1, 2, 64, 32), 50 + i) for i in range(4))
    r = oracle_mod.attn_bwd_gqa(q, k, v, do, True, 32 ** -0.5)
    o_bf = torch.from_numpy(r["o"]).to(torch.bfloat16)
    Dr = oracle_mod.bwd_rowdot(o_bf, do)
    bound = 2.0 ** -8 * (np.abs(do.to(torch.float64).numpy()) * np.abs(r["o"])).sum(-1)
    assert np.all(np.abs(Dr - r["D"]) <= bound + 1e-15)


# ----------------------------------------------------------------------------- planted mistakes

def test_planted_backward_mistakes_are_caught(oracle_mod, tmp_path):
    """Mutation check: a plausible bug planted in a copy of the oracle C source (on the CPU) must
    fail the fp64 autograd comparison above."""
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "attn_oracle.c")).read()
    mutants = {
        "dropped_D": ("const double dS = P[j] * (dP[j] - Di);", "const double dS = P[j] * dP[j];"),
        "dk_times_k": ("dkb[(size_t)j * d + c] += scale * dS * qi[c];",
                       "dkb[(size_t)j * d + c] += scale * dS * kb[(size_t)j * d + c];"),
        "dv_from_dS": ("dvb[(size_t)j * d + c] += P[j] * doi[c];", "dvb[(size_t)j * d + c] += dS * doi[c];"),
        "dq_unscaled": ("dqi[c] += scale * dS * kb[(size_t)j * d + c];", "dqi[c] += dS * kb[(size_t)j * d + c];"),
        "gqa_interleaved": ("const int h = g * group + hh;", "const int h = g + hh * Hkv;"),
    }
    B, Hq, Hkv, Nq, Nkv, d = 1, 4, 2, 9, 11, 4
    q, k, v, do = (rand_bf16(s, 60 + i) for i, s in enumerate(
        [(B, Hq, Nq, d), (B, Hkv, Nkv, d), (B, Hkv, Nkv, d), (B, Hq, Nq, d)]))
    gq, gk, gv, _ = torch_grads(q, k, v, do, True, 0.5)
    f = lambda t: np.ascontiguousarray(t.to(torch.float64).numpy())
    qd, kd, vd, dod = f(q), f(k), f(v), f(do)
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(a, b, 1))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"], check=True)
        lib = ctypes.CDLL(str(so))
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.oracle_attn_bwd_gqa_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double,
                                                P, P, P, P, P, P, I]
        dq, dk, dv = np.empty_like(qd), np.empty_like(kd), np.empty_like(vd)
        lib.oracle_attn_bwd_gqa_f64(qd.ctypes.data, kd.ctypes.data, vd.ctypes.data, dod.ctypes.data, None, B, Hq,
                                    Hkv, Nq, Nkv, d, 1, 0.5, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, None,
                                    None, None, 1)
        caught = not (np.allclose(dq, gq, atol=1e-9) and np.allclose(dk, gk, atol=1e-9)
                      and np.allclose(dv, gv, atol=1e-9))
        assert caught, f"planted mistake {name} not caught"
