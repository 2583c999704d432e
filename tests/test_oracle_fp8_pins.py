"""Pins for the FP8 (E4M3) part of the oracle: the code table against hand-worked values of the
format's definition, the rounding (nearest, ties to even, saturating) against a brute-force
search and hand-made ties, and the FP8 paged decode against the pinned bf16 decode through
exact identities.  Every test here runs on the CPU."""
import json
import os
import subprocess

import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_table_hand_values(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))
    v = oracle_mod.e4m3_values()
    for code, want in g["values"].items():
        assert v[int(code)] == want and np.signbit(v[int(code)]) == np.signbit(want), code
    for code in g["nan_codes"]:
        assert np.isnan(v[code])
    assert np.isnan(v).sum() == 2


def test_e4m3_table_structure(oracle_mod):
    v = oracle_mod.e4m3_values()
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0..126 increase strictly
    np.testing.assert_array_equal(v[0x80:0xFF], -pos)  # sign bit mirrors
    # every e4m3 value is a bf16 value (3 mantissa bits, exponents within bf16's range)
    fin = v[np.isfinite(v)]
    assert np.array_equal(torch.tensor(fin).to(torch.bfloat16).double().numpy(), fin)


def test_e4m3_rounding_is_nearest_ties_even_saturating(oracle_mod):
    v = oracle_mod.e4m3_values()
    pos = v[:0x7F]
    # round trip of every finite non-negative code
    for c in range(0x7F):
        assert oracle_mod.e4m3_code(pos[c]) == c
        if c:
            assert oracle_mod.e4m3_code(-pos[c]) == 0x80 | c
    # exact midpoints go to the code with an even mantissa
    for c in range(0x7E):
        mid = (pos[c] + pos[c + 1]) / 2
        assert np.float32(mid) == mid
        assert oracle_mod.e4m3_code(mid) == (c if c % 2 == 0 else c + 1)
    # brute force on random fp32 values
    rng = np.random.default_rng(0)
    ys = np.concatenate([rng.standard_normal(2000) * s for s in (0.01, 1, 30, 300)]).astype(np.float32)
    for y in ys:
        c = oracle_mod.e4m3_code(y)
        a = abs(float(y))
        if a > 448:
            assert c & 0x7F == 0x7E
            continue
        err = np.abs(pos - a)
        assert err[c & 0x7F] == err.min()
        assert (c >> 7) == (1 if y < 0 else 0) or (c & 0x7F) == 0
    assert oracle_mod.e4m3_code(1e9) == 0x7E and oracle_mod.e4m3_code(-500.0) == 0xFE
    # signed zero: -0 and negatives that round to zero keep the sign bit
    assert oracle_mod.e4m3_code(-0.0) == 0x80 and oracle_mod.e4m3_code(-1e-6) == 0x80
    assert oracle_mod.e4m3_code(0.0) == 0x00


@pytest.mark.parametrize("scale", [1.0, 0.37, 6.0 / 448])
def test_quantize_equals_code_of_the_scaled_value(oracle_mod, scale):
    # the bulk quantiser is code(fp32(x) * fp32(1/scale)) for every finite bf16 x
    bits = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    codes = oracle_mod.e4m3_quantize(x, scale)
    inv = np.float32(1.0) / np.float32(scale)
    xs = x.float().numpy()
    with np.errstate(over="ignore"):  # products past the fp32 range become inf and saturate
        for xi, c in zip(xs, codes):
            assert c == oracle_mod.e4m3_code(np.float32(xi) * inv)


def test_quantize_applies_the_fp32_inverse_scale(oracle_mod):
    x = torch.tensor([1.0, -2.0, 0.0078125, 100.0, 3.0e4]).to(torch.bfloat16)
    codes = oracle_mod.e4m3_quantize(x, 0.5)  # x * 2
    v = oracle_mod.e4m3_values()
    # 200 lies halfway between 192 (mantissa 4) and 208 (mantissa 5): ties go to the even mantissa
    np.testing.assert_array_equal(v[codes], [2.0, -4.0, 0.015625, 192.0, 448.0])


def _fp8_case(seed=5, B=4, H=8, Hkv=2, d=64, ctx=(37, 300, 16, 129)):
    shape = workloads.DecodeShape("fp8", B, H, d, (1, max(ctx)), seed=seed)
    inp = workloads.decode_inputs(shape, ctx_lens=list(ctx), kv_heads=Hkv)
    return shape, inp


def test_fp8_decode_with_unit_scales_equals_bf16_decode(oracle_mod):
    # e4m3 values are bf16 values: decoding codes at scale 1 is the bf16 decode of those values
    shape, inp = _fp8_case()
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], 1.0)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], 1.0)
    table = oracle_mod.e4m3_values()
    kb = torch.tensor(table[kc]).to(torch.bfloat16)
    vb = torch.tensor(table[vc]).to(torch.bfloat16)
    o8, l8 = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc, vc, 1.0, 1.0, inp["page_table"], inp["ctx_lens"],
                                             shape.scale)
    ob, lb = oracle_mod.paged_decode_gqa(inp["q"], kb, vb, inp["page_table"], inp["ctx_lens"], shape.scale)
    np.testing.assert_allclose(o8, ob, atol=1e-13)
    np.testing.assert_allclose(l8, lb, atol=1e-13)


def test_fp8_scales_fold_into_score_scale_and_output(oracle_mod):
    # k_scale multiplies every score (= a larger softmax scale); v_scale multiplies O and not LSE
    shape, inp = _fp8_case(seed=6)
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], 0.05)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], 0.05)
    args = (inp["page_table"], inp["ctx_lens"])
    o1, l1 = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc, vc, 1.0, 1.0, *args, shape.scale * 0.25)
    o2, l2 = oracle_mod.paged_decode_fp8_gqa(inp["q"], kc, vc, 0.25, 3.0, *args, shape.scale)
    np.testing.assert_allclose(o2, 3.0 * o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)


def _fp8_prefill_case(seed=7, B=3, H=4, Hkv=2, d=32, ctx=(40, 150, 17), Nq=24):
    shape = workloads.DecodeShape("fp8 prefill", B, H, d, (1, max(ctx)), seed=seed)
    inp = workloads.decode_inputs(shape, ctx_lens=list(ctx), kv_heads=Hkv)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    return shape, inp, q


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_paged_prefill_with_unit_scales_equals_bf16_paged_prefill(oracle_mod, causal):
    # e4m3 values are bf16 values: the chunked prefill over codes at scale 1 is the bf16 chunked
    # prefill of those values (same masks, same order of operations: equal to the last bit)
    shape, inp, q = _fp8_prefill_case()
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], 0.5)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], 0.5)
    table = oracle_mod.e4m3_values()
    kb = torch.tensor(table[kc]).to(torch.bfloat16)
    vb = torch.tensor(table[vc]).to(torch.bfloat16)
    o8, l8 = oracle_mod.paged_prefill_fp8_gqa(q, kc, vc, 1.0, 1.0, inp["page_table"], inp["ctx_lens"], causal,
                                              shape.scale)
    ob, lb = oracle_mod.paged_prefill_gqa(q, kb, vb, inp["page_table"], inp["ctx_lens"], causal, shape.scale)
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)


def test_fp8_paged_prefill_scales_fold_into_score_scale_and_output(oracle_mod):
    shape, inp, q = _fp8_prefill_case(seed=8)
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], 0.05)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], 0.05)
    args = (inp["page_table"], inp["ctx_lens"], True)
    o1, l1 = oracle_mod.paged_prefill_fp8_gqa(q, kc, vc, 1.0, 1.0, *args, shape.scale * 0.25)
    o2, l2 = oracle_mod.paged_prefill_fp8_gqa(q, kc, vc, 0.25, 3.0, *args, shape.scale)
    np.testing.assert_allclose(o2, 3.0 * o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)


def test_fp8_paged_prefill_against_torch_fp64(oracle_mod):
    # the definition over the dequantised cache, written with torch primitives and an explicit
    # bottom-right causal mask (a library special case, independent of the oracle's gather)
    shape, inp, q = _fp8_prefill_case(seed=9, d=64)
    ks, vs = 0.04, 0.02
    kc = oracle_mod.e4m3_quantize(inp["k_pages"], ks)
    vc = oracle_mod.e4m3_quantize(inp["v_pages"], vs)
    o, lse = oracle_mod.paged_prefill_fp8_gqa(q, kc, vc, ks, vs, inp["page_table"], inp["ctx_lens"], True,
                                              shape.scale)
    vals = torch.from_numpy(oracle_mod.e4m3_values())
    kd = vals[torch.from_numpy(kc).long()] * ks
    vd = vals[torch.from_numpy(vc).long()] * vs
    Nq = q.shape[2]
    for b, n in enumerate(inp["ctx_lens"].tolist()):
        pages = inp["page_table"][b, :(n + 15) // 16].long()
        for h in range(q.shape[1]):
            kvh = h // 2
            kk = kd[pages, kvh].reshape(-1, 64)[:n]
            vv = vd[pages, kvh].reshape(-1, 64)[:n]
            s_ = (q[b, h].to(torch.float64) @ kk.T) * shape.scale
            mask = torch.arange(n)[None, :] <= torch.arange(Nq)[:, None] + n - Nq
            s_ = s_.masked_fill(~mask, float("-inf"))
            ref_l = torch.logsumexp(s_, -1)
            ref_o = torch.softmax(s_, -1).nan_to_num(0.0) @ vv
            fin = torch.isfinite(ref_l).numpy()
            np.testing.assert_allclose(o[b, h], ref_o.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h][fin], ref_l.numpy()[fin], rtol=0, atol=1e-12)
            assert np.all(lse[b, h][~fin] == -np.inf)


def test_planted_fp8_mistakes_are_caught(oracle_mod, tmp_path):
    """A plausible bug planted in a copy of the oracle C source must fail the pins above."""
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "attn_oracle.c")).read()
    g = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))
    mutants = {
        "bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
        "subnormal_2^-10": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
        "ties_odd": ("(c & 1) == 0)", "(c & 1) == 1)"),
        "sign_dropped": ("return (uint8_t)((signbit(y) ? 0x80 : 0) | best);", "return (uint8_t)best;"),
    }
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(a, b, 1))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"], check=True)
        lib = ctypes.CDLL(str(so))
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_code.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_code.restype = ctypes.c_uint8
        table_ok = all(lib.oracle_e4m3_value(int(c)) == w for c, w in g["values"].items())
        ties_ok = lib.oracle_e4m3_code(1.0625) == 0x38 and lib.oracle_e4m3_code(1.1875) == 0x3A
        sat_ok = lib.oracle_e4m3_code(1e6) == 0x7E and lib.oracle_e4m3_code(-1.0) == 0xB8
        assert not (table_ok and ties_ok and sat_ok), f"planted mistake {name} not caught"
