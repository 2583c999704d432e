"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by
element, on the same seeded inputs.

Tolerances (stated for this method with N(0,1) inputs): O max-abs <= 1e-2 and
mean-abs <= 1e-3; LSE abs <= 1e-3.  Rows with no valid key must give O = 0 and
LSE = -inf exactly."""
import math

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


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", o_max=O_MAX):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= o_max, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: O mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: -inf pattern of LSE differs"
        d = np.abs(l[~inf_ref] - lse_ref[~inf_ref])
        if d.size:
            assert d.max() <= LSE_MAX, f"{what}: LSE max-abs {d.max():.3e}"
        if inf_ref.any():
            assert np.all(o[inf_ref] == 0.0), f"{what}: fully masked rows must be zero"
    return float(err.max()), float(err.mean())


def run_prefill(lib, shape, kv_lens=None, with_lse=True, inputs=None):
    inp = inputs or workloads.prefill_inputs(shape)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    kl = inp["kv_lens"] if kv_lens is None else torch.tensor(kv_lens, dtype=torch.int32)
    # NaN-filled outputs: every element the kernel should write is checked to be written
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda") if with_lse else None
    if kl is None:
        lib.attn_fwd(q, k, v, shape.causal, shape.scale, out=o, lse=lse, return_lse=with_lse)
    else:
        lib.attn_fwd_kvlen(q, k, v, shape.causal, shape.scale, kv_lens=kl.cuda(), out=o, lse=lse,
                           return_lse=with_lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    return inp, kl, o, lse


SMALL_PREFILL = [
    workloads.TILE_128x64,
    workloads.PrefillShape("ragged 2x3 N300 d64 causal", 2, 3, 300, 300, 64, True, seed=11),
    workloads.PrefillShape("ragged 2x3 N300 d64", 2, 3, 300, 300, 64, False, seed=12),
    workloads.PrefillShape("ragged 2x2 N300 d128 causal", 2, 2, 300, 300, 128, True, seed=13),
    workloads.PrefillShape("ragged 1x2 N260 d128", 1, 2, 260, 260, 128, False, seed=14),
    workloads.PrefillShape("Nq<Nkv causal d128", 1, 2, 200, 457, 128, True, seed=15),
    workloads.PrefillShape("Nq>Nkv causal d64 (masked rows)", 1, 2, 333, 150, 64, True, seed=16),
    workloads.PrefillShape("Nq<Nkv non-causal d64", 2, 1, 77, 515, 64, False, seed=17),
    workloads.PrefillShape("tiny N1", 1, 1, 1, 1, 64, True, seed=18),
    workloads.PrefillShape("tiny N5 d128", 2, 1, 5, 9, 128, False, seed=19),
    workloads.PrefillShape("x0.5 inputs d128 causal", 1, 2, 512, 512, 128, True, value_scale=0.5, seed=20),
    workloads.PrefillShape("scale 1.0: peaked softmax, rescale path", 1, 2, 640, 640, 64, True, seed=21,
                           softmax_scale=1.0),
    workloads.PrefillShape("scale 2.0 d128 non-causal", 1, 2, 384, 384, 128, False, seed=24, softmax_scale=2.0),
    workloads.PrefillShape("key padding 3x2 N384 d64", 3, 2, 384, 384, 64, False, kv_len_range=(1, 384), seed=22),
    workloads.PrefillShape("key padding causal 3x2 N384 d128", 3, 2, 384, 384, 128, True, kv_len_range=(1, 384),
                           seed=23),
]


@pytest.mark.parametrize("shape", SMALL_PREFILL, ids=lambda s: s.name)
def test_prefill_small_vs_oracle(lib, oracle_mod, shape):
    inp, kl, o, lse = run_prefill(lib, shape)
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=kl)
    o_max = O_MAX
    if shape.softmax_scale is not None:
        # Outside the stated conditions (scale 1/sqrt(d)) the softmax can be nearly one-hot;
        # then rounding P to bf16 moves O by up to 2^-9 * max|V| and rounding O by 2^-9 * |O|,
        # so the bound is 2^-8 * max|V|.
        o_max = max(O_MAX, 2.0 ** -8 * float(inp["v"].float().abs().max()))
    compare(o, lse, o_ref, lse_ref, shape.name, o_max=o_max)


GROWING_KEYS = [
    workloads.PrefillShape("growing keys d128 causal", 1, 2, 520, 520, 128, True, seed=25),
    workloads.PrefillShape("growing keys d128 non-causal", 2, 1, 130, 600, 128, False, seed=26),
    workloads.PrefillShape("growing keys d64 causal", 1, 2, 520, 520, 64, True, seed=27),
]


@pytest.mark.parametrize("shape", GROWING_KEYS, ids=lambda s: s.name)
def test_prefill_running_max_jumps(lib, oracle_mod, shape):
    """Key j scaled by 1 + j/16: a row's largest score grows by about 30 (log2 units) from one
    128-key tile to the next, far past the lazy-rescale threshold of 8, so the running maximum,
    the normaliser and O move on most tiles (82-98 % of the fully visible (row, tile) pairs of
    these inputs, counted in fp64 from the scores)."""
    inp = workloads.prefill_inputs(shape)
    grow = 1.0 + torch.arange(shape.Nkv, dtype=torch.float32) / 16.0
    inp["k"] = (inp["k"].float() * grow[:, None]).to(torch.bfloat16)
    inp, kl, o, lse = run_prefill(lib, shape, inputs=inp)
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=kl)
    # the softmax is nearly one-hot here: the bound of the peaked-softmax cases applies
    o_max = max(O_MAX, 2.0 ** -8 * float(inp["v"].float().abs().max()))
    compare(o, lse, o_ref, lse_ref, shape.name, o_max=o_max)


def test_prefill_zero_length_and_full_padding(lib, oracle_mod):
    shape = workloads.PrefillShape("kv_len 0 / 129 / 256", 3, 2, 256, 256, 64, True, seed=30)
    inp, kl, o, lse = run_prefill(lib, shape, kv_lens=[0, 129, 256])
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], True, shape.scale, kv_lens=kl)
    compare(o, lse, o_ref, lse_ref, shape.name)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_prefill_without_lse(lib, oracle_mod):
    shape = workloads.PrefillShape("no lse", 1, 2, 200, 200, 128, True, seed=31)
    inp, kl, o, _ = run_prefill(lib, shape, with_lse=False)
    o_ref, _ = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], True, shape.scale)
    compare(o, None, o_ref, None, shape.name)


def test_prefill_is_deterministic(lib):
    shape = workloads.PrefillShape("determinism", 2, 4, 700, 700, 128, True, seed=32)
    _, _, o1, l1 = run_prefill(lib, shape)
    _, _, o2, l2 = run_prefill(lib, shape)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_guard_regions_untouched(lib):
    # outputs carved out of a larger buffer: the bytes around them must not change
    B, H, N, d = 1, 2, 200, 64
    shape = workloads.PrefillShape("guard", B, H, N, N, d, True, seed=33)
    inp = workloads.prefill_inputs(shape)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    n_o = B * H * N * d
    pad = 4096
    big = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    big_l = torch.full((B * H * N + 2 * pad,), 7.0, device="cuda")
    o = big[pad:pad + n_o].view(B, H, N, d)
    lse = big_l[pad:pad + B * H * N].view(B, H, N)
    lib.attn_fwd(q, k, v, True, shape.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(big[:pad] == 7.0) and torch.all(big[pad + n_o:] == 7.0)
    assert torch.all(big_l[:pad] == 7.0) and torch.all(big_l[pad + B * H * N:] == 7.0)


@pytest.mark.parametrize("shape", [workloads.ENCODER_PAD, workloads.DECODER_CAUSAL], ids=lambda s: s.name)
def test_prefill_full_size_all_rows(lib, oracle_mod, shape):
    inp, kl, o, lse = run_prefill(lib, shape)
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=kl)
    compare(o, lse, o_ref, lse_ref, shape.name)


def test_prefill_long_context_sampled_rows(lib, oracle_mod):
    shape = workloads.LONG_CAUSAL
    inp, kl, o, lse = run_prefill(lib, shape)
    B, H, N, d = shape.B, shape.H, shape.Nq, shape.d
    g = np.random.default_rng(1234)
    rows = np.concatenate([
        g.integers(0, B * H * N, 384),
        [0, N - 1, N, B * H * N - 1, 127, 128, 8191 - 128],  # tile edges
    ]).astype(np.int64)
    o_ref, lse_ref = oracle_mod.attn_rows(inp["q"], inp["k"], inp["v"], True, shape.scale, rows)
    og = o.reshape(-1, d)[torch.as_tensor(rows, device="cuda")]
    lg = lse.reshape(-1)[torch.as_tensor(rows, device="cuda")]
    compare(og, lg, o_ref, lse_ref, shape.name)
    # properties over every row: finite, |O| bounded by max |V|, LSE >= max score lower bound
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert o.abs().max().item() <= inp["v"].abs().max().item() + 1e-2


def test_prefill_long_context_all_rows(lib, oracle_mod):
    # every row of the long-context workload (2 x 32 x 8192 rows of d = 128) against the fp64
    # oracle, element by element: about 1.1e12 oracle FLOPs, half a minute on 16 host cores
    shape = workloads.LONG_CAUSAL
    inp, kl, o, lse = run_prefill(lib, shape)
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], True, shape.scale)
    max_err, mean_err = compare(o, lse, o_ref, lse_ref, shape.name + " (all rows)")
    assert np.isfinite(lse_ref).all()


# ----------------------------------------------------------------------------- paged decode

def run_decode(lib, shape, ctx_lens=None):
    inp = workloads.decode_inputs(shape, ctx_lens=ctx_lens)
    dev = {k: v.cuda() for k, v in inp.items()}
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full(dev["q"].shape[:2], float("nan"), device="cuda")
    lib.paged_attn_decode(dev["q"], dev["k_pages"], dev["v_pages"], dev["page_table"], dev["ctx_lens"],
                          shape.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert lib.attn_check_device_status() == 0
    return inp, o, lse


SMALL_DECODE = [
    (workloads.DecodeShape("d128 short contexts", 5, 3, 128, (1, 70), seed=40), [1, 16, 17, 70, 33]),
    (workloads.DecodeShape("d64 short contexts", 5, 3, 64, (1, 70), seed=41), [2, 15, 31, 64, 49]),
    (workloads.DecodeShape("multi-chunk contexts", 4, 2, 128, (1, 2000), seed=42), [512, 513, 2000, 1023]),
    (workloads.DecodeShape("empty context", 3, 2, 128, (1, 100), seed=43), [0, 100, 1]),
    (workloads.DecodeShape("drawn lengths", 6, 4, 128, (512, 4096), seed=44), None),
    # more chunks (1024 tokens at d = 64, 512 at d = 128) than the merge keeps weights for in
    # shared memory (256) and than it has threads (64 / 128): the merge's strided loops and its
    # recomputed-weight path
    (workloads.DecodeShape("over 256 chunks d64", 2, 2, 64, (1, 280000), seed=46), [280000, 262145]),
    (workloads.DecodeShape("over 256 chunks d128", 1, 1, 128, (1, 131585), seed=47), [131585]),
]


@pytest.mark.parametrize("shape,ctx", SMALL_DECODE, ids=[s[0].name for s in SMALL_DECODE])
def test_decode_small_vs_oracle(lib, oracle_mod, shape, ctx):
    inp, o, lse = run_decode(lib, shape, ctx)
    o_ref, lse_ref = oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                             inp["ctx_lens"], shape.scale)
    compare(o, lse, o_ref, lse_ref, shape.name)


def test_decode_full_size_vs_oracle(lib, oracle_mod):
    shape = workloads.PAGED_DECODE
    inp, o, lse = run_decode(lib, shape)
    o_ref, lse_ref = oracle_mod.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
                                             inp["ctx_lens"], shape.scale)
    compare(o, lse, o_ref, lse_ref, shape.name)


def test_decode_equals_contiguous_prefill(lib):
    # the paged result equals a contiguous-cache attention of the same tokens (recipe 03's claim)
    shape = workloads.DecodeShape("paged vs contiguous", 2, 4, 128, (1, 700), seed=45)
    inp, o, lse = run_decode(lib, shape, [700, 300])
    ps = 16
    for b, n in enumerate(inp["ctx_lens"].tolist()):
        pages = inp["page_table"][b, :(n + ps - 1) // ps].long()
        kc = inp["k_pages"][pages].permute(1, 0, 2, 3).reshape(4, -1, 128)[:, :n]
        vc = inp["v_pages"][pages].permute(1, 0, 2, 3).reshape(4, -1, 128)[:, :n]
        oc, lc = lib.attn_fwd(inp["q"][b][None, :, None].contiguous().cuda(), kc[None].contiguous().cuda(),
                              vc[None].contiguous().cuda(), False, shape.scale)
        torch.cuda.synchronize()
        assert (oc[0, :, 0].float() - o[b].float()).abs().max().item() <= 1e-2
        assert (lc[0, :, 0] - lse[b]).abs().max().item() <= 1e-3
