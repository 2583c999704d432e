"""Host-only checks of the C-ABI library: it loads without a GPU, exports every
function include/attn_gb300.h declares, and rejects bad arguments before
touching the device.  No test here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from attn_fwd_02_gb300 import build as buildmod
    from attn_fwd_02_gb300 import binding
    buildmod.build()
    return binding.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_kvlen", "paged_attn_decode", "paged_attn_decode_workspace_size",
              "attn_check_device_status", "attn_status_string", "attn_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_signatures_cover_the_header():
    from attn_fwd_02_gb300 import binding
    assert set(binding.SIGNATURES) == set(declared_functions())


def test_status_strings(lib):
    from attn_fwd_02_gb300 import binding
    for code in range(7):
        assert binding.attn_status_string(code)
    assert binding.attn_status_string(99) == "unknown status"
    assert lib.attn_version().decode().count(".") == 2


def test_workspace_size(lib):
    ws = lib.paged_attn_decode_workspace_size
    # 32 x 32 heads, 512 pages of 16 tokens -> 16 chunks of 512 tokens, (d + 4) floats each
    assert ws(32, 32, 128, 512, 16) == 32 * 32 * 16 * (128 + 4) * 4
    assert ws(1, 1, 64, 1, 16) == 1 * 1 * 1 * (64 + 4) * 4
    assert ws(0, 1, 64, 1, 16) == 0
    assert ws(1, 1, 96, 1, 16) == 1 * 1 * 1 * (96 + 4) * 4
    assert ws(3, 2, 80, 33, 16) == 3 * 2 * 1 * (80 + 4) * 4  # 528 tokens: one 1024-token split at d = 80
    assert ws(3, 2, 96, 33, 16) == 3 * 2 * 1 * (96 + 4) * 4
    assert ws(3, 2, 128, 33, 16) == 3 * 2 * 2 * (128 + 4) * 4  # two 512-token splits at d = 128
    assert ws(1, 1, 32, 129, 16) == 3 * (32 + 4) * 4  # 2064 tokens: three 1024-token splits at d = 32
    assert ws(1, 1, 48, 1, 16) == 0  # not a supported head dim
    assert ws(1, 1, 64, 1, 32) == 0


def test_workspace_size_by_context_length(lib):
    ws, ws_ctx = lib.paged_attn_decode_workspace_size, lib.paged_attn_decode_workspace_size_ctx
    # the longest context in 16-token pages: 8192 tokens = 512 pages; 8193 needs a 513th page
    assert ws_ctx(32, 32, 128, 8192) == ws(32, 32, 128, 512, 16)
    assert ws_ctx(32, 32, 128, 8193) == ws(32, 32, 128, 513, 16)
    assert ws_ctx(2, 3, 64, 1) == ws(2, 3, 64, 1, 16)
    assert ws_ctx(1, 1, 64, 0) == 0
    assert ws_ctx(1, 1, 64, -16) == 0


def test_grouped_query_workspace_size(lib):
    ws, ws_g = lib.paged_attn_decode_workspace_size, lib.paged_attn_decode_gqa_workspace_size
    # groups of an even number of query heads use 1024-token splits: 8 of them over 8192 tokens
    assert ws_g(32, 32, 8, 128, 512, 16) == 32 * 32 * 8 * (128 + 4) * 4
    assert ws_g(32, 32, 8, 128, 512, 16) * 2 == ws(32, 32, 128, 512, 16)
    assert ws_g(4, 6, 2, 64, 3, 16) == 4 * 6 * 1 * (64 + 4) * 4  # 48 tokens: one split
    # odd groups and multi-head attention keep the 512-token splits
    assert ws_g(2, 9, 3, 64, 100, 16) == ws(2, 9, 64, 100, 16)
    assert ws_g(2, 8, 8, 128, 100, 16) == ws(2, 8, 128, 100, 16)
    assert ws_g(2, 8, 3, 128, 100, 16) == 0  # 8 % 3 != 0
    assert ws_g(2, 8, 0, 128, 100, 16) == 0


def test_last_device_status_without_synchronising(lib):
    # no device here: the set-up fails and says so; on a GPU machine a clean device reads ATTN_OK
    import torch
    st = lib.attn_last_device_status()
    assert st == (0 if torch.cuda.is_available() else 5)


ALIGNED = 1 << 20  # fake, 16-byte aligned addresses: the checks below fail before any use


def call_fwd(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=None, B=1, H=1, Nq=128, Nkv=128, d=64,
             causal=0, scale=0.125, kv_lens=None):
    return lib.attn_fwd_kvlen(q, k, v, o, lse, B, H, Nq, Nkv, d, causal, scale, kv_lens, None)


def test_prefill_argument_checks(lib):
    assert call_fwd(lib, q=None) == 1
    assert call_fwd(lib, o=None) == 1
    assert call_fwd(lib, B=0) == 1
    assert call_fwd(lib, Nkv=-5) == 1
    assert call_fwd(lib, causal=2) == 1
    assert call_fwd(lib, scale=0.0) == 1
    assert call_fwd(lib, scale=-1.0) == 1
    assert call_fwd(lib, scale=float("nan")) == 1
    assert call_fwd(lib, scale=float("inf")) == 1
    assert call_fwd(lib, d=48) == 2
    assert call_fwd(lib, d=16) == 2
    assert call_fwd(lib, d=192) == 2
    assert call_fwd(lib, q=ALIGNED + 8) == 3
    assert call_fwd(lib, o=ALIGNED + 2) == 3
    assert call_fwd(lib, lse=ALIGNED + 2) == 3
    assert call_fwd(lib, B=1 << 16, H=1 << 16) == 1  # B*H beyond the grid
    assert lib.attn_fwd(None, ALIGNED, ALIGNED, ALIGNED, None, 1, 1, 1, 1, 64, 0, 0.1, None) == 1


def call_bwd(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, do=ALIGNED, dq=ALIGNED, dk=ALIGNED,
             dv=ALIGNED, B=1, Hq=2, Hkv=1, Nq=128, Nkv=128, d=64, causal=1, scale=0.125, kv_lens=None, ws=ALIGNED,
             wsb=1 << 20):
    return lib.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, causal, scale, kv_lens, ws, wsb,
                        None)


def test_backward_argument_checks(lib):
    assert lib.attn_bwd_workspace_size(2, 4, 100) == 2 * 4 * 100 * 4 + 256 - (2 * 4 * 100 * 4) % 256
    assert lib.attn_bwd_workspace_size(0, 4, 100) == 0
    for name in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv"):
        assert call_bwd(lib, **{name: None}) == 1, name
    assert call_bwd(lib, Hkv=3) == 1
    assert call_bwd(lib, causal=5) == 1
    assert call_bwd(lib, scale=float("nan")) == 1
    assert call_bwd(lib, d=48) == 2
    assert call_bwd(lib, d=112) == 2
    for name in ("q", "o", "do", "dq", "dk", "dv"):
        assert call_bwd(lib, **{name: ALIGNED + 8}) == 3, name
    assert call_bwd(lib, lse=ALIGNED + 2) == 3
    assert call_bwd(lib, ws=None) == 4
    assert call_bwd(lib, ws=ALIGNED + 4) == 4
    assert call_bwd(lib, wsb=lib.attn_bwd_workspace_size(1, 2, 128) - 1) == 4


def test_fp8_argument_checks(lib):
    q = ALIGNED
    # decode over an e4m3 cache: the decode checks plus positive, finite cache scales
    dec = lambda **kw: lib.paged_attn_decode_fp8(
        kw.get("q", q), ALIGNED, ALIGNED, kw.get("ks", 0.1), kw.get("vs", 0.1), ALIGNED, ALIGNED, 16, ALIGNED, None,
        2, kw.get("H", 2), kw.get("Hkv", 2), kw.get("d", 128), 4, 8, 0.1, kw.get("ws", ALIGNED), 1 << 20, None)
    assert dec(q=None) == 1
    assert dec(ks=0.0) == 1 and dec(vs=float("inf")) == 1 and dec(ks=float("nan")) == 1
    assert dec(Hkv=3) == 1
    assert dec(d=48) == 2 and dec(d=160) == 2
    assert dec(q=ALIGNED + 4) == 3
    assert dec(ws=None) == 4
    assert lib.kv_quantize_fp8(None, ALIGNED, 64, 1.0, None) == 1
    assert lib.kv_quantize_fp8(ALIGNED, ALIGNED, 12, 1.0, None) == 1  # not a multiple of 8
    assert lib.kv_quantize_fp8(ALIGNED, ALIGNED, 64, -1.0, None) == 1
    assert lib.kv_quantize_fp8(ALIGNED + 8, ALIGNED, 64, 1.0, None) == 3
    app = lambda **kw: lib.paged_kv_append_fp8(ALIGNED, ALIGNED, ALIGNED, ALIGNED, kw.get("ks", 1.0), 1.0,
                                               kw.get("pt", ALIGNED), ALIGNED, 16, 1, 1, 4, kw.get("d", 64), 4, 8,
                                               None)
    assert app(pt=None) == 1 and app(ks=0.0) == 1 and app(d=48) == 2 and app(d=256) == 2


def call_dec(lib, q=ALIGNED, kp=ALIGNED, vp=ALIGNED, pt=ALIGNED, cl=ALIGNED, ps=16, o=ALIGNED, lse=None,
             B=2, H=2, d=128, maxp=4, npages=8, scale=0.1, ws=ALIGNED, wsb=1 << 20):
    return lib.paged_attn_decode(q, kp, vp, pt, cl, ps, o, lse, B, H, d, maxp, npages, scale, ws, wsb, None)


def test_decode_argument_checks(lib):
    assert call_dec(lib, pt=None) == 1
    assert call_dec(lib, cl=None) == 1
    assert call_dec(lib, B=0) == 1
    assert call_dec(lib, npages=0) == 1
    assert call_dec(lib, scale=0.0) == 1
    assert call_dec(lib, d=48) == 2
    assert call_dec(lib, d=256) == 2
    assert call_dec(lib, ps=32) == 2
    assert call_dec(lib, kp=ALIGNED + 4) == 3
    assert call_dec(lib, pt=ALIGNED + 2) == 3
    assert call_dec(lib, ws=None) == 4
    assert call_dec(lib, ws=ALIGNED + 4) == 4
    need = lib.paged_attn_decode_workspace_size(2, 2, 128, 4, 16)
    assert call_dec(lib, wsb=need - 1) == 4
    assert call_dec(lib, B=70000) == 1


def test_binding_rejects_cpu_tensors():
    import torch

    from attn_fwd_02_gb300 import binding
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        binding.attn_fwd(q, q, q, causal=False)
    with pytest.raises(TypeError):
        binding.attn_fwd(q.float(), q, q, causal=False)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from attn_fwd_02_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_HERE", str(tmp_path))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "attn_fwd_02_gb300")
    pat = re.compile(r"(import\s+oracle|from\s+oracle|liboracle|attn_oracle)")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f


def test_grouped_query_argument_checks(lib):
    gqa = lambda Hq=4, Hkv=2, **kw: lib.attn_fwd_gqa(
        kw.get("q", ALIGNED), ALIGNED, ALIGNED, ALIGNED, None, 1, Hq, Hkv, 128, 128, kw.get("d", 64), 1, 0.125, None,
        None)
    assert gqa(Hkv=3) == 1  # query heads not a multiple of the key/value heads
    assert gqa(Hkv=0) == 1
    assert gqa(Hq=2, Hkv=4) == 1
    assert gqa(d=48) == 2
    assert gqa(q=ALIGNED + 8) == 3
    dec = lambda H=4, Hkv=2, **kw: lib.paged_attn_decode_gqa(
        ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 16, ALIGNED, None, 2, H, Hkv, kw.get("d", 128), 4, 8, 0.1,
        kw.get("ws", ALIGNED), 1 << 20, None)
    assert dec(Hkv=3) == 1
    assert dec(Hkv=-1) == 1
    assert dec(d=112) == 2
    assert dec(ws=None) == 4


def test_paged_prefill_and_append_argument_checks(lib):
    pre = lambda **kw: lib.paged_attn_prefill(
        ALIGNED, ALIGNED, ALIGNED, kw.get("pt", ALIGNED), kw.get("cl", ALIGNED), kw.get("ps", 16),
        kw.get("o", ALIGNED), None, 1, kw.get("H", 4), kw.get("Hkv", 2), kw.get("Nq", 64), kw.get("d", 128),
        kw.get("maxp", 8), kw.get("npages", 16), 1, kw.get("scale", 0.1), None)
    assert pre(pt=None) == 1 and pre(cl=None) == 1 and pre(o=None) == 1
    assert pre(Nq=0) == 1 and pre(maxp=0) == 1 and pre(npages=0) == 1
    assert pre(Hkv=3) == 1
    assert pre(scale=float("nan")) == 1
    assert pre(maxp=1 << 27) == 1  # capacity past 2^30 tokens
    assert pre(ps=32) == 2 and pre(d=48) == 2
    assert pre(pt=ALIGNED + 2) == 3 and pre(cl=ALIGNED + 1) == 3 and pre(o=ALIGNED + 8) == 3
    app = lambda **kw: lib.paged_kv_append(
        kw.get("kn", ALIGNED), ALIGNED, kw.get("kp", ALIGNED), ALIGNED, kw.get("pt", ALIGNED), kw.get("sp", ALIGNED),
        kw.get("ps", 16), 1, 2, kw.get("n", 4), kw.get("d", 96), 4, 8, None)
    assert app(kn=None) == 1 and app(pt=None) == 1 and app(sp=None) == 1
    assert app(n=0) == 1
    assert app(d=48) == 2 and app(ps=8) == 2
    assert app(kn=ALIGNED + 8) == 3 and app(kp=ALIGNED + 4) == 3 and app(sp=ALIGNED + 2) == 3


def test_paged_prefill_fp8_argument_checks(lib):
    pre = lambda **kw: lib.paged_attn_prefill_fp8(
        kw.get("q", ALIGNED), ALIGNED, ALIGNED, kw.get("ks", 0.1), kw.get("vs", 0.1), kw.get("pt", ALIGNED), ALIGNED,
        kw.get("ps", 16), ALIGNED, None, 2, 4, kw.get("Hkv", 2), kw.get("n", 64), kw.get("d", 128), 4, 8, 1, 0.1, None)
    assert pre(pt=None) == 1
    assert pre(ks=0.0) == 1 and pre(vs=float("nan")) == 1 and pre(ks=-1.0) == 1
    assert pre(Hkv=3) == 1 and pre(n=0) == 1
    assert pre(ps=32) == 2 and pre(d=48) == 2
    assert pre(q=ALIGNED + 4) == 3
