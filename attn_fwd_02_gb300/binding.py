"""ctypes binding of the C ABI declared in include/attn_gb300.h.

Argument marshalling only: shapes are read off the torch tensors, pointers and
the current CUDA stream are handed to the library, and a non-zero status
raises ``AttnError``.  Every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the shared library has not been built
(``__graft_entry__.build()`` or ``python -m attn_fwd_02_gb300.build``), every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libattn_gb300.so"
_lib = None
_lock = threading.Lock()

ATTN_OK = 0
_STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_CUDA", 6: "ATTN_ERR_DEVICE_TIMEOUT", 7: "ATTN_ERR_SCRATCH_LIMIT",
}

# name -> (restype, argtypes); mirrors include/attn_gb300.h
P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (I, [P, P, P, P, P, I, I, I, I, I, I, F, P]),
    "attn_fwd_kvlen": (I, [P, P, P, P, P, I, I, I, I, I, I, F, P, P]),
    "attn_fwd_gqa": (I, [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P]),
    "paged_attn_decode_workspace_size": (Z, [I, I, I, I, I]),
    "paged_attn_decode_workspace_size_ctx": (Z, [I, I, I, I]),
    "paged_attn_decode_gqa_workspace_size": (Z, [I, I, I, I, I, I]),
    "paged_attn_decode": (I, [P, P, P, P, P, I, P, P, I, I, I, I, I, F, P, Z, P]),
    "paged_attn_decode_noalloc": (I, [P, P, P, P, P, I, P, P, I, I, I, I, I, F, P]),
    "paged_attn_decode_gqa": (I, [P, P, P, P, P, I, P, P, I, I, I, I, I, I, F, P, Z, P]),
    "paged_attn_prefill": (I, [P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, I, F, P]),
    "paged_kv_append": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, P]),
    "attn_bwd_workspace_size": (Z, [I, I, I]),
    "paged_attn_decode_fp8": (I, [P, P, P, F, F, P, P, I, P, P, I, I, I, I, I, I, F, P, Z, P]),
    "kv_quantize_fp8": (I, [P, P, Z, F, P]),
    "paged_attn_prefill_fp8": (I, [P, P, P, F, F, P, P, I, P, P, I, I, I, I, I, I, I, I, F, P]),
    "paged_kv_append_fp8": (I, [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, P]),
    "attn_bwd": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, Z, P]),
    "attn_check_device_status": (I, [P]),
    "attn_last_device_status": (I, []),
    "attn_selftest_bounded_wait": (I, [P]),
    "attn_status_string": (ctypes.c_char_p, [I]),
    "attn_version": (ctypes.c_char_p, []),
}


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {_STATUS_NAMES.get(status, status)} ({text})")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, LIB_NAME)


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{LIB_NAME} is not built; run `python -m attn_fwd_02_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnError(fn, status, attn_status_string(status))


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require(t, name, dtype, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _out_like(out, like, name):
    """``out`` given by the caller must match ``like`` (dtype, shape, device) and be contiguous;
    None allocates one with torch."""
    import torch
    if out is None:
        return torch.empty_like(like)
    _require(out, name, like.dtype, like.dim())
    if tuple(out.shape) != tuple(like.shape) or out.device != like.device:
        raise ValueError(f"{name} must be {tuple(like.shape)} on {like.device}, got {tuple(out.shape)} "
                         f"on {out.device}")
    return out


def _lse_out(lse, shape, device, want: bool):
    """fp32 log-sum-exp output of the given shape on ``device``: checked if given, allocated
    if None and wanted."""
    import torch
    if lse is None:
        return torch.empty(shape, dtype=torch.float32, device=device) if want else None
    _require(lse, "lse", torch.float32, len(shape))
    if tuple(lse.shape) != tuple(shape) or lse.device != device:
        raise ValueError(f"lse must be {tuple(shape)} on {device}, got {tuple(lse.shape)} on {lse.device}")
    return lse


def attn_fwd_kvlen(q, k, v, causal: bool, scale: float | None = None, kv_lens=None,
                   out=None, lse=None, return_lse: bool = True, stream=None):
    """Prefill attention. q [B,H,Nq,d], k/v [B,H,Nkv,d] bf16 CUDA tensors;
    kv_lens optional int32 [B] CUDA tensor.  Returns (o, lse)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16, 4)
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if tuple(k.shape) != (B, H, Nkv, d) or tuple(v.shape) != (B, H, Nkv, d):
        raise ValueError("k and v must be [B, H, Nkv, d] matching q")
    if kv_lens is not None:
        _require(kv_lens, "kv_lens", torch.int32, 1)
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H, Nq), q.device, return_lse)
    lib = load_library()
    st = lib.attn_fwd_kvlen(_dptr(q), _dptr(k), _dptr(v), _dptr(out), _dptr(lse), B, H, Nq, Nkv, d,
                            int(bool(causal)), float(scale), _dptr(kv_lens), _stream_ptr(stream))
    _check("attn_fwd_kvlen", st)
    return out, lse


def attn_fwd_gqa(q, k, v, causal: bool, scale: float | None = None, kv_lens=None, out=None, lse=None,
                 return_lse: bool = True, stream=None):
    """Grouped-query prefill: q [B,Hq,Nq,d], k/v [B,Hkv,Nkv,d] bf16 CUDA tensors with
    Hq % Hkv == 0 (query head h reads key/value head h // (Hq // Hkv)).  Returns (o, lse)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16, 4)
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nkv, d) or tuple(v.shape) != (B, Hkv, Nkv, d):
        raise ValueError("k and v must be [B, Hkv, Nkv, d] matching q")
    if kv_lens is not None:
        _require(kv_lens, "kv_lens", torch.int32, 1)
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, Hq, Nq), q.device, return_lse)
    st = load_library().attn_fwd_gqa(_dptr(q), _dptr(k), _dptr(v), _dptr(out), _dptr(lse), B, Hq, Hkv, Nq, Nkv,
                                     d, int(bool(causal)), float(scale), _dptr(kv_lens), _stream_ptr(stream))
    _check("attn_fwd_gqa", st)
    return out, lse


def kv_quantize_fp8(x, scale: float, out=None, stream=None):
    """bf16 CUDA tensor -> uint8 e4m3 codes of the same shape under a per-tensor scale
    (value = e4m3(code) * scale; code = nearest-even e4m3 of fp32(x) * fp32(1/scale), saturating)."""
    import torch
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous bf16 CUDA tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    else:
        _require(out, "out", torch.uint8, x.dim())
        if tuple(out.shape) != tuple(x.shape) or out.device != x.device:
            raise ValueError("out must be a uint8 tensor of x's shape on x's device")
    st = load_library().kv_quantize_fp8(_dptr(x), _dptr(out), x.numel(), float(scale), _stream_ptr(stream))
    _check("kv_quantize_fp8", st)
    return out


def paged_kv_append_fp8(k_new, v_new, k_pages, v_pages, k_scale: float, v_scale: float, page_table, start_pos,
                        stream=None):
    """paged_kv_append into an e4m3 cache (k_pages/v_pages uint8 [P,Hkv,16,d]); new K/V bf16
    [B,Hkv,Nnew,d] are converted with the cache's scales."""
    import torch
    _require(k_new, "k_new", torch.bfloat16, 4)
    _require(v_new, "v_new", torch.bfloat16, 4)
    _require(k_pages, "k_pages", torch.uint8, 4)
    _require(v_pages, "v_pages", torch.uint8, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(start_pos, "start_pos", torch.int32, 1)
    B, Hkv, Nnew, d = k_new.shape
    P, Hk, ps, dk = k_pages.shape
    if (Hk, dk) != (Hkv, d) or tuple(v_new.shape) != tuple(k_new.shape) or tuple(v_pages.shape) != tuple(
            k_pages.shape):
        raise ValueError("shape mismatch between new K/V and the pages")
    st = load_library().paged_kv_append_fp8(_dptr(k_new), _dptr(v_new), _dptr(k_pages), _dptr(v_pages),
                                            float(k_scale), float(v_scale), _dptr(page_table), _dptr(start_pos), ps,
                                            B, Hkv, Nnew, d, page_table.shape[1], P, _stream_ptr(stream))
    _check("paged_kv_append_fp8", st)


def paged_attn_decode_fp8(q, k_pages, v_pages, k_scale: float, v_scale: float, page_table, ctx_lens,
                          scale: float | None = None, out=None, lse=None, workspace=None, return_lse: bool = True,
                          stream=None):
    """Paged decode over an e4m3 cache: q [B,H,d] bf16; k_pages/v_pages uint8 codes [P,Hkv,16,d]
    with per-tensor scales.  Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(k_pages, "k_pages", torch.uint8, 4)
    _require(v_pages, "v_pages", torch.uint8, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, d = q.shape
    P, Hkv, ps, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages and v_pages must be [num_pages, Hkv, page_size, d]")
    if scale is None:
        scale = d ** -0.5
    max_pages = page_table.shape[1]
    lib = load_library()
    need = int(lib.paged_attn_decode_gqa_workspace_size(B, H, Hkv, d, max_pages, ps))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H), q.device, return_lse)
    st = lib.paged_attn_decode_fp8(_dptr(q), _dptr(k_pages), _dptr(v_pages), float(k_scale), float(v_scale),
                                   _dptr(page_table), _dptr(ctx_lens), ps, _dptr(out), _dptr(lse), B, H, Hkv, d,
                                   max_pages, P, float(scale), _dptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("paged_attn_decode_fp8", st)
    return out, lse


def attn_bwd_workspace_size(B: int, Hq: int, Nq: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, Hq, Nq))


def attn_bwd(q, k, v, o, lse, dout, causal: bool, scale: float | None = None, kv_lens=None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_fwd_gqa: q, o, dout [B,Hq,Nq,d] and k, v [B,Hkv,Nkv,d] bf16 CUDA tensors,
    lse [B,Hq,Nq] fp32 from the forward; causal, scale and kv_lens as in the forward call.
    Returns (dq, dk, dv) bf16.  The workspace (uint8, attn_bwd_workspace_size bytes) ends up
    holding the row term D [B,Hq,Nq] fp32."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _require(t, n, torch.bfloat16, 4)
    _require(lse, "lse", torch.float32, 3)
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nkv, d) or tuple(v.shape) != (B, Hkv, Nkv, d):
        raise ValueError("k and v must be [B, Hkv, Nkv, d] matching q")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("o and dout must match q, lse must be [B, Hq, Nq]")
    if kv_lens is not None:
        _require(kv_lens, "kv_lens", torch.int32, 1)
    if scale is None:
        scale = d ** -0.5
    dq = _out_like(dq, q, "dq")
    dk = _out_like(dk, k, "dk")
    dv = _out_like(dv, v, "dv")
    lib = load_library()
    need = int(lib.attn_bwd_workspace_size(B, Hq, Nq))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = lib.attn_bwd(_dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse), _dptr(dout), _dptr(dq), _dptr(dk),
                      _dptr(dv), B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)), float(scale), _dptr(kv_lens),
                      _dptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("attn_bwd", st)
    return dq, dk, dv


def attn_fwd(q, k, v, causal: bool, scale: float | None = None, out=None, lse=None,
             return_lse: bool = True, stream=None):
    """Prefill attention without key padding (calls the C entry point attn_fwd)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16, 4)
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if tuple(k.shape) != (B, H, Nkv, d) or tuple(v.shape) != (B, H, Nkv, d):
        raise ValueError("k and v must be [B, H, Nkv, d] matching q")
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H, Nq), q.device, return_lse)
    lib = load_library()
    st = lib.attn_fwd(_dptr(q), _dptr(k), _dptr(v), _dptr(out), _dptr(lse), B, H, Nq, Nkv, d,
                      int(bool(causal)), float(scale), _stream_ptr(stream))
    _check("attn_fwd", st)
    return out, lse


def paged_attn_decode_workspace_size(B: int, H: int, d: int, max_pages_per_seq: int,
                                     page_size: int = 16) -> int:
    return int(load_library().paged_attn_decode_workspace_size(B, H, d, max_pages_per_seq, page_size))


def paged_attn_decode_workspace_size_ctx(B: int, H: int, d: int, max_ctx_len: int) -> int:
    return int(load_library().paged_attn_decode_workspace_size_ctx(B, H, d, max_ctx_len))


def paged_attn_decode_gqa_workspace_size(B: int, H: int, Hkv: int, d: int, max_pages_per_seq: int,
                                         page_size: int = 16) -> int:
    return int(load_library().paged_attn_decode_gqa_workspace_size(B, H, Hkv, d, max_pages_per_seq, page_size))


def paged_attn_decode(q, k_pages, v_pages, page_table, ctx_lens, scale: float | None = None,
                      out=None, lse=None, workspace=None, return_lse: bool = True, stream=None):
    """Paged decode. q [B,H,d]; k_pages/v_pages [P,H,page_size,d] bf16; page_table
    [B,max_pages] int32; ctx_lens [B] int32 (all CUDA).  ``workspace``: optional uint8
    CUDA tensor of at least paged_attn_decode_workspace_size() bytes (allocated with torch
    here if not given).  Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, d = q.shape
    num_pages, Hk, page_size, dk = k_pages.shape
    if (Hk, dk) != (H, d) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages must be [num_pages, H, page_size, d] matching q")
    if page_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages] and ctx_lens [B]")
    max_pages = page_table.shape[1]
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H), q.device, return_lse)
    lib = load_library()
    need = int(lib.paged_attn_decode_workspace_size(B, H, d, max_pages, page_size))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = lib.paged_attn_decode(_dptr(q), _dptr(k_pages), _dptr(v_pages), _dptr(page_table),
                               _dptr(ctx_lens), page_size, _dptr(out), _dptr(lse), B, H, d,
                               max_pages, num_pages, float(scale), _dptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("paged_attn_decode", st)
    return out, lse


def paged_attn_decode_gqa(q, k_pages, v_pages, page_table, ctx_lens, scale: float | None = None,
                          out=None, lse=None, workspace=None, return_lse: bool = True, stream=None):
    """Grouped-query paged decode: q [B,H,d]; k_pages/v_pages [P,Hkv,page_size,d] with
    H % Hkv == 0; page_table [B,max_pages] int32; ctx_lens [B] int32.  Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, d = q.shape
    num_pages, Hkv, page_size, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages must be [num_pages, Hkv, page_size, d] matching q")
    if page_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages] and ctx_lens [B]")
    max_pages = page_table.shape[1]
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H), q.device, return_lse)
    lib = load_library()
    need = int(lib.paged_attn_decode_gqa_workspace_size(B, H, Hkv, d, max_pages, page_size))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = lib.paged_attn_decode_gqa(_dptr(q), _dptr(k_pages), _dptr(v_pages), _dptr(page_table), _dptr(ctx_lens),
                                   page_size, _dptr(out), _dptr(lse), B, H, Hkv, d, max_pages, num_pages,
                                   float(scale), _dptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream_ptr(stream))
    _check("paged_attn_decode_gqa", st)
    return out, lse


def paged_attn_decode_noalloc(q, k_pages, v_pages, page_table, ctx_lens, scale: float | None = None,
                              out=None, lse=None, return_lse: bool = True, stream=None):
    """paged_attn_decode without a workspace, for callers that cannot allocate device
    memory: the library keeps the chunk partials in its own fixed 12 MiB device array.
    Pass ``out`` (bf16, q's shape) and ``lse`` (fp32 [B, H]), both contiguous on q's device,
    to avoid any allocation here as well.  Calls that may overlap on the GPU share that
    array and must be ordered by the caller.
    Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, d = q.shape
    num_pages, Hk, page_size, dk = k_pages.shape
    if (Hk, dk) != (H, d) or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages must be [num_pages, H, page_size, d] matching q")
    if page_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages] and ctx_lens [B]")
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H), q.device, return_lse)
    st = load_library().paged_attn_decode_noalloc(
        _dptr(q), _dptr(k_pages), _dptr(v_pages), _dptr(page_table), _dptr(ctx_lens), page_size, _dptr(out),
        _dptr(lse), B, H, d, page_table.shape[1], num_pages, float(scale), _stream_ptr(stream))
    _check("paged_attn_decode_noalloc", st)
    return out, lse


def paged_attn_prefill(q, k_pages, v_pages, page_table, ctx_lens, causal: bool, scale: float | None = None,
                       out=None, lse=None, return_lse: bool = True, stream=None):
    """Chunked prefill over the paged cache: q [B,H,Nq,d] are the last Nq of the ctx_lens[b]
    cached tokens of each sequence; k_pages/v_pages [P,Hkv,page_size,d]; page_table
    [B,max_pages] int32; ctx_lens [B] int32 (all CUDA).  Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 4)
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, Nq, d = q.shape
    num_pages, Hkv, page_size, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages must be [num_pages, Hkv, page_size, d] matching q")
    if page_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages] and ctx_lens [B]")
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H, Nq), q.device, return_lse)
    st = load_library().paged_attn_prefill(_dptr(q), _dptr(k_pages), _dptr(v_pages), _dptr(page_table),
                                           _dptr(ctx_lens), page_size, _dptr(out), _dptr(lse), B, H, Hkv, Nq, d,
                                           page_table.shape[1], num_pages, int(bool(causal)), float(scale),
                                           _stream_ptr(stream))
    _check("paged_attn_prefill", st)
    return out, lse


def paged_attn_prefill_fp8(q, k_pages, v_pages, k_scale: float, v_scale: float, page_table, ctx_lens,
                           causal: bool, scale: float | None = None, out=None, lse=None, return_lse: bool = True,
                           stream=None):
    """paged_attn_prefill over an e4m3 cache: q [B,H,Nq,d] bf16; k_pages/v_pages uint8 codes
    [P,Hkv,16,d] with per-tensor scales (value = e4m3(code) * scale).  Returns (o, lse)."""
    import torch
    _require(q, "q", torch.bfloat16, 4)
    _require(k_pages, "k_pages", torch.uint8, 4)
    _require(v_pages, "v_pages", torch.uint8, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(ctx_lens, "ctx_lens", torch.int32, 1)
    B, H, Nq, d = q.shape
    num_pages, Hkv, page_size, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages/v_pages must be [num_pages, Hkv, page_size, d] matching q")
    if page_table.shape[0] != B or ctx_lens.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages] and ctx_lens [B]")
    if scale is None:
        scale = d ** -0.5
    out = _out_like(out, q, "out")
    lse = _lse_out(lse, (B, H, Nq), q.device, return_lse)
    st = load_library().paged_attn_prefill_fp8(_dptr(q), _dptr(k_pages), _dptr(v_pages), float(k_scale),
                                               float(v_scale), _dptr(page_table), _dptr(ctx_lens), page_size,
                                               _dptr(out), _dptr(lse), B, H, Hkv, Nq, d, page_table.shape[1],
                                               num_pages, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check("paged_attn_prefill_fp8", st)
    return out, lse


def paged_kv_append(k_new, v_new, k_pages, v_pages, page_table, start_pos, stream=None) -> None:
    """Write new tokens' K/V ([B,Hkv,Nnew,d] bf16) into the pages at positions start_pos[b] + t."""
    import torch
    _require(k_new, "k_new", torch.bfloat16, 4)
    _require(v_new, "v_new", torch.bfloat16, 4)
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(page_table, "page_table", torch.int32, 2)
    _require(start_pos, "start_pos", torch.int32, 1)
    B, Hkv, Nnew, d = k_new.shape
    num_pages, Hk, page_size, dk = k_pages.shape
    if (Hk, dk) != (Hkv, d) or tuple(v_new.shape) != tuple(k_new.shape) or tuple(v_pages.shape) != tuple(
            k_pages.shape):
        raise ValueError("shape mismatch between new K/V and the pages")
    st = load_library().paged_kv_append(_dptr(k_new), _dptr(v_new), _dptr(k_pages), _dptr(v_pages),
                                        _dptr(page_table), _dptr(start_pos), page_size, B, Hkv, Nnew, d,
                                        page_table.shape[1], num_pages, _stream_ptr(stream))
    _check("paged_kv_append", st)


def attn_selftest_bounded_wait(stream=None) -> None:
    """Launch the bounded-wait self-test kernel (its wait runs out after about 2 s)."""
    _check("attn_selftest_bounded_wait", load_library().attn_selftest_bounded_wait(_stream_ptr(stream)))


def attn_check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status word."""
    return int(load_library().attn_check_device_status(_stream_ptr(stream)))


def attn_last_device_status() -> int:
    """The current device's host-visible timeout flag, without synchronising or clearing."""
    return int(load_library().attn_last_device_status())
