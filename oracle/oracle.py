"""fp64 CPU oracle for exact attention (prefill) and paged-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this module.  The product
path (the ``attn_fwd_02_gb300`` package and its CUDA library) never imports,
loads or calls anything here, and this module imports nothing from the
product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over query
rows); this file compiles it with gcc and marshals arrays through ctypes.
What it computes is the plain three-pass definition of attention:

    s_j   = scale * q_i . k_j            over the valid keys J of row i
    O_i   = sum_J exp(s_j - m) v_j / sum_J exp(s_j - m),   m = max_J s_j
    LSE_i = m + ln sum_J exp(s_j - m)

with J the keys that survive the key-padding mask and, if causal, the
bottom-right causal mask j <= i + Nkv - Nq.  FlashAttention is stated on the
pages to reach exactly this result without materialising the score matrix
(NanoInfer README, Flash Attention bullets; inference-kernel-cookbook README,
recipe 01).  The paged form gathers pages through the page table into a
contiguous cache and applies the same definition (inference-kernel-cookbook
README, recipe 03 "Paged Attention").

The backward is the exact gradient of that definition for an upstream gradient
dO (gpu-inference blog, section 02: D preprocessing, dK/dV and dQ passes):
dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P * (dP - D),
dQ = scale dS K, dK = scale dS^T Q.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_attn_rows_f64.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double,
                                                 P, ctypes.c_int64, P, P, I]
            lib.oracle_attn_fwd_f64.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double,
                                                P, P, I]
            lib.oracle_paged_decode_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I,
                                                    ctypes.c_double, P, P, I]
            lib.oracle_num_threads.argtypes = [I]
            lib.oracle_attn_gqa_rows_f64.argtypes = [P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double,
                                                     P, ctypes.c_int64, P, P, I]
            lib.oracle_paged_decode_gqa_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I,
                                                        ctypes.c_double, P, P, I, I]
            lib.oracle_paged_prefill_gqa_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I,
                                                         ctypes.c_double, P, P, I, I]
            lib.oracle_paged_prefill_gqa_f64.restype = ctypes.c_int
            lib.oracle_attn_bwd_gqa_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double,
                                                    P, P, P, P, P, P, I]
            lib.oracle_attn_bwd_gqa_f64.restype = ctypes.c_int
            lib.oracle_bwd_rowdot_f64.argtypes = [P, P, ctypes.c_int64, I, P]
            lib.oracle_bwd_rowdot_f64.restype = ctypes.c_int
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_code.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_code.restype = ctypes.c_uint8
            lib.oracle_e4m3_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_float, P]
            lib.oracle_e4m3_quantize.restype = ctypes.c_int
            lib.oracle_paged_decode_fp8_gqa_f64.argtypes = [P, P, P, ctypes.c_double, ctypes.c_double, P, P, I, I,
                                                            I, I, I, I, I, ctypes.c_double, P, P, I, I]
            lib.oracle_paged_decode_fp8_gqa_f64.restype = ctypes.c_int
            lib.oracle_paged_prefill_fp8_gqa_f64.argtypes = [P, P, P, ctypes.c_double, ctypes.c_double, P, P, I,
                                                             I, I, I, I, I, I, I, I, ctypes.c_double, P, P, I, I]
            lib.oracle_paged_prefill_fp8_gqa_f64.restype = ctypes.c_int
            lib.oracle_attn_gqa_rows_f64.restype = ctypes.c_int
            lib.oracle_paged_decode_gqa_f64.restype = ctypes.c_int
            for f in (lib.oracle_attn_rows_f64, lib.oracle_attn_fwd_f64,
                      lib.oracle_paged_decode_f64, lib.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns (uint16, C-contiguous) of a torch bf16 tensor or a uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # plain CPU PyTorch, used only to reinterpret bits
    if x.dtype != torch.bfloat16:
        raise TypeError("torch input must be bfloat16")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_to_f64(x) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = bf16_bits(x).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _i32(x) -> np.ndarray | None:
    if x is None:
        return None
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads(nthreads: int = 0) -> int:
    return int(_load().oracle_num_threads(nthreads))


def attn_fwd(q, k, v, causal: bool, scale: float, kv_lens=None, nthreads: int = 0):
    """Full prefill attention. q [B,H,Nq,d], k/v [B,H,Nkv,d] bf16.

    Returns (O float64 [B,H,Nq,d], LSE float64 [B,H,Nq])."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    B, H, Nq, d = qb.shape
    Nkv = kb.shape[2]
    if kb.shape != (B, H, Nkv, d) or vb.shape != kb.shape:
        raise ValueError("shape mismatch")
    kl = _i32(kv_lens)
    if kl is not None and kl.shape != (B,):
        raise ValueError("kv_lens must be [B]")
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    err = _load().oracle_attn_fwd_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(kl), B, H, Nq, Nkv, d,
                                      int(bool(causal)), float(scale), _ptr(o), _ptr(lse), nthreads)
    if err:
        raise RuntimeError(f"oracle_attn_fwd_f64 failed ({err})")
    return o, lse


def attn_rows(q, k, v, causal: bool, scale: float, rows, kv_lens=None, nthreads: int = 0):
    """Selected query rows, flat index r = (b*H + h)*Nq + i.

    Returns (O float64 [n,d], LSE float64 [n])."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    B, H, Nq, d = qb.shape
    Nkv = kb.shape[2]
    if kb.shape != (B, H, Nkv, d) or vb.shape != kb.shape:
        raise ValueError("shape mismatch")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    kl = _i32(kv_lens)
    o = np.empty((len(r), d), np.float64)
    lse = np.empty((len(r),), np.float64)
    err = _load().oracle_attn_rows_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(kl), B, H, Nq, Nkv, d,
                                       int(bool(causal)), float(scale), _ptr(r), len(r), _ptr(o),
                                       _ptr(lse), nthreads)
    if err:
        raise RuntimeError(f"oracle_attn_rows_f64 failed ({err})")
    return o, lse


def paged_decode(q, k_pages, v_pages, page_table, ctx_lens, scale: float, nthreads: int = 0):
    """Paged decode. q [B,H,d]; k_pages/v_pages [P,H,page_size,d] bf16;
    page_table [B,max_pages] int32; ctx_lens [B] int32.

    Returns (O float64 [B,H,d], LSE float64 [B,H])."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k_pages), bf16_bits(v_pages)
    B, H, d = qb.shape
    P, Hk, ps, dk = kb.shape
    if (Hk, dk) != (H, d) or vb.shape != kb.shape:
        raise ValueError("shape mismatch")
    pt = _i32(page_table)
    cl = _i32(ctx_lens)
    if pt.ndim != 2 or pt.shape[0] != B or cl.shape != (B,):
        raise ValueError("page_table must be [B,max_pages] and ctx_lens [B]")
    o = np.empty((B, H, d), np.float64)
    lse = np.empty((B, H), np.float64)
    err = _load().oracle_paged_decode_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(cl), ps, B,
                                          H, d, pt.shape[1], P, float(scale), _ptr(o), _ptr(lse),
                                          nthreads)
    if err:
        raise RuntimeError(f"oracle_paged_decode_f64 failed ({err})")
    return o, lse


def attn_fwd_gqa(q, k, v, causal: bool, scale: float, kv_lens=None, nthreads: int = 0):
    """Grouped-query prefill: q [B,Hq,Nq,d], k/v [B,Hkv,Nkv,d] bf16, Hq % Hkv == 0; query head h
    reads key/value head h // (Hq // Hkv).  Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq]) in float64."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    B, Hq, Nq, d = qb.shape
    Hkv, Nkv = kb.shape[1], kb.shape[2]
    if kb.shape != (B, Hkv, Nkv, d) or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    kl = _i32(kv_lens)
    rows = np.arange(B * Hq * Nq, dtype=np.int64)
    o = np.empty((B * Hq * Nq, d), np.float64)
    lse = np.empty((B * Hq * Nq,), np.float64)
    err = _load().oracle_attn_gqa_rows_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(kl), B, Hq, Hkv, Nq, Nkv, d,
                                           int(bool(causal)), float(scale), _ptr(rows), len(rows), _ptr(o),
                                           _ptr(lse), nthreads)
    if err:
        raise RuntimeError(f"oracle_attn_gqa_rows_f64 failed ({err})")
    return o.reshape(B, Hq, Nq, d), lse.reshape(B, Hq, Nq)


def paged_decode_gqa(q, k_pages, v_pages, page_table, ctx_lens, scale: float, nthreads: int = 0,
                     skip_bad_pages: bool = False):
    """Grouped-query paged decode: q [B,Hq,d]; k_pages/v_pages [P,Hkv,page_size,d].
    A page id outside [0, P) is an error, or with ``skip_bad_pages`` an unmapped page whose
    positions hold no token.  Returns (O [B,Hq,d], LSE [B,Hq]) in float64."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k_pages), bf16_bits(v_pages)
    B, Hq, d = qb.shape
    P, Hkv, ps, dk = kb.shape
    if dk != d or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    pt = _i32(page_table)
    cl = _i32(ctx_lens)
    o = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    err = _load().oracle_paged_decode_gqa_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(cl), ps, B, Hq,
                                              Hkv, d, pt.shape[1], P, float(scale), _ptr(o), _ptr(lse),
                                              nthreads, int(bool(skip_bad_pages)))
    if err:
        raise RuntimeError(f"oracle_paged_decode_gqa_f64 failed ({err})")
    return o, lse


def paged_prefill_gqa(q, k_pages, v_pages, page_table, ctx_lens, causal: bool, scale: float, nthreads: int = 0,
                      skip_bad_pages: bool = False):
    """Chunked prefill over the paged cache: q [B,Hq,Nq,d] are the last Nq of the ctx_lens[b]
    cached tokens of sequence b (bottom-right causal); k_pages/v_pages [P,Hkv,page_size,d].
    A page id outside [0, P) is an error, or with ``skip_bad_pages`` an unmapped page whose
    positions hold no token (the other positions keep theirs).
    Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq]) in float64."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k_pages), bf16_bits(v_pages)
    B, Hq, Nq, d = qb.shape
    P, Hkv, ps, dk = kb.shape
    if dk != d or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    pt = _i32(page_table)
    cl = _i32(ctx_lens)
    o = np.empty((B, Hq, Nq, d), np.float64)
    lse = np.empty((B, Hq, Nq), np.float64)
    err = _load().oracle_paged_prefill_gqa_f64(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pt), _ptr(cl), ps, B, Hq, Hkv,
                                               Nq, d, pt.shape[1], P, int(bool(causal)), float(scale), _ptr(o),
                                               _ptr(lse), nthreads, int(bool(skip_bad_pages)))
    if err:
        raise RuntimeError(f"oracle_paged_prefill_gqa_f64 failed ({err})")
    return o, lse


def _f64(x) -> np.ndarray:
    """float64 copy of a bf16 tensor (exact widening) or of a float array."""
    if isinstance(x, np.ndarray) and x.dtype != np.uint16:
        return np.ascontiguousarray(x, dtype=np.float64)
    if not isinstance(x, np.ndarray):
        import torch
        if x.dtype != torch.bfloat16:
            return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())
    return np.ascontiguousarray(bf16_to_f64(x))


def attn_bwd_gqa(q, k, v, dout, causal: bool, scale: float, kv_lens=None, nthreads: int = 0):
    """Gradients of exact attention for upstream gradient dout.  q, dout [B,Hq,Nq,d]; k, v
    [B,Hkv,Nkv,d]; bf16 tensors are widened exactly, float inputs are taken as they are (finite
    differences).  Returns a dict of float64 arrays: dq, dk, dv, and the forward o, lse and the
    row term D = rowsum(P * dP) of the same inputs."""
    qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Nq, d = qd.shape
    Hkv, Nkv = kd.shape[1], kd.shape[2]
    if kd.shape != (B, Hkv, Nkv, d) or vd.shape != kd.shape or dod.shape != qd.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    kl = _i32(kv_lens)
    out = {n: np.empty(qd.shape, np.float64) for n in ("dq", "o")}
    out.update({n: np.empty(kd.shape, np.float64) for n in ("dk", "dv")})
    out.update({n: np.empty((B, Hq, Nq), np.float64) for n in ("lse", "D")})
    err = _load().oracle_attn_bwd_gqa_f64(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dod), _ptr(kl), B, Hq, Hkv, Nq, Nkv,
                                          d, int(bool(causal)), float(scale), _ptr(out["dq"]), _ptr(out["dk"]),
                                          _ptr(out["dv"]), _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["D"]),
                                          nthreads)
    if err:
        raise RuntimeError(f"oracle_attn_bwd_gqa_f64 failed ({err})")
    return out


def bwd_rowdot(o, dout):
    """The backward's preprocessing term D_i = dO_i . O_i from bf16 o, dout [..., d]; float64 [...]."""
    ob, db = bf16_bits(o), bf16_bits(dout)
    if ob.shape != db.shape:
        raise ValueError("shape mismatch")
    d = ob.shape[-1]
    n = ob.size // d
    D = np.empty((n,), np.float64)
    err = _load().oracle_bwd_rowdot_f64(_ptr(ob), _ptr(db), n, d, _ptr(D))
    if err:
        raise RuntimeError("oracle_bwd_rowdot_f64 failed")
    return D.reshape(ob.shape[:-1])


def e4m3_values() -> np.ndarray:
    """float64 value of each of the 256 e4m3 codes (NaN for the two NaN codes)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_value(c) for c in range(256)], np.float64)


def e4m3_code(y: float) -> int:
    """Nearest e4m3 code (ties to even, saturating at 448) of one fp32 value."""
    return int(_load().oracle_e4m3_code(float(np.float32(y))))


def e4m3_quantize(x, scale: float) -> np.ndarray:
    """e4m3 codes (uint8, same shape) of bf16 x under a per-tensor scale:
    code(fp32(x) * fp32(1 / scale))."""
    xb = bf16_bits(x)
    codes = np.empty(xb.shape, np.uint8)
    inv = np.float32(1.0) / np.float32(scale)
    err = _load().oracle_e4m3_quantize(_ptr(xb), xb.size, float(inv), _ptr(codes))
    if err:
        raise RuntimeError("oracle_e4m3_quantize failed")
    return codes


def _u8(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    if x.dtype != np.uint8:
        raise TypeError("e4m3 codes must be uint8")
    return np.ascontiguousarray(x)


def paged_decode_fp8_gqa(q, k_codes, v_codes, k_scale: float, v_scale: float, page_table, ctx_lens, scale: float,
                         nthreads: int = 0, skip_bad_pages: bool = False):
    """Paged decode over an e4m3 cache (codes uint8 [P,Hkv,page_size,d]; value = e4m3 * scale).
    Returns (O [B,Hq,d], LSE [B,Hq]) in float64."""
    qb = bf16_bits(q)
    kb, vb = _u8(k_codes), _u8(v_codes)
    B, Hq, d = qb.shape
    P, Hkv, ps, dk = kb.shape
    if dk != d or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    pt = _i32(page_table)
    cl = _i32(ctx_lens)
    o = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    err = _load().oracle_paged_decode_fp8_gqa_f64(_ptr(qb), _ptr(kb), _ptr(vb), float(k_scale), float(v_scale),
                                                  _ptr(pt), _ptr(cl), ps, B, Hq, Hkv, d, pt.shape[1], P, float(scale),
                                                  _ptr(o), _ptr(lse), nthreads, int(bool(skip_bad_pages)))
    if err:
        raise RuntimeError(f"oracle_paged_decode_fp8_gqa_f64 failed ({err})")
    return o, lse


def paged_prefill_fp8_gqa(q, k_codes, v_codes, k_scale: float, v_scale: float, page_table, ctx_lens, causal: bool,
                          scale: float, nthreads: int = 0, skip_bad_pages: bool = False):
    """Chunked prefill over an e4m3 cache (codes uint8 [P,Hkv,page_size,d]; value = e4m3 * scale):
    q [B,Hq,Nq,d] bf16 are the last Nq of the ctx_lens[b] cached tokens (bottom-right causal).
    Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq]) in float64."""
    qb = bf16_bits(q)
    kb, vb = _u8(k_codes), _u8(v_codes)
    B, Hq, Nq, d = qb.shape
    P, Hkv, ps, dk = kb.shape
    if dk != d or vb.shape != kb.shape or Hq % Hkv:
        raise ValueError("shape mismatch")
    pt = _i32(page_table)
    cl = _i32(ctx_lens)
    o = np.empty((B, Hq, Nq, d), np.float64)
    lse = np.empty((B, Hq, Nq), np.float64)
    err = _load().oracle_paged_prefill_fp8_gqa_f64(_ptr(qb), _ptr(kb), _ptr(vb), float(k_scale), float(v_scale),
                                                   _ptr(pt), _ptr(cl), ps, B, Hq, Hkv, Nq, d, pt.shape[1], P,
                                                   int(bool(causal)), float(scale), _ptr(o), _ptr(lse), nthreads,
                                                   int(bool(skip_bad_pages)))
    if err:
        raise RuntimeError(f"oracle_paged_prefill_fp8_gqa_f64 failed ({err})")
    return o, lse
