"""fp64 CPU oracle for the fused attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``attention_forward_10_gb300``) never imports it, and this package imports
nothing from the product: the two share no code.

The arithmetic lives in ``attn_ref.c`` (plain C, double precision, one OpenMP
loop over query rows); this module only compiles it and marshals arguments.
What is computed, per (b, h, i):

    J(i)  = all keys (full) or keys 0..i (causal)
    s_ij  = scale * q_i . k_j
    LSE_i = max_j s_ij + ln sum_j exp(s_ij - max_j s_ij)      (natural log)
    O_i   = sum_j exp(s_ij - LSE_i) v_j

following LeetCUDA "flash_attn_mma_tiling_qk.cu" (kernel body: scaled scores,
softmax along keys, final division by the row sum) and flash-attention
"hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp" (causal masking loop; LSE is the
log-normaliser of the scaled scores) and "hopper/flash_fwd_kernel.h" (an empty
row stores O = 0 and LSE = -inf).

``attention_ex`` adds grouped K/V heads (query head h reads K/V head
h // (H / H_kv)) and a local window (keys i - window_left .. i + window_right),
the ``qhead_per_khead`` and ``window_size_left/right`` options of the same
backward page.  ``attention_bwd`` gives the gradients dQ, dK, dV of that
definition against dO (the backward page's P, dP, dPsum, dS recurrence
written out in double).  ``attention_fp8`` takes FP8 E4M3 inputs with
descale factors (the FP8 forward of the Hopper forward page).  ``attention_varlen`` takes sequences of different lengths
packed along the rows ([total, H, d], cu_seqlens offsets), the
variable-length mode of the Hopper pages.

Pins (checked by ``tests/test_oracle.py`` against facts other than this code):
closed forms (N = 1, Q = 0, hand-derived golden example), invariants (row
probabilities sum to one, constant V, key/value permutation, per-row shift of
the scores, causal row independence), library routines (PyTorch CPU float64
``scaled_dot_product_attention`` / ``logsumexp`` / ``softmax``), a separately
written blockwise online-softmax evaluation, and an exhaustive check of the
16-bit decoders against PyTorch's conversions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB_PATH = os.path.join(_HERE, "libattn_ref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_ref.c`` into ``libattn_ref.so`` beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    c_long, c_int, c_double = ctypes.c_long, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.attn_ref_fwd_u16.argtypes = [vp, vp, vp, c_int, c_long, c_long,
                                     c_long, c_long, c_double, c_int,
                                     vp, vp, c_int]
    lib.attn_ref_fwd_u16.restype = c_int
    lib.attn_ref_rows_u16.argtypes = [vp, vp, vp, c_int, c_long, c_long,
                                      c_long, c_long, c_double, c_int,
                                      vp, c_long, vp, vp, c_int]
    lib.attn_ref_rows_u16.restype = c_int
    lib.attn_ref_fwd_f64.argtypes = [vp, vp, vp, c_long, c_long, c_long,
                                     c_long, c_double, c_int, vp, vp,
                                     c_int]
    lib.attn_ref_fwd_f64.restype = c_int
    lib.attn_ref_fwd_u16_ex.argtypes = [vp, vp, vp, c_int, c_long, c_long, c_long,
                                        c_long, c_long, c_double, c_int, c_long,
                                        c_long, vp, vp, c_int]
    lib.attn_ref_fwd_u16_ex.restype = c_int
    lib.attn_ref_rows_u16_ex.argtypes = [vp, vp, vp, c_int, c_long, c_long, c_long,
                                         c_long, c_long, c_double, c_int, c_long,
                                         c_long, vp, c_long, vp, vp, c_int]
    lib.attn_ref_rows_u16_ex.restype = c_int
    lib.attn_ref_varlen_u16.argtypes = [vp, vp, vp, c_int, vp, c_long, c_long, c_long, c_long,
                                        c_long, c_double, c_int, c_long, c_long, vp, vp, c_int]
    lib.attn_ref_varlen_u16.restype = c_int
    lib.attn_ref_varlen_qk_u16.argtypes = [vp, vp, vp, c_int, vp, vp, vp, vp, c_long, c_long,
                                           c_long, c_long, c_long, c_long, c_double, c_int,
                                           c_long, c_long, vp, vp, c_int]
    lib.attn_ref_varlen_qk_u16.restype = c_int
    lib.attn_ref_bwd_u16.argtypes = [vp, vp, vp, vp, c_int, c_long, c_long, c_long, c_long,
                                     c_long, c_double, c_int, c_long, c_long, vp, vp, vp, c_int]
    lib.attn_ref_bwd_u16.restype = c_int
    lib.attn_ref_bwd_qk_u16.argtypes = [vp, vp, vp, vp, c_int, c_long, c_long, c_long, c_long,
                                        c_long, c_long, c_double, c_int, c_long, c_long, vp, vp,
                                        vp, c_int]
    lib.attn_ref_bwd_qk_u16.restype = c_int
    lib.attn_ref_e4m3.argtypes = [ctypes.c_uint8]
    lib.attn_ref_e4m3.restype = c_double
    lib.attn_ref_fwd_fp8.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_long,
                                     c_double, c_double, c_double, c_double, c_int, c_long,
                                     c_long, vp, vp, c_int]
    lib.attn_ref_fwd_fp8.restype = c_int
    lib.attn_ref_widen.argtypes = [ctypes.c_uint16, c_int]
    lib.attn_ref_widen.restype = c_double
    lib.attn_ref_max_threads.argtypes = []
    lib.attn_ref_max_threads.restype = c_int
    return lib


_override = None


def use_library(path: str | None) -> None:
    """Point this module at another build of ``attn_ref.c`` (None: the default).

    The oracle's own tests use this to plant deliberate mistakes in a copy of
    the C source and check that the pins catch each one.
    """
    global _override
    with _lock:
        _override = None if path is None else _bind(path)


def _load():
    global _lib
    with _lock:
        if _override is not None:
            return _override
        if _lib is None:
            _lib = _bind(build())
    return _lib


def max_threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return int(_load().attn_ref_max_threads())


def widen(bits: int, is_bf16: bool) -> float:
    """Decode one 16-bit word (binary16 or bfloat16) to a Python float."""
    return float(_load().attn_ref_widen(int(bits) & 0xFFFF, int(bool(is_bf16))))


def _u16_view(t) -> tuple[np.ndarray, bool]:
    """Raw 16-bit words of a CPU torch tensor (float16/bfloat16), C-contiguous."""
    import torch
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"oracle expects float16/bfloat16 inputs, got {t.dtype}")
    words = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(words), t.dtype == torch.bfloat16


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def attention(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """Full O [B,H,N,d] and LSE [B,H,N] (float64 numpy) for 16-bit CPU tensors."""
    qw, is_bf16 = _u16_view(q)
    kw, kb = _u16_view(k)
    vw, vb = _u16_view(v)
    if not (is_bf16 == kb == vb):
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = (int(x) for x in q.shape)
    if tuple(k.shape) != (B, H, N, d) or tuple(v.shape) != (B, H, N, d):
        raise ValueError("q, k, v must all be [B,H,N,d]")
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().attn_ref_fwd_u16(_ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16),
                                  B, H, N, d, float(scale), int(bool(causal)),
                                  _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_fwd_u16 failed")
    return o, lse


def attention_rows(q, k, v, scale: float, causal: bool, rows, nthreads: int = 0):
    """O rows [n,d] and LSE [n] (float64) for the listed (b, h, i) triples."""
    qw, is_bf16 = _u16_view(q)
    kw, _ = _u16_view(k)
    vw, _ = _u16_view(v)
    B, H, N, d = (int(x) for x in q.shape)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = _load().attn_ref_rows_u16(_ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16),
                                   B, H, N, d, float(scale), int(bool(causal)),
                                   _ptr(rows), n, _ptr(o), _ptr(lse),
                                   int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_rows_u16 failed")
    return o, lse


def attention_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  causal: bool, nthreads: int = 0):
    """Same definition on float64 numpy inputs [B,H,N,d]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B,H,N,d]")
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().attn_ref_fwd_f64(_ptr(q), _ptr(k), _ptr(v), B, H, N, d,
                                  float(scale), int(bool(causal)), _ptr(o),
                                  _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_fwd_f64 failed")
    return o, lse


def _check_ex(q, k, v):
    B, H, N, d = (int(x) for x in q.shape)
    Bk, H_kv, Nk, dk = (int(x) for x in k.shape)
    if (Bk, Nk, dk) != (B, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k, v must be [B, H_kv, N, d] matching q's B, N, d")
    if H_kv <= 0 or H % H_kv != 0:
        raise ValueError("H must be a multiple of H_kv")
    return B, H, H_kv, N, d


def attention_ex(q, k, v, scale: float, causal: bool, window_left: int = -1,
                 window_right: int = -1, nthreads: int = 0):
    """O and LSE with grouped K/V heads ([B, H_kv, N, d]) and a local window.

    Query i sees keys j with i - window_left <= j <= i + window_right
    (negative bound: unbounded), and j <= i when causal.
    """
    qw, is_bf16 = _u16_view(q)
    kw, _ = _u16_view(k)
    vw, _ = _u16_view(v)
    B, H, H_kv, N, d = _check_ex(q, k, v)
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().attn_ref_fwd_u16_ex(_ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16), B, H,
                                     H_kv, N, d, float(scale), int(bool(causal)),
                                     int(window_left), int(window_right), _ptr(o),
                                     _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_fwd_u16_ex failed")
    return o, lse


def attention_rows_ex(q, k, v, scale: float, causal: bool, rows, window_left: int = -1,
                      window_right: int = -1, nthreads: int = 0):
    """attention_ex for the listed (b, h, i) triples only."""
    qw, is_bf16 = _u16_view(q)
    kw, _ = _u16_view(k)
    vw, _ = _u16_view(v)
    B, H, H_kv, N, d = _check_ex(q, k, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = _load().attn_ref_rows_u16_ex(_ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16), B, H,
                                      H_kv, N, d, float(scale), int(bool(causal)),
                                      int(window_left), int(window_right), _ptr(rows), n,
                                      _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_rows_u16_ex failed")
    return o, lse


def attention_varlen(q, k, v, cu_seqlens, scale: float, causal: bool, window_left: int = -1,
                     window_right: int = -1, nthreads: int = 0):
    """Sequences packed along the rows: q [total, H, d], k, v [total, H_kv, d],
    sequence b = rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (self-attention within
    each sequence, mask and window counted from its start).  Returns O
    [total, H, d] and LSE [H, total] (float64); rows outside every sequence
    are NaN."""
    qw, is_bf16 = _u16_view(q)
    kw, kb = _u16_view(k)
    vw, vb = _u16_view(v)
    if not (is_bf16 == kb == vb):
        raise TypeError("q, k, v must share one dtype")
    total, H, d = (int(x) for x in q.shape)
    if k.shape != v.shape or k.shape[0] != total or k.shape[2] != d or H % int(k.shape[1]):
        raise ValueError("k, v must be [total, H_kv, d] with H a multiple of H_kv")
    H_kv = int(k.shape[1])
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64).reshape(-1))
    o = np.full((total, H, d), np.nan, dtype=np.float64)
    lse = np.full((H, total), np.nan, dtype=np.float64)
    rc = _load().attn_ref_varlen_u16(_ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16), _ptr(cu),
                                     cu.size - 1, total, H, H_kv, d, float(scale),
                                     int(bool(causal)), int(window_left), int(window_right),
                                     _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_varlen_u16 failed")
    return o, lse


def attention_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool,
                        window_left: int = -1, window_right: int = -1, seqused_q=None,
                        seqused_k=None, nthreads: int = 0):
    """Separate query and key sequences packed along the rows: q [total_q, H,
    d], k, v [total_k, H_kv, d]; sequence b has seqused_q[b] queries (all of
    rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 when seqused_q is None) and
    seqused_k[b] keys likewise, masks bottom-right aligned (query i at key
    position i + n_k - n_q).  Returns O [total_q, H, d] and LSE [H, total_q]
    (float64); rows outside every sequence's used queries are NaN, queries
    with no admissible key get O = 0 and LSE = -inf."""
    qw, is_bf16 = _u16_view(q)
    kw, kb = _u16_view(k)
    vw, vb = _u16_view(v)
    if not (is_bf16 == kb == vb):
        raise TypeError("q, k, v must share one dtype")
    total_q, H, d = (int(x) for x in q.shape)
    if k.shape != v.shape or k.shape[2] != d or H % int(k.shape[1]):
        raise ValueError("k, v must be [total_k, H_kv, d] with H a multiple of H_kv")
    total_k, H_kv = int(k.shape[0]), int(k.shape[1])

    def arr(x):
        return None if x is None else np.ascontiguousarray(
            np.asarray(x, dtype=np.int64).reshape(-1))
    cu_q, cu_k = arr(cu_seqlens_q), arr(cu_seqlens_k)
    used_q, used_k = arr(seqused_q), arr(seqused_k)
    batch = cu_q.size - 1
    if cu_k.size != cu_q.size or any(u is not None and u.size < batch for u in (used_q, used_k)):
        raise ValueError("cu_seqlens_q/k need batch + 1 entries, seqused_q/k batch entries")
    o = np.full((total_q, H, d), np.nan, dtype=np.float64)
    lse = np.full((H, total_q), np.nan, dtype=np.float64)
    rc = _load().attn_ref_varlen_qk_u16(
        _ptr(qw), _ptr(kw), _ptr(vw), int(is_bf16), _ptr(cu_q), _ptr(cu_k),
        None if used_q is None else _ptr(used_q), None if used_k is None else _ptr(used_k),
        batch, total_q, total_k, H, H_kv, d, float(scale), int(bool(causal)), int(window_left),
        int(window_right), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_varlen_qk_u16 failed")
    return o, lse


def attention_bwd(q, k, v, dout, scale: float, causal: bool, window_left: int = -1,
                  window_right: int = -1, nthreads: int = 0):
    """Gradients (dQ [B,H,N,d], dK, dV [B,H_kv,N,d], float64) of the forward
    definition against dO, for the mask, window and head grouping of
    ``attention_ex``: P = exp(S - LSE), dV = P^T dO, dP = dO V^T,
    D = rowsum(P * dP), dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q."""
    qw, is_bf16 = _u16_view(q)
    kw, kb = _u16_view(k)
    vw, vb = _u16_view(v)
    gw, gb = _u16_view(dout)
    if not (is_bf16 == kb == vb == gb):
        raise TypeError("q, k, v, dout must share one dtype")
    B, H, H_kv, N, d = _check_ex(q, k, v)
    if tuple(dout.shape) != tuple(q.shape):
        raise ValueError("dout must have q's shape")
    dq = np.empty((B, H, N, d), dtype=np.float64)
    dk = np.empty((B, H_kv, N, d), dtype=np.float64)
    dv = np.empty((B, H_kv, N, d), dtype=np.float64)
    rc = _load().attn_ref_bwd_u16(_ptr(qw), _ptr(kw), _ptr(vw), _ptr(gw), int(is_bf16), B, H,
                                  H_kv, N, d, float(scale), int(bool(causal)),
                                  int(window_left), int(window_right), _ptr(dq), _ptr(dk),
                                  _ptr(dv), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_bwd_u16 failed")
    return dq, dk, dv


def attention_bwd_qk(q, k, v, dout, scale: float, causal: bool, window_left: int = -1,
                     window_right: int = -1, nthreads: int = 0):
    """Gradients of attention with Nq query rows and Nk key rows per head:
    q, dout [B,H,Nq,d], k, v [B,H_kv,Nk,d]; dQ [B,H,Nq,d], dK, dV [B,H_kv,Nk,d]
    (float64).  Masks and windows are aligned bottom-right (query i at key
    position i + Nk - Nq, the shift of the backward page's masking loops); a
    query row that sees no key contributes nothing and gets dQ = 0."""
    qw, is_bf16 = _u16_view(q)
    kw, kb = _u16_view(k)
    vw, vb = _u16_view(v)
    gw, gb = _u16_view(dout)
    if not (is_bf16 == kb == vb == gb):
        raise TypeError("q, k, v, dout must share one dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B,H,N,d] tensors")
    B, H, Nq, d = (int(x) for x in q.shape)
    _, H_kv, Nk, dk_ = (int(x) for x in k.shape)
    if (tuple(v.shape) != tuple(k.shape) or int(k.shape[0]) != B or dk_ != d or H_kv < 1
            or H % H_kv != 0):
        raise ValueError("k and v must be [B,H_kv,Nk,d] with H a multiple of H_kv")
    if tuple(dout.shape) != tuple(q.shape):
        raise ValueError("dout must have q's shape")
    dq = np.empty((B, H, Nq, d), dtype=np.float64)
    dk = np.empty((B, H_kv, Nk, d), dtype=np.float64)
    dv = np.empty((B, H_kv, Nk, d), dtype=np.float64)
    rc = _load().attn_ref_bwd_qk_u16(_ptr(qw), _ptr(kw), _ptr(vw), _ptr(gw), int(is_bf16), B,
                                     H, H_kv, Nq, Nk, d, float(scale), int(bool(causal)),
                                     int(window_left), int(window_right), _ptr(dq), _ptr(dk),
                                     _ptr(dv), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_bwd_qk_u16 failed")
    return dq, dk, dv


def e4m3(code: int) -> float:
    """The oracle's decoding of one OCP FP8 E4M3 byte."""
    return float(_load().attn_ref_e4m3(int(code)))


def _u8_view(t) -> np.ndarray:
    import torch
    if t.dtype != torch.float8_e4m3fn:
        raise TypeError("expected a torch.float8_e4m3fn tensor")
    return np.ascontiguousarray(t.contiguous().view(torch.uint8).numpy())


def attention_fp8(q, k, v, scale: float, descale_q: float, descale_k: float,
                  descale_v: float, causal: bool, window_left: int = -1,
                  window_right: int = -1, nthreads: int = 0):
    """O [B,H,N,d] and LSE [B,H,N] (float64) of attention on FP8 E4M3 inputs
    (torch.float8_e4m3fn, k/v may have fewer heads) scaled by their descale
    factors: the definition on q = descale_q * Q, k = descale_k * K,
    v = descale_v * V."""
    B, H, H_kv, N, d = _check_ex(q, k, v)
    qw, kw, vw = _u8_view(q), _u8_view(k), _u8_view(v)
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().attn_ref_fwd_fp8(_ptr(qw), _ptr(kw), _ptr(vw), B, H, H_kv, N, d, float(scale),
                                  float(descale_q), float(descale_k), float(descale_v),
                                  int(bool(causal)), int(window_left), int(window_right),
                                  _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle attn_ref_fwd_fp8 failed")
    return o, lse
