"""GB300 (sm_103a) fused attention forward: thin Python binding of libfa_gb300.so.

Every entry point of the C ABI (``include/fa.h``) is exposed here under the
same name with plain-integer arguments (device pointers, sizes, a CUDA stream
handle); the binding only marshals arguments.  ``fwd()`` is the PyTorch
convenience on top: it allocates O and LSE with torch on the inputs' device
and passes ``data_ptr()`` values and the current stream to ``fa_fwd``.

All compute runs in the library's CUDA kernels.  There is no fallback: the
library is loaded on the first call, and if it has not been built that call
raises ImportError.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

FA_DTYPE_F16 = 0
FA_DTYPE_BF16 = 1

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_ERR_SCRATCH_LIMIT = 6

# Size of the library's fixed per-device split-KV scratch (fa.h).
FA_NOALLOC_SCRATCH_BYTES = 32 << 20

# Every exported symbol of include/fa.h, with its ctypes signature.
_vp, _i, _f, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
_ull = ctypes.c_ulonglong
SIGNATURES = {
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "fa_fwd_ext": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i, _vp], _i),
    "fa_fwd_fp8": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _f, _f, _i, _i, _i,
                    _vp, _ull, _vp], _i),
    "fa_fwd_fp8_workspace_bytes": ([_i, _i, _i, _i, ctypes.POINTER(_ull)], _i),
    "fa_fwd_host": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i, _vp, _ull,
                     _vp], _i),
    "fa_fwd_host_workspace_bytes": ([_i, _i, _i, _i, _i, _i, ctypes.POINTER(_ull)], _i),
    "fa_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ull, _i, _i, _i, _i, _i, _f,
                _i, _i, _i, _i, _vp], _i),
    "fa_bwd_workspace_bytes": ([_i, _i, _i, ctypes.POINTER(_ull)], _i),
    "fa_bwd_varlen": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                       _f, _i, _i, _i, _i, _vp, _ull, _vp], _i),
    "fa_bwd_varlen_qk": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i,
                          _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i, _vp, _ull, _vp], _i),
    "fa_fwd_varlen": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i,
                       _vp], _i),
    "fa_fwd_varlen_qk": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                          _i, _i, _f, _i, _i, _i, _i, _vp], _i),
    "fa_fwd_splitkv": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i, _i,
                        _vp, _ull, _vp], _i),
    "fa_splitkv_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_ull)], _i),
    "fa_fwd_splitkv_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i,
                                _i, _vp], _i),
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_get_device_status": ([_vp, ctypes.POINTER(_i)], _i),
    "fa_set_wait_timeout_us": ([_ll], _i),
    "fa_set_max_ctas": ([_i], _i),
    "fa_set_gqa_pack": ([_i], _i),
    "fa_selftest_watchdog": ([_ll, _vp], _i),
    "fa_num_sms": ([], _i),
}


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)} ({status})")


_lib_handle = None


def _load():
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or attention_forward_10_gb300/build.py); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib_handle = lib
    return lib


class _LazyLib:
    def __getattr__(self, name):
        return getattr(_load(), name)


_lib = _LazyLib()


# ---------------------------------------------------------------- raw C ABI
def fa_fwd(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, N: int,
           d: int, scale: float, causal: int, dtype: int, stream: int | None) -> int:
    return int(_lib.fa_fwd(q, k, v, o, lse or None, B, H, N, d, scale, causal, dtype,
                           stream or None))


def fa_fwd_ext(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int,
               N: int, d: int, scale: float, causal: int, window_left: int,
               window_right: int, dtype: int, stream: int | None) -> int:
    return int(_lib.fa_fwd_ext(q, k, v, o, lse or None, B, H, H_kv, N, d, scale, causal,
                               window_left, window_right, dtype, stream or None))


def fa_fwd_fp8(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int,
               N: int, d: int, scale: float, descale_q: float, descale_k: float,
               descale_v: float, causal: int, window_left: int, window_right: int,
               workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    return int(_lib.fa_fwd_fp8(q, k, v, o, lse or None, B, H, H_kv, N, d, scale, descale_q,
                               descale_k, descale_v, causal, window_left, window_right,
                               workspace or None, int(workspace_bytes), stream or None))


def fa_fwd_fp8_workspace_bytes(B: int, H_kv: int, N: int, d: int) -> tuple[int, int]:
    out = ctypes.c_ulonglong(0)
    st = int(_lib.fa_fwd_fp8_workspace_bytes(B, H_kv, N, d, ctypes.byref(out)))
    return st, int(out.value)


def fa_fwd_host(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, H_kv: int,
                N: int, d: int, scale: float, causal: int, window_left: int,
                window_right: int, dtype: int, workspace: int | None, workspace_bytes: int,
                stream: int | None) -> int:
    return int(_lib.fa_fwd_host(q, k, v, o, lse or None, B, H, H_kv, N, d, scale, causal,
                                window_left, window_right, dtype, workspace or None,
                                int(workspace_bytes), stream or None))


def fa_fwd_host_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int,
                                with_lse: int) -> tuple[int, int]:
    out = ctypes.c_ulonglong(0)
    st = int(_lib.fa_fwd_host_workspace_bytes(B, H, H_kv, N, d, with_lse, ctypes.byref(out)))
    return st, int(out.value)


def fa_bwd(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int, dk: int, dv: int,
           workspace: int, workspace_bytes: int, B: int, H: int, H_kv: int, N: int, d: int,
           scale: float, causal: int, window_left: int, window_right: int, dtype: int,
           stream: int | None) -> int:
    return int(_lib.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace or None,
                           int(workspace_bytes), B, H, H_kv, N, d, scale, causal, window_left,
                           window_right, dtype, stream or None))


def fa_bwd_varlen(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int, dk: int,
                  dv: int, cu_seqlens: int, batch: int, max_seqlen: int, total: int, H: int,
                  H_kv: int, d: int, scale: float, causal: int, window_left: int,
                  window_right: int, dtype: int, workspace: int | None, workspace_bytes: int,
                  stream: int | None) -> int:
    return int(_lib.fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens or None, batch,
                                  max_seqlen, total, H, H_kv, d, scale, causal, window_left,
                                  window_right, dtype, workspace or None, int(workspace_bytes),
                                  stream or None))


def fa_bwd_varlen_qk(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int, dk: int,
                     dv: int, cu_seqlens_q: int, cu_seqlens_k: int, seqused_q: int | None,
                     seqused_k: int | None, batch: int, max_seqlen_q: int, max_seqlen_k: int,
                     total_q: int, total_k: int, H: int, H_kv: int, d: int, scale: float,
                     causal: int, window_left: int, window_right: int, dtype: int,
                     workspace: int | None, workspace_bytes: int, stream: int | None) -> int:
    return int(_lib.fa_bwd_varlen_qk(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q or None,
                                     cu_seqlens_k or None, seqused_q or None, seqused_k or None,
                                     batch, max_seqlen_q, max_seqlen_k, total_q, total_k, H,
                                     H_kv, d, scale, causal, window_left, window_right, dtype,
                                     workspace or None, int(workspace_bytes), stream or None))


def fa_bwd_workspace_bytes(B: int, H: int, N: int) -> tuple[int, int]:
    out = ctypes.c_ulonglong(0)
    st = int(_lib.fa_bwd_workspace_bytes(B, H, N, ctypes.byref(out)))
    return st, int(out.value)


def fa_fwd_varlen_qk(q: int, k: int, v: int, o: int, lse: int | None, cu_seqlens_q: int,
                     cu_seqlens_k: int, seqused_q: int | None, seqused_k: int | None,
                     batch: int, max_seqlen_q: int, max_seqlen_k: int, total_q: int,
                     total_k: int, H: int, H_kv: int, d: int, scale: float, causal: int,
                     window_left: int, window_right: int, dtype: int,
                     stream: int | None) -> int:
    return int(_lib.fa_fwd_varlen_qk(q, k, v, o, lse or None, cu_seqlens_q or None,
                                     cu_seqlens_k or None, seqused_q or None, seqused_k or None,
                                     batch, max_seqlen_q, max_seqlen_k, total_q, total_k, H,
                                     H_kv, d, scale, causal, window_left, window_right, dtype,
                                     stream or None))


def fa_fwd_varlen(q: int, k: int, v: int, o: int, lse: int | None, cu_seqlens: int,
                  batch: int, max_seqlen: int, total: int, H: int, H_kv: int, d: int,
                  scale: float, causal: int, window_left: int, window_right: int, dtype: int,
                  stream: int | None) -> int:
    return int(_lib.fa_fwd_varlen(q, k, v, o, lse or None, cu_seqlens or None, batch,
                                  max_seqlen, total, H, H_kv, d, scale, causal, window_left,
                                  window_right, dtype, stream or None))


def fa_fwd_splitkv(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int,
                   H_kv: int, N: int, d: int, scale: float, causal: int, window_left: int,
                   window_right: int, dtype: int, num_splits: int, workspace: int | None,
                   workspace_bytes: int, stream: int | None) -> int:
    return int(_lib.fa_fwd_splitkv(q, k, v, o, lse or None, B, H, H_kv, N, d, scale, causal,
                                   window_left, window_right, dtype, num_splits,
                                   workspace or None, int(workspace_bytes), stream or None))


def fa_fwd_splitkv_noalloc(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int,
                           H_kv: int, N: int, d: int, scale: float, causal: int,
                           window_left: int, window_right: int, dtype: int, num_splits: int,
                           stream: int | None) -> int:
    return int(_lib.fa_fwd_splitkv_noalloc(q, k, v, o, lse or None, B, H, H_kv, N, d, scale,
                                           causal, window_left, window_right, dtype,
                                           num_splits, stream or None))


def fa_splitkv_workspace_bytes(B: int, H: int, N: int, d: int, causal: int, window_left: int,
                               window_right: int, num_splits: int) -> tuple[int, int]:
    """(status, bytes) of the scratch fa_fwd_splitkv needs."""
    out = ctypes.c_ulonglong(0)
    st = int(_lib.fa_splitkv_workspace_bytes(B, H, N, d, causal, window_left, window_right,
                                             num_splits, ctypes.byref(out)))
    return st, int(out.value)


def fa_status_string(status: int) -> str:
    return _lib.fa_status_string(int(status)).decode()


def fa_get_device_status(stream: int | None = None) -> tuple[int, int]:
    """(status, site) after synchronising ``stream``; clears the status word."""
    site = ctypes.c_int(0)
    st = int(_lib.fa_get_device_status(stream or None, ctypes.byref(site)))
    return st, int(site.value)


def fa_set_wait_timeout_us(timeout_us: int) -> int:
    return int(_lib.fa_set_wait_timeout_us(int(timeout_us)))


def fa_set_max_ctas(max_ctas: int) -> int:
    return int(_lib.fa_set_max_ctas(int(max_ctas)))


def fa_set_gqa_pack(enable: int) -> int:
    return int(_lib.fa_set_gqa_pack(enable))


def fa_selftest_watchdog(timeout_us: int, stream: int | None = None) -> int:
    return int(_lib.fa_selftest_watchdog(int(timeout_us), stream or None))


def fa_num_sms() -> int:
    return int(_lib.fa_num_sms())


# ------------------------------------------------------- torch convenience
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    raise TypeError(f"q/k/v must be float16 or bfloat16, got {t.dtype}")


def _check_qkv(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, H, N, d] and k, v one [B, H_kv, N, d] shape")
    if (k.shape[0], k.shape[2], k.shape[3]) != (q.shape[0], q.shape[2], q.shape[3]):
        raise ValueError("k, v must match q in B, N and d")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors (no CPU path)")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")


def _outputs(q, out, lse, return_lse, stream):
    import torch
    B, H, N, _ = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return out, lse, handle


def fwd(q, k, v, *, scale: float | None = None, causal: bool = False,
        window: tuple[int, int] = (-1, -1), out=None, lse=None, return_lse: bool = True,
        stream=None):
    """Attention forward on CUDA tensors q [B, H, N, d] and k, v [B, H_kv, N, d].

    Returns ``(o, lse)``: o in the input dtype [B,H,N,d], lse float32 [B,H,N]
    (natural-log log-sum-exp of the scaled scores; None if ``return_lse`` is
    False).  ``scale`` defaults to 1/sqrt(d).  H must be a multiple of H_kv
    (grouped heads); ``window = (left, right)`` restricts query i to keys
    i-left .. i+right (negative: unbounded).  Runs on ``stream`` (default:
    torch's current stream of the inputs' device) and does not synchronise.
    """
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = (int(x) for x in q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse, handle = _outputs(q, out, lse, return_lse, stream)
    with torch.cuda.device(q.device):
        st = fa_fwd_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr() if (return_lse and lse is not None) else None,
                        B, H, int(k.shape[1]), N, d, float(scale), int(bool(causal)),
                        int(window[0]), int(window[1]), _dtype_code(q), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return out, (lse if return_lse else None)


def fwd_host(q, k, v, *, scale: float | None = None, causal: bool = False,
             window: tuple[int, int] = (-1, -1), out=None, lse=None, return_lse: bool = True,
             workspace=None, device=None, stream=None):
    """Attention forward on HOST (CPU) tensors q [B, H, N, d] and k, v
    [B, H_kv, N, d] through fa_fwd_host: the library stages chunks through
    device memory and writes o (and lse) back to host memory.

    Returns ``(o, lse)`` as CPU tensors (page-locked when allocated here),
    valid once ``stream`` (default: torch's current stream of ``device``,
    default the current CUDA device) has finished the call's work.  Page-lock
    q, k, v (``pin_memory()``) for the copies to overlap the computation.
    ``workspace``: a CUDA uint8 tensor of at least
    fa_fwd_host_workspace_bytes() bytes (allocated here when None).
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, H, N, d] and k, v one [B, H_kv, N, d] shape")
    if (k.shape[0], k.shape[2], k.shape[3]) != (q.shape[0], q.shape[2], q.shape[3]):
        raise ValueError("k, v must match q in B, N and d")
    if any(t.device.type != "cpu" for t in (q, k, v)):
        raise ValueError("fwd_host takes host (CPU) tensors; use fwd for CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = (int(x) for x in q.shape)
    H_kv = int(k.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(dev):
        if workspace is None:
            st, need = fa_fwd_host_workspace_bytes(B, H, H_kv, N, d, int(bool(return_lse)))
            if st != FA_OK:
                raise FaError(st, "fa_fwd_host_workspace_bytes")
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            if hasattr(stream, "cuda_stream") and stream != torch.cuda.current_stream(dev):
                workspace.record_stream(stream)
        st = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if (return_lse and lse is not None) else None,
                         B, H, H_kv, N, d, float(scale), int(bool(causal)), int(window[0]),
                         int(window[1]), _dtype_code(q), workspace.data_ptr(),
                         workspace.numel(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_host")
    return out, (lse if return_lse else None)


def fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, *, scale: float | None = None,
               causal: bool = False, window: tuple[int, int] = (-1, -1), out=None, lse=None,
               return_lse: bool = True, stream=None):
    """Attention forward over sequences packed along the rows.

    q is [total, H, d] and k, v are [total, H_kv, d] CUDA tensors; sequence b
    is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (``cu_seqlens``: int32 CUDA
    tensor of batch + 1 offsets; ``max_seqlen``: the longest length).
    Returns ``(o, lse)`` with o [total, H, d] and lse float32 [H, total].
    """
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("q must be [total, H, d] and k, v one [total, H_kv, d] shape")
    if (k.shape[0], k.shape[2]) != (q.shape[0], q.shape[2]):
        raise ValueError("k, v must match q in total and d")
    if not (q.is_cuda and k.is_cuda and v.is_cuda and cu_seqlens.is_cuda):
        raise ValueError("q, k, v, cu_seqlens must be CUDA tensors (no CPU path)")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    total, H, d = (int(x) for x in q.shape)
    batch = int(cu_seqlens.numel()) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        st = fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if (return_lse and lse is not None) else None,
                           cu_seqlens.data_ptr(), max(batch, 0), int(max_seqlen), total, H,
                           int(k.shape[1]), d, float(scale), int(bool(causal)),
                           int(window[0]), int(window[1]), _dtype_code(q), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return out, (lse if return_lse else None)


def fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  *, seqused_q=None, seqused_k=None, scale: float | None = None,
                  causal: bool = False, window: tuple[int, int] = (-1, -1), out=None,
                  lse=None, return_lse: bool = True, stream=None):
    """Attention forward over packed sequences with separate query and key
    rows (cross-attention, KV caches).

    q is [total_q, H, d], k and v [total_k, H_kv, d] CUDA tensors; sequence
    b has query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
    cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (int32 CUDA tensors of batch + 1
    offsets), cut to their first seqused_q[b] / seqused_k[b] rows when those
    int32 CUDA tensors are given.  Masks are bottom-right aligned.  Returns
    ``(o, lse)`` with o [total_q, H, d] and lse float32 [H, total_q]; query
    rows outside every sequence's used rows are left as they were in
    ``out`` / ``lse``.
    """
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or k.shape[2] != q.shape[2]:
        raise ValueError("q must be [total_q, H, d] and k, v one [total_k, H_kv, d] shape")
    idx = [t for t in (cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k) if t is not None]
    if not all(t.is_cuda for t in (q, k, v, *idx)):
        raise ValueError("q, k, v and the offset tensors must be CUDA tensors (no CPU path)")
    if any(t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous() for t in idx):
        raise ValueError("offsets and used lengths must be contiguous 1-D int32 tensors")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    total_q, H, d = (int(x) for x in q.shape)
    total_k = int(k.shape[0])
    batch = int(cu_seqlens_q.numel()) - 1
    if int(cu_seqlens_k.numel()) != batch + 1 or any(
            t is not None and int(t.numel()) < batch for t in (seqused_q, seqused_k)):
        raise ValueError("cu_seqlens_k needs batch + 1 offsets, seqused_q/k batch lengths")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    with torch.cuda.device(q.device):
        st = fa_fwd_varlen_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr() if (return_lse and lse is not None) else None,
                              cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), ptr(seqused_q),
                              ptr(seqused_k), max(batch, 0), int(max_seqlen_q),
                              int(max_seqlen_k), total_q, total_k, H, int(k.shape[1]), d,
                              float(scale), int(bool(causal)), int(window[0]), int(window[1]),
                              _dtype_code(q), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen_qk")
    return out, (lse if return_lse else None)


def fwd_fp8(q, k, v, *, scale: float | None = None, descale_q: float = 1.0,
            descale_k: float = 1.0, descale_v: float = 1.0, causal: bool = False,
            window: tuple[int, int] = (-1, -1), out=None, lse=None, return_lse: bool = True,
            workspace=None, stream=None):
    """Attention forward on torch.float8_e4m3fn CUDA tensors q [B,H,N,128] and
    k, v [B,H_kv,N,128] with descale factors; returns (o bf16, lse fp32)."""
    import torch
    if not (q.dtype == k.dtype == v.dtype == torch.float8_e4m3fn):
        raise TypeError("q, k, v must be torch.float8_e4m3fn")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, H, N, d] and k, v one [B, H_kv, N, d] shape")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors (no CPU path)")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = (int(x) for x in q.shape)
    H_kv = int(k.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        st, need = fa_fwd_fp8_workspace_bytes(B, H_kv, N, d)
        if st != FA_OK:
            raise FaError(st, "fa_fwd_fp8_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        st = fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr() if (return_lse and lse is not None) else None, B, H,
                        H_kv, N, d, float(scale), float(descale_q), float(descale_k),
                        float(descale_v), int(bool(causal)), int(window[0]), int(window[1]),
                        workspace.data_ptr(), workspace.numel(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return out, (lse if return_lse else None)


def bwd(q, k, v, o, lse, dout, *, scale: float | None = None, causal: bool = False,
        window: tuple[int, int] = (-1, -1), dq=None, dk=None, dv=None, workspace=None,
        stream=None):
    """Gradients (dq, dk, dv) of the forward pass ``fwd`` produced (o, lse) for,
    against dout; shapes and dtype as in ``fwd``.  d must be 64 or 128."""
    import torch
    _check_qkv(q, k, v)
    if o.shape != q.shape or dout.shape != q.shape or not (o.is_contiguous() and
                                                            dout.is_contiguous()):
        raise ValueError("o and dout must be contiguous and shaped like q")
    B, H, N, d = (int(x) for x in q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        st, need = fa_bwd_workspace_bytes(B, H, N)
        if st != FA_OK:
            raise FaError(st, "fa_bwd_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                    workspace.data_ptr(), workspace.numel(), B, H, int(k.shape[1]), N, d,
                    float(scale), int(bool(causal)), int(window[0]), int(window[1]),
                    _dtype_code(q), handle)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv


def bwd_varlen(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, *,
               scale: float | None = None, causal: bool = False,
               window: tuple[int, int] = (-1, -1), workspace=None, stream=None):
    """Gradients (dq, dk, dv) of ``fwd_varlen`` for packed sequences: q, o, dout
    [total, H, d], k, v [total, H_kv, d], lse [H, total]."""
    import torch
    total, H, d = (int(x) for x in q.shape)
    batch = int(cu_seqlens.numel()) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        st, need = fa_bwd_workspace_bytes(max(batch, 0), H, int(max_seqlen))
        if st != FA_OK:
            raise FaError(st, "fa_bwd_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        st = fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), cu_seqlens.data_ptr(), max(batch, 0), int(max_seqlen),
                           total, H, int(k.shape[1]), d, float(scale), int(bool(causal)),
                           int(window[0]), int(window[1]), _dtype_code(q), workspace.data_ptr(),
                           workspace.numel(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_varlen")
    return dq, dk, dv


def bwd_varlen_qk(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, *, seqused_q=None, seqused_k=None,
                  scale: float | None = None, causal: bool = False,
                  window: tuple[int, int] = (-1, -1), workspace=None, stream=None):
    """Gradients (dq, dk, dv) of ``fwd_varlen_qk``: q, o, dout [total_q, H, d],
    k, v [total_k, H_kv, d], lse [H, total_q]; separate query and key offsets
    (int32 CUDA tensors of batch + 1 entries) and optional used lengths.
    Rows past the used lengths are left as torch.empty_like made them."""
    import torch
    total_q, H, d = (int(x) for x in q.shape)
    total_k = int(k.shape[0])
    batch = int(cu_seqlens_q.numel()) - 1
    if int(cu_seqlens_k.numel()) != batch + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        st, need = fa_bwd_workspace_bytes(max(batch, 0), H, int(max_seqlen_q))
        if st != FA_OK:
            raise FaError(st, "fa_bwd_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        st = fa_bwd_varlen_qk(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(),
            cu_seqlens_k.data_ptr(), seqused_q.data_ptr() if seqused_q is not None else None,
            seqused_k.data_ptr() if seqused_k is not None else None, max(batch, 0),
            int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, H, int(k.shape[1]), d,
            float(scale), int(bool(causal)), int(window[0]), int(window[1]), _dtype_code(q),
            workspace.data_ptr(), workspace.numel(), handle)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_varlen_qk")
    return dq, dk, dv


def fwd_splitkv(q, k, v, *, num_splits: int = 0, scale: float | None = None,
                causal: bool = False, window: tuple[int, int] = (-1, -1), out=None,
                lse=None, return_lse: bool = True, workspace=None, stream=None):
    """``fwd`` with each row's keys cut into ``num_splits`` ranges run as
    separate work units and merged (0: a count that fills the SMs).

    ``workspace`` is an optional uint8 CUDA tensor of at least the bytes
    ``fa_splitkv_workspace_bytes`` reports (256-byte aligned); without one it
    is allocated with torch on the inputs' device.
    """
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = (int(x) for x in q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse, handle = _outputs(q, out, lse, return_lse, stream)
    with torch.cuda.device(q.device):
        st, need = fa_splitkv_workspace_bytes(B, H, N, d, int(bool(causal)), int(window[0]),
                                              int(window[1]), int(num_splits))
        if st != FA_OK:
            raise FaError(st, "fa_splitkv_workspace_bytes")
        if need > 0 and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if (return_lse and lse is not None) else None,
                            B, H, int(k.shape[1]), N, d, float(scale), int(bool(causal)),
                            int(window[0]), int(window[1]), _dtype_code(q), int(num_splits),
                            ws_ptr, ws_bytes, handle)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_splitkv")
    return out, (lse if return_lse else None)


__all__ = [
    "LIB_PATH", "SIGNATURES", "FaError", "fwd", "bwd", "fwd_fp8", "fwd_varlen", "fwd_splitkv",
    "fa_fwd", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes",
    "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_varlen", "bwd_varlen", "fa_bwd_varlen_qk",
    "bwd_varlen_qk",
    "fa_fwd_ext", "fa_fwd_varlen",
    "fa_fwd_splitkv", "fa_splitkv_workspace_bytes", "fa_fwd_splitkv_noalloc",
    "fa_status_string",
    "fa_get_device_status", "fa_set_wait_timeout_us", "fa_set_max_ctas",
    "fa_selftest_watchdog", "fa_num_sms",
    "FA_DTYPE_F16", "FA_DTYPE_BF16", "FA_OK", "FA_ERR_INVALID_ARG",
    "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED", "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT",
    "FA_ERR_SCRATCH_LIMIT", "FA_NOALLOC_SCRATCH_BYTES",
]
