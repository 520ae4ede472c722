"""Python binding of the tl_gemm C ABI (include/tl_gemm.h).

Argument marshalling only: every step of the GEMM runs in the CUDA library
``_build/libtl_gemm.so`` (built by ``tiled_gemm_gb300.build``).  PyTorch supplies
device memory and the current stream.  If the library is missing, importing the
binding raises: there is no CPU or PyTorch fallback.

Names follow the C ABI: ``tl_gemm``, ``tl_gemm_with_plan``, ``tl_gemm_noalloc``,
``tl_gemm_plan``, ``tl_plan_complete``, ``tl_status_string``, ``tl_device_status``,
``tl_last_device_status``, ``tl_set_wait_timeout_ns``, ``tl_version``.  ``gemm`` is the tensor-level call.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

TL_F16 = 0
TL_BF16 = 1
TL_E4M3 = 2
TL_E5M2 = 3
TL_EPI_NONE = 0
TL_EPI_RELU = 1

STATUS_NAMES = ["TL_OK", "TL_ERR_INVALID_ARG", "TL_ERR_NULL_PTR", "TL_ERR_ALIGNMENT",
                "TL_ERR_UNSUPPORTED", "TL_ERR_ALIAS", "TL_ERR_DEVICE", "TL_ERR_LAUNCH",
                "TL_ERR_TIMEOUT"]
TL_OK = 0
TL_ERR_INVALID_ARG = 1
TL_ERR_NULL_PTR = 2
TL_ERR_ALIGNMENT = 3
TL_ERR_UNSUPPORTED = 4
TL_ERR_ALIAS = 5
TL_ERR_DEVICE = 6
TL_ERR_LAUNCH = 7
TL_ERR_TIMEOUT = 8


class TLError(RuntimeError):
    def __init__(self, status: int, what: str = "tl_gemm"):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{what} failed: {name}")


class Plan(ctypes.Structure):
    """Mirror of ``tl_plan``."""
    _fields_ = [
        ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("bk", ctypes.c_int32),
        ("stages", ctypes.c_int32), ("raster_group", ctypes.c_int32), ("grid", ctypes.c_int32),
        ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64), ("tiles", ctypes.c_int64),
        ("k_blocks", ctypes.c_int64), ("ring_bytes", ctypes.c_int64),
        ("smem_bytes", ctypes.c_int64), ("tmem_cols", ctypes.c_int32),
        ("tx_bytes", ctypes.c_int32), ("repack_a", ctypes.c_int32),
        ("repack_b", ctypes.c_int32), ("tma_store", ctypes.c_int32),
        ("l2_prefetch", ctypes.c_int32), ("producers", ctypes.c_int32),
        ("stream_k", ctypes.c_int32), ("dp_tiles", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32), ("sk_iters", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64), ("ksplit", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"tl_gemm CUDA library not built ({LIB_PATH} is missing); run "
            "`python tiled_gemm_gb300/build.py` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, ci, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
    lib.tl_gemm.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci, ci, p]
    lib.tl_gemm.restype = ci
    lib.tl_gemm_with_plan.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci, ci,
                                      ctypes.POINTER(Plan), p]
    lib.tl_gemm_with_plan.restype = ci
    lib.tl_gemm_plan.argtypes = [i64, i64, i64, ci, ci, ci, ci, ctypes.POINTER(Plan)]
    lib.tl_gemm_plan.restype = ci
    lib.tl_plan_complete.argtypes = [i64, i64, i64, ci, ci, ci, ci, ctypes.POINTER(Plan)]
    lib.tl_plan_complete.restype = ci
    lib.tl_gemm_fp8.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci, ci, ci,
                                ctypes.c_float, ci, ctypes.POINTER(Plan), p]
    lib.tl_gemm_fp8.restype = ci
    lib.tl_gemm_mx.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, i64, ci, ci, ci,
                               ci, p]
    lib.tl_gemm_mx.restype = ci
    lib.tl_gemm_noalloc.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci, ci, p]
    lib.tl_gemm_noalloc.restype = ci
    lib.tl_gemm_noalloc_scratch_bytes.argtypes = []
    lib.tl_gemm_noalloc_scratch_bytes.restype = i64
    lib.tl_status_string.argtypes = [ci]
    lib.tl_status_string.restype = ctypes.c_char_p
    lib.tl_device_status.argtypes = [ci, ctypes.POINTER(u32)]
    lib.tl_device_status.restype = ci
    lib.tl_last_device_status.argtypes = []
    lib.tl_last_device_status.restype = ci
    lib.tl_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.tl_set_wait_timeout_ns.restype = None
    lib.tl_attention_fwd.argtypes = [p, p, p, p, i64, i64, i64, i64, ci, ci, p]
    lib.tl_attention_fwd.restype = ci
    lib.tl_debug_set_stall.argtypes = [ci]
    lib.tl_debug_set_stall.restype = None
    lib.tl_version.argtypes = []
    lib.tl_version.restype = ci
    return lib


_lib = _load()
LIBRARY = _lib


# ---- C-ABI names ---------------------------------------------------------------

def tl_gemm(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
            dtype: int, trans_a: int, trans_b: int, epilogue: int, stream: int) -> int:
    """Raw call with integer device pointers and a raw stream handle; returns tl_status."""
    return _lib.tl_gemm(A, B, C, M, N, K, lda, ldb, ldc, dtype, trans_a, trans_b, epilogue,
                        stream)


def tl_gemm_with_plan(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                      ldc: int, dtype: int, trans_a: int, trans_b: int, epilogue: int,
                      plan: Plan, stream: int) -> int:
    return _lib.tl_gemm_with_plan(A, B, C, M, N, K, lda, ldb, ldc, dtype, trans_a, trans_b,
                                  epilogue, ctypes.byref(plan), stream)


def tl_gemm_mx(A: int, B: int, SFA: int, SFB: int, C: int, M: int, N: int, K: int, lda: int,
               ldb: int, ldc: int, sfa_ld: int, sfb_ld: int, a_type: int, b_type: int,
               c_type: int, epilogue: int, stream: int) -> int:
    """Raw block-scaled 8-bit call (K-major codes, E8M0 scales per 32 K); returns tl_status."""
    return _lib.tl_gemm_mx(A, B, SFA, SFB, C, M, N, K, lda, ldb, ldc, sfa_ld, sfb_ld, a_type,
                           b_type, c_type, epilogue, stream)


def tl_gemm_fp8(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                a_type: int, b_type: int, c_type: int, trans_a: int, trans_b: int, alpha: float,
                epilogue: int, plan: Plan | None, stream: int) -> int:
    """Raw FP8 call (8-bit operand codes, fp16/bf16 output); returns tl_status."""
    return _lib.tl_gemm_fp8(A, B, C, M, N, K, lda, ldb, ldc, a_type, b_type, c_type, trans_a,
                            trans_b, float(alpha), epilogue,
                            ctypes.byref(plan) if plan is not None else None, stream)


def tl_gemm_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                    ldc: int, dtype: int, trans_a: int, trans_b: int, epilogue: int,
                    stream: int) -> int:
    """tl_gemm for callers that cannot allocate device memory: operands that need a
    padded copy go through the library's fixed 32 MiB device scratch array instead of
    the stream-ordered allocator (see include/tl_gemm.h).  Returns tl_status."""
    return _lib.tl_gemm_noalloc(A, B, C, M, N, K, lda, ldb, ldc, dtype, trans_a, trans_b,
                                epilogue, stream)


def tl_gemm_noalloc_scratch_bytes() -> int:
    return _lib.tl_gemm_noalloc_scratch_bytes()


def tl_gemm_plan(M: int, N: int, K: int, dtype: int = TL_F16, trans_a: int = 0,
                 trans_b: int = 0, num_sms: int = 0) -> Plan:
    pl = Plan()
    st = _lib.tl_gemm_plan(M, N, K, dtype, trans_a, trans_b, num_sms, ctypes.byref(pl))
    if st != TL_OK:
        raise TLError(st, "tl_gemm_plan")
    return pl


def tl_plan_complete(M: int, N: int, K: int, bm: int, bn: int, bk: int, stages: int,
                     dtype: int = TL_F16, trans_a: int = 0, trans_b: int = 0,
                     num_sms: int = 0, raster_group: int = 16, grid: int = 0,
                     l2_prefetch: int = -1, producers: int = 0, stream_k: int = 0,
                     swap_ab: int = 0, ksplit: int = 0) -> Plan:
    pl = Plan(bm=bm, bn=bn, bk=bk, stages=stages, raster_group=raster_group, grid=grid,
              l2_prefetch=l2_prefetch, producers=producers, stream_k=stream_k, swap_ab=swap_ab,
              ksplit=ksplit)
    st = _lib.tl_plan_complete(M, N, K, dtype, trans_a, trans_b, num_sms, ctypes.byref(pl))
    if st != TL_OK:
        raise TLError(st, "tl_plan_complete")
    return pl


def tl_status_string(status: int) -> str:
    return _lib.tl_status_string(status).decode()


def tl_device_status(reset: bool = False) -> tuple[int, int]:
    """(tl_status, raw status word) of the device-side bounded waits; synchronises."""
    word = ctypes.c_uint32(0)
    st = _lib.tl_device_status(1 if reset else 0, ctypes.byref(word))
    return st, word.value


def tl_last_device_status() -> int:
    """tl_status of the device-side bounded waits since the flag was last cleared;
    synchronises the device and clears nothing."""
    return _lib.tl_last_device_status()


def tl_set_wait_timeout_ns(ns: int) -> None:
    _lib.tl_set_wait_timeout_ns(int(ns))


def tl_attention_fwd(Q: int, K: int, V: int, O: int, B: int, S: int, H: int, D: int,
                     dtype: int, causal: int, stream: int) -> int:
    """Raw attention call on [B, S, H, D] device buffers; returns tl_status."""
    return _lib.tl_attention_fwd(Q, K, V, O, B, S, H, D, dtype, causal, stream)


def tl_debug_set_stall(mode: int) -> None:
    """Test hook: 1 makes the following launches' MMA thread wait on a barrier that
    nothing arrives on, so the bounded wait runs out (TL_ERR_TIMEOUT, site 7); 0 = off."""
    _lib.tl_debug_set_stall(int(mode))


def tl_version() -> int:
    return _lib.tl_version()


# ---- tensor-level call ------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return TL_F16
    if t.dtype == torch.bfloat16:
        return TL_BF16
    raise TypeError(f"tl_gemm supports float16 and bfloat16, got {t.dtype}")


def _ld(t, name: str) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.stride(1) != 1 and t.size(1) > 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return max(t.stride(0), t.size(1), 1)


def gemm(a, b, *, trans_a: bool = False, trans_b: bool = False, relu: bool = False,
         out=None, plan: Plan | None = None, stream=None):
    """C = epi(op(a) . op(b)) on the current CUDA device.

    ``a`` is [M, K] (or [K, M] with ``trans_a``), ``b`` is [K, N] (or [N, K] with
    ``trans_b``); both row-major with unit inner stride, same dtype (fp16/bf16),
    on the current device.  ``out`` (optional) is [M, N] of that dtype, unit inner
    stride.  Runs on ``stream`` (a torch.cuda.Stream) or the current stream.
    """
    torch = _torch()
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("a and b must be CUDA tensors")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    dt = _dtype_code(a)
    M, K = (a.size(1), a.size(0)) if trans_a else (a.size(0), a.size(1))
    Kb, N = (b.size(1), b.size(0)) if trans_b else (b.size(0), b.size(1))
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if out is None:
        out = torch.empty((M, N), dtype=a.dtype, device=a.device)
    elif tuple(out.shape) != (M, N) or out.dtype != a.dtype:
        raise ValueError("out has the wrong shape or dtype")
    lda, ldb, ldc = _ld(a, "a"), _ld(b, "b"), _ld(out, "out")
    s = stream if stream is not None else torch.cuda.current_stream(a.device)
    handle = s.cuda_stream
    epi = TL_EPI_RELU if relu else TL_EPI_NONE
    if plan is None:
        st = tl_gemm(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc, dt,
                     int(trans_a), int(trans_b), epi, handle)
    else:
        st = tl_gemm_with_plan(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, lda, ldb,
                               ldc, dt, int(trans_a), int(trans_b), epi, plan, handle)
    if st != TL_OK:
        raise TLError(st)
    return out


def plan_for(M: int, N: int, K: int, bm: int, bn: int, bk: int, stages: int,
             raster_group: int = 16, grid: int = 0, l2_prefetch: int = -1,
             producers: int = 0, stream_k: int = 0, swap_ab: int = 0,
             tma_store: int = 0, ksplit: int = 0) -> Plan:
    """A plan with a fixed tiling, to pass as ``gemm(..., plan=...)``; l2_prefetch < 0,
    producers <= 0 and stream_k = 0 take the library's defaults for the problem
    (stream_k -1 forces whole tiles only, 1 forces the split of the last waves);
    swap_ab = 1 runs the kernel on C^T = op(B)^T op(A)^T (bm x bn tiles of C^T);
    tma_store = -1 writes C with plain stores instead of TMA bulk stores; ksplit 0 is
    automatic, 1 off, 2 two CTAs of a cluster per tile (cluster split-K)."""
    return Plan(bm=bm, bn=bn, bk=bk, stages=stages, raster_group=raster_group, grid=grid,
                l2_prefetch=l2_prefetch, producers=producers, stream_k=stream_k,
                swap_ab=swap_ab, tma_store=tma_store, ksplit=ksplit)


def _fp8_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float8_e4m3fn:
        return TL_E4M3
    if t.dtype == torch.float8_e5m2:
        return TL_E5M2
    raise TypeError(f"gemm_fp8 takes float8_e4m3fn / float8_e5m2 operands, got {t.dtype}")


def gemm_fp8(a, b, *, trans_a: bool = False, trans_b: bool = False, relu: bool = False,
             alpha: float = 1.0, out_dtype=None, out=None, plan: Plan | None = None,
             stream=None):
    """C = epi(alpha * op(a) . op(b)) with 8-bit float operands, on the current device.

    ``a`` and ``b`` are torch.float8_e4m3fn or torch.float8_e5m2 tensors (the two may
    differ), laid out as for ``gemm``; the output is ``out_dtype`` (torch.bfloat16 by
    default, or torch.float16), or ``out``'s dtype when ``out`` is given.
    """
    torch = _torch()
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("a and b must be CUDA tensors")
    at, bt = _fp8_code(a), _fp8_code(b)
    M, K = (a.size(1), a.size(0)) if trans_a else (a.size(0), a.size(1))
    Kb, N = (b.size(1), b.size(0)) if trans_b else (b.size(0), b.size(1))
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if out is None:
        odt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((M, N), dtype=odt, device=a.device)
    elif tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    ct = _dtype_code(out)
    lda, ldb, ldc = _ld(a, "a"), _ld(b, "b"), _ld(out, "out")
    s = stream if stream is not None else torch.cuda.current_stream(a.device)
    st = tl_gemm_fp8(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc, at, bt,
                     ct, int(trans_a), int(trans_b), alpha,
                     TL_EPI_RELU if relu else TL_EPI_NONE, plan, s.cuda_stream)
    if st != TL_OK:
        raise TLError(st, "tl_gemm_fp8")
    return out


def gemm_mx(a, b, sfa, sfb, *, relu: bool = False, out_dtype=None, out=None, stream=None):
    """C = epi(A B^T) in a block-scaled 8-bit format, on the current device.

    ``a`` [M, K] and ``b`` [N, K] are K-major torch.float8_e4m3fn / torch.float8_e5m2
    tensors; ``sfa`` [M, >= 4*ceil(K/128)] and ``sfb`` [N, ...] are uint8 E8M0 scale
    codes, one per 32 elements of K.  The output is ``out_dtype`` (torch.bfloat16 by
    default, or torch.float16), or ``out``'s dtype when ``out`` is given.
    """
    torch = _torch()
    if not all(t.is_cuda for t in (a, b, sfa, sfb)):
        raise ValueError("a, b, sfa and sfb must be CUDA tensors")
    if sfa.dtype != torch.uint8 or sfb.dtype != torch.uint8:
        raise ValueError("the scales must be uint8 E8M0 codes")
    at, bt = _fp8_code(a), _fp8_code(b)
    M, K = a.size(0), a.size(1)
    N = b.size(0)
    if b.size(1) != K:
        raise ValueError(f"inner dimensions differ: {K} vs {b.size(1)}")
    if out is None:
        odt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((M, N), dtype=odt, device=a.device)
    elif tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    ct = _dtype_code(out)
    s = stream if stream is not None else torch.cuda.current_stream(a.device)
    st = tl_gemm_mx(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), out.data_ptr(),
                    M, N, K, _ld(a, "a"), _ld(b, "b"), _ld(out, "out"), _ld(sfa, "sfa"),
                    _ld(sfb, "sfb"), at, bt, ct, TL_EPI_RELU if relu else TL_EPI_NONE,
                    s.cuda_stream)
    if st != TL_OK:
        raise TLError(st, "tl_gemm_mx")
    return out


def attention(q, k, v, *, causal: bool = False, out=None, stream=None):
    """O = softmax(q k^T / sqrt(D)) v per batch and head; q, k, v (and out) are
    contiguous [B, S, H, D] fp16/bf16 CUDA tensors of one dtype, D = 64 or 128."""
    torch = _torch()
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k and v must be CUDA tensors")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must all be [B, S, H, D]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k and v must be contiguous")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must have the same dtype")
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like q")
    B, S, H, D = q.shape
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    st = tl_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, D,
                          dt, int(causal), s.cuda_stream)
    if st != TL_OK:
        raise TLError(st, "tl_attention_fwd")
    return out
