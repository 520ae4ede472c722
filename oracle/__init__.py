"""CPU oracle for the tiled GEMM: C = epilogue(op(A) . op(B)), rounded to fp16/bf16.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never loads it, and it shares no code with the CUDA library: the
arithmetic lives in ``tl_oracle.c`` (plain C, binary64 accumulation, its own
fp16/bf16 decoders and round-to-nearest-even encoders), built by ``build()``
with gcc and called here through ctypes.

Every function follows the plain definition of the product written out in
``tl_oracle.c``'s header, from the pages' T.gemm semantics ("TileLang core
primitives" page, section 3.3: transpose_A / transpose_B choose between [M,K]
and [K,M], [K,N] and [N,K]; section 3.8: ReLU as max(x, 0) on the fp32
accumulator) and the GEMM skeleton's numerics ("TileLang: from tile dataflow to
controllable AI kernels", section "minimal but complete GEMM skeleton": fp16
inputs, fp32 accumulation, cast to the output dtype at the end).

Pins (checked by ``tests/test_oracle_pins.py`` without a GPU): every decoder and
encoder against numpy/torch's own conversions over all 65536 bit patterns and all
midpoints; the GEMM against closed forms (identity, permutation, all-ones = K,
rank-1, K = 1, ReLU zeroing), exact integer products from numpy, exact rational
sums (fractions.Fraction) within the binary64 error bound, and a hand-computed
2x2x2 case.  The FP8 forms (E4M3 / E5M2 operands, one product scale alpha) are
pinned the same way: both decoders against torch's float8 conversions over all 256
codes plus the formats' defining values, and the FP8 product against closed forms
and exact integer products.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tl_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16 = 0
BF16 = 1
E4M3 = 2
E5M2 = 3

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``tl_oracle.c`` into ``_build/liboracle.so`` (gcc -O2 -fopenmp, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_gemm.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci, ci, ci]
        lib.oracle_gemm.restype = ci
        lib.oracle_gemm_entries.argtypes = [p, p, i64, i64, i64, i64, i64, ci, ci, ci, ci,
                                            p, p, i64, p, p, ci]
        lib.oracle_gemm_entries.restype = ci
        lib.oracle_decode_array.argtypes = [p, p, i64, ci]
        lib.oracle_decode_array.restype = None
        lib.oracle_encode_array.argtypes = [p, p, i64, ci]
        lib.oracle_encode_array.restype = None
        lib.oracle_gemm_fp8.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ci, ci, ci,
                                         ci, ci, ctypes.c_double, ci, ci]
        lib.oracle_gemm_fp8.restype = ci
        lib.oracle_gemm_fp8_entries.argtypes = [p, p, i64, i64, i64, i64, i64, ci, ci, ci, ci,
                                                ci, ctypes.c_double, ci, p, p, i64, p, p, ci]
        lib.oracle_gemm_fp8_entries.restype = ci
        lib.oracle_attention.argtypes = [p, p, p, p, p, i64, i64, i64, i64, ci, ci, ci]
        lib.oracle_attention.restype = ci
        lib.oracle_attention_rows.argtypes = [p, p, p, i64, i64, i64, i64, ci, ci, p, p, p, i64,
                                              p, ci]
        lib.oracle_attention_rows.restype = ci
        lib.oracle_gemm_mx.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, i64,
                                       ci, ci, ci, ci, ci]
        lib.oracle_gemm_mx.restype = ci
        lib.oracle_gemm_mx_entries.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, i64,
                                               ci, ci, ci, ci, p, p, i64, p, p, ci]
        lib.oracle_gemm_mx_entries.restype = ci
        lib.oracle_decode8_array.argtypes = [p, p, i64, ci]
        lib.oracle_decode8_array.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ci
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _as_u16(x) -> np.ndarray:
    """Accept a numpy uint16/float16 array or a CPU torch fp16/bf16 tensor; return raw bits."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.float16:
            return np.ascontiguousarray(x).view(np.uint16)
        if x.dtype == np.uint16:
            return np.ascontiguousarray(x)
        raise TypeError(f"expected uint16/float16 bits, got {x.dtype}")
    import torch  # CPU-side helper only
    if not isinstance(x, torch.Tensor) or x.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("expected a 16-bit float tensor or uint16 bit array")
    t = x.detach().to("cpu").contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact binary64 value of each 16-bit pattern."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_array(_ptr(bits), _ptr(out), bits.size, dtype)
    return out


def encode(values: np.ndarray, dtype: int) -> np.ndarray:
    """Round-to-nearest-even of binary64 values into 16-bit patterns."""
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=np.uint16)
    _load().oracle_encode_array(_ptr(values), _ptr(out), values.size, dtype)
    return out


def gemm(A, B, M: int, N: int, K: int, *, lda: int | None = None, ldb: int | None = None,
         ldc: int | None = None, dtype: int = F16, trans_a: bool = False,
         trans_b: bool = False, relu: bool = False, threads: int = 0,
         want_sums: bool = False):
    """C (uint16 bits, shape (M, ldc) viewed as (M, N)) and optionally the binary64 sums.

    ``A`` and ``B`` hold the storage exactly as the library reads it: A is
    [M, lda] (or [K, lda] when ``trans_a``), B is [K, ldb] (or [N, ldb] when
    ``trans_b``), flattened row-major.
    """
    a = _as_u16(A).reshape(-1)
    b = _as_u16(B).reshape(-1)
    lda = lda if lda is not None else (M if trans_a else K)
    ldb = ldb if ldb is not None else (K if trans_b else N)
    ldc = ldc if ldc is not None else N
    c = np.zeros((M, ldc), dtype=np.uint16)
    sums = np.zeros((M, N), dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm(_ptr(a), _ptr(b), _ptr(c),
                             _ptr(sums) if sums is not None else None,
                             M, N, K, lda, ldb, ldc, dtype, int(trans_a), int(trans_b),
                             int(relu), threads)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    c = c[:, :N]
    return (c, sums) if want_sums else c


def gemm_entries(A, B, M: int, N: int, K: int, rows, cols, *, lda: int | None = None,
                 ldb: int | None = None, dtype: int = F16, trans_a: bool = False,
                 trans_b: bool = False, relu: bool = False, threads: int = 0,
                 want_sums: bool = False):
    """C[rows[t], cols[t]] for each t, computed one by one (for sampled parity at full size)."""
    a = _as_u16(A).reshape(-1)
    b = _as_u16(B).reshape(-1)
    lda = lda if lda is not None else (M if trans_a else K)
    ldb = ldb if ldb is not None else (K if trans_b else N)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    cidx = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != cidx.shape:
        raise ValueError("rows and cols must have the same shape")
    out = np.zeros(r.shape, dtype=np.uint16)
    sums = np.zeros(r.shape, dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm_entries(_ptr(a), _ptr(b), M, N, K, lda, ldb, dtype,
                                     int(trans_a), int(trans_b), int(relu), _ptr(r),
                                     _ptr(cidx), r.size, _ptr(out),
                                     _ptr(sums) if sums is not None else None, threads)
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return (out, sums) if want_sums else out


# ---- FP8 operands -----------------------------------------------------------------

def _as_u8(x) -> np.ndarray:
    """Accept a numpy uint8 array or a CPU torch float8/uint8 tensor; return raw codes."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.uint8:
            return np.ascontiguousarray(x)
        raise TypeError(f"expected uint8 codes, got {x.dtype}")
    import torch  # CPU-side helper only
    if not isinstance(x, torch.Tensor) or x.element_size() != 1:
        raise TypeError("expected an 8-bit tensor or uint8 code array")
    t = x.detach().to("cpu").contiguous()
    return t.view(torch.uint8).numpy()


def decode8(codes: np.ndarray, fmt: int) -> np.ndarray:
    """Exact binary64 value of each E4M3 (fmt 2) or E5M2 (fmt 3) code."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().oracle_decode8_array(_ptr(codes), _ptr(out), codes.size, fmt)
    return out


def gemm_fp8(A, B, M: int, N: int, K: int, *, a_fmt: int = E4M3, b_fmt: int = E4M3,
             out_dtype: int = BF16, alpha: float = 1.0, lda: int | None = None,
             ldb: int | None = None, ldc: int | None = None, trans_a: bool = False,
             trans_b: bool = False, relu: bool = False, threads: int = 0,
             want_sums: bool = False):
    """C = round_out(epi(alpha * op(A) . op(B))) from 8-bit operands; uint16 bits (M, N)."""
    a = _as_u8(A).reshape(-1)
    b = _as_u8(B).reshape(-1)
    lda = lda if lda is not None else (M if trans_a else K)
    ldb = ldb if ldb is not None else (K if trans_b else N)
    ldc = ldc if ldc is not None else N
    c = np.zeros((M, ldc), dtype=np.uint16)
    sums = np.zeros((M, N), dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm_fp8(_ptr(a), _ptr(b), _ptr(c),
                                 _ptr(sums) if sums is not None else None,
                                 M, N, K, lda, ldb, ldc, a_fmt, b_fmt, out_dtype,
                                 int(trans_a), int(trans_b), float(alpha), int(relu), threads)
    if rc != 0:
        raise ValueError("oracle_gemm_fp8 rejected its arguments")
    c = c[:, :N]
    return (c, sums) if want_sums else c


def gemm_mx(A, B, SA, SB, M: int, N: int, K: int, *, a_fmt: int = E4M3, b_fmt: int = E4M3,
            out_dtype: int = BF16, lda: int | None = None, ldb: int | None = None,
            ldc: int | None = None, sfa_ld: int | None = None, sfb_ld: int | None = None,
            relu: bool = False, threads: int = 0, want_sums: bool = False):
    """Block-scaled 8-bit product: A [M,K] and B [N,K] K-major codes, SA [M, sfa_ld] and
    SB [N, sfb_ld] E8M0 codes, one per 32 K elements; uint16 bits (M, N)."""
    a, b = _as_u8(A).reshape(-1), _as_u8(B).reshape(-1)
    sa, sb = _as_u8(SA).reshape(-1), _as_u8(SB).reshape(-1)
    lda = lda if lda is not None else K
    ldb = ldb if ldb is not None else K
    ldc = ldc if ldc is not None else N
    sfa_ld = sfa_ld if sfa_ld is not None else K // 32
    sfb_ld = sfb_ld if sfb_ld is not None else K // 32
    c = np.zeros((M, ldc), dtype=np.uint16)
    sums = np.zeros((M, N), dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm_mx(_ptr(a), _ptr(b), _ptr(sa), _ptr(sb), _ptr(c),
                                _ptr(sums) if sums is not None else None, M, N, K, lda, ldb,
                                ldc, sfa_ld, sfb_ld, a_fmt, b_fmt, out_dtype, int(relu), threads)
    if rc != 0:
        raise ValueError("oracle_gemm_mx rejected its arguments")
    c = c[:, :N]
    return (c, sums) if want_sums else c


def gemm_mx_entries(A, B, SA, SB, M: int, N: int, K: int, rows, cols, *, a_fmt: int = E4M3,
                    b_fmt: int = E4M3, out_dtype: int = BF16, lda: int | None = None,
                    ldb: int | None = None, sfa_ld: int | None = None, sfb_ld: int | None = None,
                    relu: bool = False, threads: int = 0, want_sums: bool = False):
    """Selected entries of the block-scaled product, computed one by one."""
    a, b = _as_u8(A).reshape(-1), _as_u8(B).reshape(-1)
    sa, sb = _as_u8(SA).reshape(-1), _as_u8(SB).reshape(-1)
    lda = lda if lda is not None else K
    ldb = ldb if ldb is not None else K
    sfa_ld = sfa_ld if sfa_ld is not None else K // 32
    sfb_ld = sfb_ld if sfb_ld is not None else K // 32
    r = np.ascontiguousarray(rows, dtype=np.int64)
    cidx = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.zeros(r.shape, dtype=np.uint16)
    sums = np.zeros(r.shape, dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm_mx_entries(_ptr(a), _ptr(b), _ptr(sa), _ptr(sb), M, N, K, lda, ldb,
                                        sfa_ld, sfb_ld, a_fmt, b_fmt, out_dtype, int(relu),
                                        _ptr(r), _ptr(cidx), r.size, _ptr(out),
                                        _ptr(sums) if sums is not None else None, threads)
    if rc != 0:
        raise ValueError("oracle_gemm_mx_entries rejected its arguments")
    return (out, sums) if want_sums else out


def gemm_fp8_entries(A, B, M: int, N: int, K: int, rows, cols, *, a_fmt: int = E4M3,
                     b_fmt: int = E4M3, out_dtype: int = BF16, alpha: float = 1.0,
                     lda: int | None = None, ldb: int | None = None, trans_a: bool = False,
                     trans_b: bool = False, relu: bool = False, threads: int = 0,
                     want_sums: bool = False):
    """Selected entries of the FP8 product, computed one by one."""
    a = _as_u8(A).reshape(-1)
    b = _as_u8(B).reshape(-1)
    lda = lda if lda is not None else (M if trans_a else K)
    ldb = ldb if ldb is not None else (K if trans_b else N)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    cidx = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.zeros(r.shape, dtype=np.uint16)
    sums = np.zeros(r.shape, dtype=np.float64) if want_sums else None
    rc = _load().oracle_gemm_fp8_entries(_ptr(a), _ptr(b), M, N, K, lda, ldb, a_fmt, b_fmt,
                                         out_dtype, int(trans_a), int(trans_b), float(alpha),
                                         int(relu), _ptr(r), _ptr(cidx), r.size, _ptr(out),
                                         _ptr(sums) if sums is not None else None, threads)
    if rc != 0:
        raise ValueError("oracle_gemm_fp8_entries rejected its arguments")
    return (out, sums) if want_sums else out


# ---- attention --------------------------------------------------------------------

def attention(Q, K, V, *, dtype: int = F16, causal: bool = False, threads: int = 0,
              want_sums: bool = False):
    """O = softmax(Q K^T / sqrt(D)) V per (batch, head), all four [B, S, H, D]; uint16 bits."""
    shape = tuple(Q.shape)
    if len(shape) != 4 or tuple(K.shape) != shape or tuple(V.shape) != shape:
        raise ValueError("Q, K and V must all be [B, S, H, D]")
    B, S, H, D = shape
    q, k, v = (_as_u16(x).reshape(-1) for x in (Q, K, V))
    o = np.zeros(shape, dtype=np.uint16)
    sums = np.zeros(shape, dtype=np.float64) if want_sums else None
    rc = _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                  _ptr(sums) if sums is not None else None, B, S, H, D, dtype,
                                  int(causal), threads)
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return (o, sums) if want_sums else o


def attention_rows(Q, K, V, bs, is_, hs, *, dtype: int = F16, causal: bool = False,
                   threads: int = 0):
    """Rows O[bs[t], is_[t], hs[t], :] computed one by one (sampled parity); (count, D)."""
    B, S, H, D = tuple(Q.shape)
    q, k, v = (_as_u16(x).reshape(-1) for x in (Q, K, V))
    b_ = np.ascontiguousarray(bs, dtype=np.int64)
    i_ = np.ascontiguousarray(is_, dtype=np.int64)
    h_ = np.ascontiguousarray(hs, dtype=np.int64)
    out = np.zeros((b_.size, D), dtype=np.uint16)
    rc = _load().oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, dtype, int(causal),
                                       _ptr(b_), _ptr(i_), _ptr(h_), b_.size, _ptr(out), threads)
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return out
