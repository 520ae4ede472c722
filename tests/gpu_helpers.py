"""Helpers for the GPU parity tests: run the C ABI on guarded buffers, compare with
the CPU oracle.

The output buffer is surrounded by a guard band filled with a NaN canary pattern,
so a test sees both "every element of C was written" (no canary left inside) and
"nothing outside C was written" (the guard band is intact): the persistent
scheduler covers each tile exactly once and partial tiles skip out-of-range
stores ("TileLang core primitives" page, section 4.2; "TileLang: from tile
dataflow to controllable AI kernels", section "concurrency correctness").
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_gemm_gb300 as tl

CANARY = 0x7E55          # a NaN in fp16; in bf16 (0x7E55) also a NaN
GUARD = 64               # elements of guard before C (keeps C 128-byte aligned)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_device_padded(x_cpu: torch.Tensor, ld: int | None = None, offset: int = 0):
    """Copy a CPU 2-D tensor to the GPU with leading dimension ``ld`` (>= cols) and the
    first element ``offset`` elements past a 256-byte aligned base.  Returns
    (pointer, ld, keep-alive tensor)."""
    rows, cols = x_cpu.shape
    ld = cols if ld is None else ld
    buf = torch.zeros(offset + max(rows, 1) * ld + 8, dtype=x_cpu.dtype, device="cuda")
    view = buf[offset:offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(x_cpu.cuda())
    return view.data_ptr(), ld, buf


class GuardedC:
    """C of shape (M, N) with leading dimension ldc inside a canary-filled buffer."""

    def __init__(self, M: int, N: int, ldc: int, dtype: torch.dtype, offset: int = GUARD):
        self.M, self.N, self.ldc, self.offset = M, N, ldc, offset
        total = offset + M * ldc + GUARD
        self.buf = torch.full((total,), CANARY, dtype=torch.int16, device="cuda").view(dtype)
        self.ptr = self.buf.data_ptr() + 2 * offset

    def host_bits(self) -> np.ndarray:
        return bits_of(self.buf)

    def result(self) -> np.ndarray:
        b = self.host_bits()
        body = b[self.offset:self.offset + self.M * self.ldc].reshape(self.M, self.ldc)
        return body[:, :self.N].copy()

    def check_guards(self) -> None:
        b = self.host_bits()
        mask = np.ones(b.shape, dtype=bool)
        body = np.arange(self.M * self.ldc).reshape(self.M, self.ldc)[:, :self.N]
        mask[self.offset + body.ravel()] = False
        outside = b[mask]
        assert np.all(outside == CANARY), \
            f"{int(np.sum(outside != CANARY))} elements outside C were written"
        inside = b[~mask]
        assert not np.any(inside == CANARY), \
            f"{int(np.sum(inside == CANARY))} elements of C were never written"


def run_tl(a_cpu, b_cpu, M, N, K, dtype_code, trans_a=False, trans_b=False, relu=False,
           plan=None, lda=None, ldb=None, ldc=None, a_off=0, b_off=0, c_off=GUARD,
           stream=None):
    """Run tl_gemm (or tl_gemm_with_plan) on copies of the CPU operands; returns
    (C bits as (M, N) uint16, GuardedC)."""
    pa, lda, keep_a = to_device_padded(a_cpu, lda, a_off)
    pb, ldb, keep_b = to_device_padded(b_cpu, ldb, b_off)
    ldc = N if ldc is None else ldc
    tdt = torch.float16 if dtype_code == tl.TL_F16 else torch.bfloat16
    c = GuardedC(M, N, ldc, tdt, c_off)
    s = stream or torch.cuda.current_stream()
    epi = tl.TL_EPI_RELU if relu else tl.TL_EPI_NONE
    if plan is None:
        st = tl.tl_gemm(pa, pb, c.ptr, M, N, K, lda, ldb, ldc, dtype_code, int(trans_a),
                        int(trans_b), epi, s.cuda_stream)
    else:
        st = tl.tl_gemm_with_plan(pa, pb, c.ptr, M, N, K, lda, ldb, ldc, dtype_code,
                                  int(trans_a), int(trans_b), epi, plan, s.cuda_stream)
    assert st == tl.TL_OK, tl.tl_status_string(st)
    torch.cuda.synchronize()
    dev_st, word = tl.tl_device_status(reset=True)
    assert dev_st == tl.TL_OK, f"device-side wait gave up: status word {word:#x}"
    del keep_a, keep_b
    return c.result(), c


def oracle_full(a_cpu, b_cpu, M, N, K, dtype_code, trans_a, trans_b, relu):
    return oracle.gemm(a_cpu, b_cpu, M, N, K, dtype=dtype_code, trans_a=trans_a,
                       trans_b=trans_b, relu=relu)


def assert_within_tolerance(got_bits, ref_bits, dtype_code, rtol=1e-2, atol=1e-2):
    """|C - C_ref| <= atol + rtol |C_ref| element by element; returns error statistics."""
    got = oracle.decode(got_bits, dtype_code)
    ref = oracle.decode(ref_bits, dtype_code)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    ref_max = float(np.abs(ref).max(initial=0.0))
    ref_rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    stats = {"max_abs": float(err.max(initial=0.0)),
             "max_rel": float((err / np.maximum(np.abs(ref), 1e-30)).max(initial=0.0)),
             # scale-free figures: the largest error over the largest output, and the
             # RMS error over the RMS output (0 where the reference is all zero)
             "norm_max": float(err.max(initial=0.0)) / ref_max if ref_max > 0 else 0.0,
             "rel_rms": (float(np.sqrt(np.mean(err * err))) / ref_rms
                         if ref_rms > 0 else 0.0),
             "mismatch": float(bad.mean()) if bad.size else 0.0}
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside tolerance; {stats}"
    return stats


def assert_bit_exact(got_bits, ref_bits):
    """Identical 16-bit patterns, with -0 and +0 counted equal."""
    g = np.where((got_bits & 0x7FFF) == 0, 0, got_bits)
    r = np.where((ref_bits & 0x7FFF) == 0, 0, ref_bits)
    diff = g != r
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} elements differ"


def sample_indices(M, N, count, rng, bm=128, bn=64, per_edge=16):
    """Entries to compare with the oracle one by one: `count` random ones; the whole of
    the first and last row and of the first and last column (the ragged edges, where
    boxes are zero-filled and stores clipped); and, for every row tile and every column
    tile, its first and last row (column) at `per_edge` random columns (rows)."""
    rows = list(rng.integers(0, M, count))
    cols = list(rng.integers(0, N, count))
    for r in sorted({0, M - 1}):
        rows += [r] * N
        cols += list(range(N))
    for c in sorted({0, N - 1}):
        rows += list(range(M))
        cols += [c] * M
    edge_r = sorted({min(M - 1, x) for t in range(0, M, bm) for x in (t, t + bm - 1)})
    edge_c = sorted({min(N - 1, x) for t in range(0, N, bn) for x in (t, t + bn - 1)})
    for r in edge_r:
        rows += [r] * per_edge
        cols += list(rng.integers(0, N, per_edge))
    for c in edge_c:
        rows += list(rng.integers(0, M, per_edge))
        cols += [c] * per_edge
    return np.asarray(rows, np.int64), np.asarray(cols, np.int64)


def exact_integer_product(a_cpu, b_cpu, trans_a, trans_b, relu):
    """The exact product of small-integer operands as float64: every partial sum is an
    integer far below 2^53, so float64 evaluation is exact in any order (a closed form,
    not a second implementation of the oracle); ReLU gives +0 for negatives."""
    a = a_cpu.to(torch.float64).numpy()
    b = b_cpu.to(torch.float64).numpy()
    c = (a.T if trans_a else a) @ (b.T if trans_b else b)
    return np.where(c > 0, c, 0.0) if relu else c
