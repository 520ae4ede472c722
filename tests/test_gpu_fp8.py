"""GPU parity of the FP8 path (tl_gemm_fp8) against the CPU oracle.

C = epi(alpha * op(A) . op(B)) with E4M3 / E5M2 operands, fp32 accumulation in
Tensor Memory and an fp16 or bf16 output.  Bars as for the 16-bit path:
* small-integer operands (exact in both 8-bit formats, every fp32 partial sum an
  exact integer, alpha a power of two): bit-exact;
* random operands: |C - C_ref| <= 1e-2 + 1e-2 |C_ref| element by element;
* full-size workloads: sampled entries against the oracle computed one by one, and
  the canary guard band around C for coverage.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import GuardedC, assert_bit_exact, assert_within_tolerance, sample_indices

pytestmark = pytest.mark.gpu

E4M3, E5M2 = workloads.E4M3, workloads.E5M2
F16, BF16 = workloads.F16, workloads.BF16


def _upload8(x_cpu, ld=None, offset=0):
    """8-bit CPU tensor -> device bytes with leading dimension ld and a byte offset."""
    rows, cols = x_cpu.shape
    ld = cols if ld is None else ld
    buf = torch.zeros(offset + max(rows, 1) * ld + 16, dtype=torch.uint8, device="cuda")
    view = buf[offset:offset + rows * ld].view(rows, ld)[:, :cols]
    view.copy_(x_cpu.view(torch.uint8).cuda())
    return view.data_ptr(), ld, buf


def run_fp8(w, a, b, plan=None, lda=None, ldb=None, ldc=None, a_off=0, b_off=0):
    pa, lda, keep_a = _upload8(a, lda, a_off)
    pb, ldb, keep_b = _upload8(b, ldb, b_off)
    ldc = w.N if ldc is None else ldc
    c = GuardedC(w.M, w.N, ldc, w.torch_dtype)
    st = tl.tl_gemm_fp8(pa, pb, c.ptr, w.M, w.N, w.K, lda, ldb, ldc, w.dtype, w.b_fmt,
                        w.c_dtype, int(w.trans_a), int(w.trans_b), w.alpha,
                        tl.TL_EPI_RELU if w.relu else tl.TL_EPI_NONE, plan,
                        torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_OK, tl.tl_status_string(st)
    torch.cuda.synchronize()
    dev_st, word = tl.tl_device_status(reset=True)
    assert dev_st == tl.TL_OK, f"device-side wait gave up: status word {word:#x}"
    c.check_guards()
    del keep_a, keep_b
    return c.result()


def _w(M, N, K, ta, tb, relu, dist, seed, a_fmt=E4M3, b_fmt=E4M3, out=BF16, alpha=1.0):
    return workloads.Workload("fp8", M, N, K, a_fmt, ta, tb, relu, dist, dist, seed=seed,
                              b_dtype=b_fmt, out_dtype=out, alpha=alpha)


def _oracle(w, a, b):
    return oracle.gemm_fp8(a, b, w.M, w.N, w.K, a_fmt=w.dtype, b_fmt=w.b_fmt,
                           out_dtype=w.c_dtype, alpha=w.alpha, trans_a=w.trans_a,
                           trans_b=w.trans_b, relu=w.relu)


def _check(w, plan=None, exact=False, **kw):
    a, b = workloads.make_inputs(w)
    got = run_fp8(w, a, b, plan=plan, **kw)
    ref = _oracle(w, a, b)
    if exact:
        assert_bit_exact(got, ref)
    return assert_within_tolerance(got, ref, w.c_dtype)


# every 8-bit tiling: bm, bn, bk (K elements per stage), deepest ring that fits
TILINGS8 = ((128, 64, 128, 8), (128, 64, 256, 4), (128, 128, 128, 6), (128, 128, 256, 3),
            (128, 256, 128, 4), (128, 256, 256, 2), (256, 128, 128, 8), (256, 128, 256, 4),
            (256, 256, 128, 6), (256, 256, 256, 3))


@pytest.mark.parametrize("bm,bn,bk,smax", TILINGS8)
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_every_fp8_tiling_integer_bit_exact(bm, bn, bk, smax, ta, tb):
    if not tb and (bn // (bm // 128)) % 128 != 0:
        pytest.skip("an N-major B needs 128-column boxes per CTA")
    for stages in sorted({2, smax}):
        plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=3)
        w = _w(300, 2 * bn + 40, 5 * bk + 72, ta, tb, True, "int_small",
               bm + bn + bk + stages + 2 * ta + tb, a_fmt=E4M3, b_fmt=E5M2, out=F16, alpha=0.5)
        _check(w, plan=plan, exact=True)


@pytest.mark.parametrize("bm,bn,bk,smax", TILINGS8)
def test_every_fp8_tiling_random_tolerance(bm, bn, bk, smax):
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, smax, raster_group=2)
    _check(_w(515, 3 * bn + 17, 4 * bk + 31, False, True, False, "normal", bm + bn + bk,
              alpha=0.3), plan=plan)


@pytest.mark.parametrize("a_fmt,b_fmt", [(E4M3, E4M3), (E4M3, E5M2), (E5M2, E4M3),
                                         (E5M2, E5M2)])
@pytest.mark.parametrize("out", [F16, BF16])
def test_formats_outputs_and_scales(a_fmt, b_fmt, out):
    for alpha, relu in ((1.0, False), (0.125, True), (-1.7, True), (3.0, False)):
        _check(_w(260, 390, 700, False, True, relu, "normal", 7 + a_fmt + 2 * b_fmt + out,
                  a_fmt=a_fmt, b_fmt=b_fmt, out=out, alpha=alpha))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 9, 13), (128, 256, 128), (129, 257, 129),
                                   (1000, 72, 2049), (33, 1100, 4096)])
def test_fp8_planner_shapes(M, N, K):
    _check(_w(M, N, K, False, True, True, "int_small", M + N + K, out=F16, alpha=2.0),
           exact=True)
    _check(_w(M, N, K, True, False, False, "normal", M + N + K + 1, alpha=0.7))


def test_fp8_unaligned_pitches_and_offsets_are_repacked():
    # K = 1000 bytes per row is not a multiple of 16: both operands go through the copy
    w = _w(300, 500, 1000, False, True, True, "int_small", 91, out=F16)
    a, b = workloads.make_inputs(w)
    ref = _oracle(w, a, b)
    assert_bit_exact(run_fp8(w, a, b), ref)
    assert_bit_exact(run_fp8(w, a, b, lda=1003, ldb=1001, a_off=3, b_off=5, ldc=517), ref)


@pytest.mark.parametrize("bm,bn,bk,grid", [(128, 128, 256, 0), (256, 256, 256, 0),
                                           (128, 64, 128, 5)])
def test_fp8_stream_k_split_bit_exact(bm, bn, bk, grid):
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, 3, raster_group=3, grid=grid, stream_k=1)
    _check(_w(700, 900, 2100, False, True, True, "int_small", 93 + bm, out=BF16, alpha=0.25),
           plan=plan, exact=True)


def test_fp8_k_zero_and_bad_arguments():
    w = _w(64, 64, 0, False, True, False, "normal", 95)
    c = GuardedC(64, 64, 64, torch.bfloat16)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = tl.tl_gemm_fp8(dummy.data_ptr(), dummy.data_ptr(), c.ptr, 64, 64, 0, 1, 1, 64, E4M3,
                        E4M3, BF16, 0, 1, 1.0, tl.TL_EPI_NONE, None, s)
    assert st == tl.TL_OK
    torch.cuda.synchronize()
    assert np.all(c.result() == 0)
    c.check_guards()
    a = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    b = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    args = (a.data_ptr(), b.data_ptr(), c.ptr, 64, 64, 64, 64, 64, 64)
    assert tl.tl_gemm_fp8(*args, BF16, E4M3, BF16, 0, 1, 1.0, 0, None, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_gemm_fp8(*args, E4M3, E4M3, E4M3, 0, 1, 1.0, 0, None, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_gemm_fp8(*args, E4M3, E4M3, BF16, 0, 1, float("inf"), 0, None, s) == \
        tl.TL_ERR_INVALID_ARG
    assert tl.tl_gemm(*args, E4M3, 0, 1, 0, s) == tl.TL_ERR_INVALID_ARG
    bad = tl.plan_for(0, 0, 0, 128, 64, 128, 4)            # N-major B with 64-wide tiles
    assert tl.tl_gemm_fp8(*args, E4M3, E4M3, BF16, 0, 0, 1.0, 0, bad, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_device_status(reset=True)[0] == tl.TL_OK


def test_fp8_tensor_call():
    w = _w(256, 384, 512, False, True, True, "normal", 97, b_fmt=E5M2, alpha=0.5)
    a, b = workloads.make_inputs(w)
    out = tl.gemm_fp8(a.cuda(), b.cuda(), trans_b=True, relu=True, alpha=0.5)
    assert out.dtype == torch.bfloat16
    assert_within_tolerance(out.cpu().view(torch.int16).numpy().view(np.uint16),
                            _oracle(w, a, b), BF16)


@pytest.mark.parametrize("name", ["gemm_4096_e4m3_tb", "gemm_8192_e4m3_tb"])
def test_fp8_workloads_sampled(name):
    w = workloads.WORKLOADS[name]
    a, b = workloads.make_inputs(w)
    got = run_fp8(w, a, b)
    rng = np.random.default_rng(11)
    rows, cols = sample_indices(w.M, w.N, 4000, rng)
    ref = oracle.gemm_fp8_entries(a, b, w.M, w.N, w.K, rows, cols, a_fmt=w.dtype,
                                  b_fmt=w.b_fmt, out_dtype=w.c_dtype, alpha=w.alpha,
                                  trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu)
    assert_within_tolerance(got[rows, cols], ref, w.c_dtype)
    wi = workloads.integer_variant(w)
    a, b = workloads.make_inputs(wi)
    got = run_fp8(wi, a, b)
    ref = oracle.gemm_fp8_entries(a, b, w.M, w.N, w.K, rows, cols, a_fmt=w.dtype,
                                  b_fmt=w.b_fmt, out_dtype=w.c_dtype, alpha=w.alpha,
                                  trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu)
    assert_bit_exact(got[rows, cols], ref)
