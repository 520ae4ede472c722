"""GPU parity of the block-scaled (MX) 8-bit GEMM (tl_gemm_mx) against the CPU oracle.

C = epi(sum_k x(A[i,k]) 2^(SFA[i][k/32]-127) x(B[j,k]) 2^(SFB[j][k/32]-127)), both
operands K-major, fp32 accumulation, fp16 or bf16 out.  Bars as for the other paths:
* small-integer operands and scales within 2^+-1: every scaled product is a multiple
  of 1/4 and every fp32 partial sum is exact, so the result must match bit for bit;
* random operands and scales: |C - C_ref| <= 1e-2 + 1e-2 |C_ref| element by element;
* full-size workloads: sampled entries against the oracle computed one by one, and the
  canary guard band around C for coverage.
"""
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


def _upload(x_cpu, ld=None):
    """CPU tensor of bytes -> device rows with pitch ld (bytes); returns (ptr, ld, keep)."""
    x = x_cpu.view(torch.uint8) if x_cpu.dtype != torch.uint8 else x_cpu
    rows, cols = x.shape
    ld = cols if ld is None else ld
    buf = torch.zeros(max(rows, 1) * ld + 64, dtype=torch.uint8, device="cuda")
    view = buf[:rows * ld].view(rows, ld)[:, :cols]
    view.copy_(x.cuda())
    return view.data_ptr(), ld, buf


def run_mx(w, a, b, sa, sb, lda=None, ldb=None, ldc=None):
    pa, lda, ka = _upload(a, lda)
    pb, ldb, kb = _upload(b, ldb)
    psa, _, ksa = _upload(sa)
    psb, _, ksb = _upload(sb)
    ldc = w.N if ldc is None else ldc
    c = GuardedC(w.M, w.N, ldc, w.c_torch_dtype)
    st = tl.tl_gemm_mx(pa, pb, psa, psb, c.ptr, w.M, w.N, w.K, lda, ldb, ldc, w.sf_ld, w.sf_ld,
                       w.a_fmt, w.b_fmt, w.out_dtype,
                       tl.TL_EPI_RELU if w.relu else tl.TL_EPI_NONE,
                       torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_OK, tl.tl_status_string(st)
    torch.cuda.synchronize()
    dev_st, word = tl.tl_device_status(reset=True)
    assert dev_st == tl.TL_OK, f"device-side wait gave up: status word {word:#x}"
    c.check_guards()
    del ka, kb, ksa, ksb
    return c.result()


def _oracle(w, a, b, sa, sb):
    return oracle.gemm_mx(a, b, sa, sb, w.M, w.N, w.K, a_fmt=w.a_fmt, b_fmt=w.b_fmt,
                          out_dtype=w.out_dtype, sfa_ld=w.sf_ld, sfb_ld=w.sf_ld, relu=w.relu)


def _w(M, N, K, seed, exact=False, **kw):
    if exact:
        kw.setdefault("dist", "int_small")
        kw.setdefault("sf_lo", 126)
        kw.setdefault("sf_hi", 128)
    return workloads.MxWorkload("mx", M, N, K, seed=seed, **kw)


SHAPES = [(128, 128, 128), (1, 1, 32), (7, 9, 64), (300, 200, 1056), (129, 257, 2080),
          (256, 384, 4096), (515, 130, 96)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out,relu", [(BF16, False), (F16, True)])
def test_integer_bit_exact(M, N, K, out, relu):
    w = _w(M, N, K, M + N + K + out, exact=True, out_dtype=out, relu=relu,
           a_fmt=E4M3, b_fmt=E5M2 if relu else E4M3)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    assert_bit_exact(run_mx(w, a, b, sa, sb), _oracle(w, a, b, sa, sb))


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("a_fmt,b_fmt", [(E4M3, E4M3), (E5M2, E4M3), (E4M3, E5M2)])
def test_random_within_tolerance(M, N, K, a_fmt, b_fmt):
    w = _w(M, N, K, 7 * M + N + K + a_fmt, a_fmt=a_fmt, b_fmt=b_fmt)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    assert_within_tolerance(run_mx(w, a, b, sa, sb), _oracle(w, a, b, sa, sb), w.out_dtype)


def test_scale_bytes_past_k_are_ignored_and_pitches_padded():
    # K = 1056 is 33 blocks: the last group of four holds one real block.  Every byte
    # past block 32, and the padding of the pitch, is the NaN code: none may reach C.
    w = _w(300, 200, 1056, 55, exact=True, sf_pad=16)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    sa[:, 33:] = 255
    sb[:, 33:] = 255
    ref = _oracle(w, a, b, sa, sb)
    assert_bit_exact(run_mx(w, a, b, sa, sb), ref)
    # padded operand and output pitches too
    assert_bit_exact(run_mx(w, a, b, sa, sb, lda=1072, ldb=1104, ldc=211), ref)


def test_nan_scale_poisons_only_its_rows():
    w = _w(200, 150, 256, 56, exact=True)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    sa[17, 3] = 255
    sb[90, 0] = 255
    got = run_mx(w, a, b, sa, sb)
    vals = oracle.decode(got, w.out_dtype)
    nan = np.isnan(vals)
    assert nan[17].all() and nan[:, 90].all()
    keep = np.ones_like(nan)
    keep[17, :] = False
    keep[:, 90] = False
    assert not nan[keep].any()
    ref = _oracle(w, a, b, sa, sb)
    assert_bit_exact(np.where(keep, got, 0), np.where(keep, ref, 0))


def test_k_zero_and_bad_arguments():
    s = torch.cuda.current_stream().cuda_stream
    c = GuardedC(64, 64, 64, torch.bfloat16)
    x = torch.zeros(64 * 256, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    st = tl.tl_gemm_mx(p, p, p, p, c.ptr, 64, 64, 0, 16, 16, 64, 16, 16, E4M3, E4M3, BF16, 0,
                       s)
    assert st == tl.TL_OK
    torch.cuda.synchronize()
    assert np.all(c.result() == 0)
    c.check_guards()
    args = (p, p, p, p, c.ptr, 64, 64, 128, 128, 128, 64)
    ok = args + (16, 16, E4M3, E4M3, BF16, 0, s)
    assert tl.tl_gemm_mx(*ok) == tl.TL_OK
    torch.cuda.synchronize()
    assert tl.tl_gemm_mx(p, p, p, p, c.ptr, 64, 64, 96 + 8, 128, 128, 64, 16, 16, E4M3, E4M3,
                         BF16, 0, s) == tl.TL_ERR_INVALID_ARG           # K % 32 != 0
    assert tl.tl_gemm_mx(*args, 16, 16, BF16, E4M3, BF16, 0, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_gemm_mx(*args, 16, 16, E4M3, E4M3, E4M3, 0, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_gemm_mx(*args, 2, 16, E4M3, E4M3, BF16, 0, s) == tl.TL_ERR_INVALID_ARG  # short
    assert tl.tl_gemm_mx(*args, 20, 16, E4M3, E4M3, BF16, 0, s) == tl.TL_ERR_ALIGNMENT   # pitch
    assert tl.tl_gemm_mx(p, p, p + 4, p, c.ptr, 64, 64, 128, 128, 128, 64, 16, 16, E4M3, E4M3,
                         BF16, 0, s) == tl.TL_ERR_ALIGNMENT
    assert tl.tl_gemm_mx(p + 8, p, p, p, c.ptr, 64, 64, 128, 128, 128, 64, 16, 16, E4M3, E4M3,
                         BF16, 0, s) == tl.TL_ERR_ALIGNMENT
    assert tl.tl_gemm_mx(p, p, p, p, p, 64, 64, 128, 128, 128, 64, 16, 16, E4M3, E4M3, BF16, 0,
                         s) == tl.TL_ERR_ALIAS
    assert tl.tl_device_status(reset=True)[0] == tl.TL_OK


def test_tensor_call():
    w = _w(256, 384, 512, 57, b_fmt=E5M2, relu=True)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    out = tl.gemm_mx(a.cuda(), b.cuda(), sa.cuda(), sb.cuda(), relu=True)
    assert out.dtype == torch.bfloat16
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_within_tolerance(got, _oracle(w, a, b, sa, sb), BF16)


@pytest.mark.parametrize("name", ["gemm_mx_4096_e4m3", "gemm_mx_8192_e4m3"])
def test_workloads_sampled(name):
    w = workloads.MX_WORKLOADS[name]
    a, b, sa, sb = workloads.make_mx_inputs(w)
    got = run_mx(w, a, b, sa, sb)
    rng = np.random.default_rng(12)
    rows, cols = sample_indices(w.M, w.N, 4000, rng)
    ref = oracle.gemm_mx_entries(a, b, sa, sb, w.M, w.N, w.K, rows, cols, a_fmt=w.a_fmt,
                                 b_fmt=w.b_fmt, out_dtype=w.out_dtype, sfa_ld=w.sf_ld,
                                 sfb_ld=w.sf_ld, relu=w.relu)
    assert_within_tolerance(got[rows, cols], ref, w.out_dtype)
    wi = _w(w.M, w.N, w.K, w.seed + 1, exact=True)
    a, b, sa, sb = workloads.make_mx_inputs(wi)
    got = run_mx(wi, a, b, sa, sb)
    ref = oracle.gemm_mx_entries(a, b, sa, sb, w.M, w.N, w.K, rows, cols, sfa_ld=wi.sf_ld,
                                 sfb_ld=wi.sf_ld)
    assert_bit_exact(got[rows, cols], ref)


def test_narrow_tiles_many_per_cta_sampled():
    # N <= 128 takes the 128-wide tile; 157 tiles over at most one CTA per SM, so CTAs
    # walk several, with K not a multiple of 128 (a partial last stage and scale group)
    w = _w(20000, 100, 1312, 58, exact=True)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    got = run_mx(w, a, b, sa, sb)
    rng = np.random.default_rng(14)
    rows, cols = sample_indices(w.M, w.N, 3000, rng, bm=128, bn=128)
    ref = oracle.gemm_mx_entries(a, b, sa, sb, w.M, w.N, w.K, rows, cols, sfa_ld=w.sf_ld,
                                 sfb_ld=w.sf_ld)
    assert_bit_exact(got[rows, cols], ref)
