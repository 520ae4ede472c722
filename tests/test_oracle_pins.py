"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the oracle so that a plausible mistake (a dropped term,
a wrong sign or index, a transposed operand, a wrong rounding rule) fails here:

* format decoders: every one of the 65536 bit patterns against numpy's binary16
  and torch's bfloat16 conversions;
* the round-to-nearest-even encoders: exact values, every midpoint between
  neighbours (ties go to the even significand), just-above/just-below midpoints,
  overflow thresholds and subnormals, against numpy / torch conversions;
* the GEMM: a hand-computed 2x2x2 case (tests/golden/hand_2x2x2.json), closed forms
  (identity, permutation, all-ones giving K, rank-1 outer products, K = 1, ReLU
  zeroing negatives, K = 0), exact integer products from numpy for all four
  transpose combinations with padded leading dimensions, and exact rational sums
  (fractions.Fraction) within the binary64 error bound.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16_bits(x):
    with np.errstate(over="ignore"):             # past binary16's range: inf, as intended
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits_from_f32(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy())
    return t.view(torch.bfloat16).to(torch.float64).numpy()


ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# ---------------------------------------------------------------- decoders ----

def test_f16_decoder_all_patterns():
    got = oracle.decode(ALL, oracle.F16)
    want = ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decoder_all_patterns():
    got = oracle.decode(ALL, oracle.BF16)
    want = bf16_values(ALL)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ---------------------------------------------------------------- encoders ----

def _finite_sorted_positive(dtype):
    vals = oracle.decode(ALL, dtype)
    return np.unique(np.abs(vals[np.isfinite(vals)]))    # +0 first, no -0


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_encoder_roundtrips_every_finite_value(dtype):
    vals = oracle.decode(ALL, dtype)
    fin = np.isfinite(vals)
    back = oracle.encode(vals[fin], dtype)
    assert np.array_equal(back, ALL[fin])


def test_f16_encoder_midpoints_ties_to_even_and_neighbours():
    pos = _finite_sorted_positive(oracle.F16)
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0                          # exact in binary64
    got = oracle.encode(mid, oracle.F16)
    lo_b, hi_b = oracle.encode(lo, oracle.F16), oracle.encode(hi, oracle.F16)
    want = np.where(lo_b % 2 == 0, lo_b, hi_b)     # tie -> even significand
    assert np.array_equal(got, want)
    assert np.array_equal(got, f16_bits(mid))      # numpy agrees
    eps = (hi - lo) * 2.0 ** -20
    assert np.array_equal(oracle.encode(mid + eps, oracle.F16), hi_b)
    assert np.array_equal(oracle.encode(mid - eps, oracle.F16), lo_b)
    neg = oracle.encode(-mid, oracle.F16)
    assert np.array_equal(neg, want | 0x8000)


def test_bf16_encoder_midpoints_ties_to_even_and_neighbours():
    pos = _finite_sorted_positive(oracle.BF16)
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0                          # 9 significant bits: exact in fp32 too
    got = oracle.encode(mid, oracle.BF16)
    lo_b, hi_b = oracle.encode(lo, oracle.BF16), oracle.encode(hi, oracle.BF16)
    want = np.where(lo_b % 2 == 0, lo_b, hi_b)
    assert np.array_equal(got, want)
    assert np.array_equal(got, bf16_bits_from_f32(mid))   # torch's fp32->bf16 agrees
    eps = (hi - lo) * 2.0 ** -30                  # below fp32 resolution: binary64 only
    assert np.array_equal(oracle.encode(mid + eps, oracle.BF16), hi_b)
    assert np.array_equal(oracle.encode(mid - eps, oracle.BF16), lo_b)


def test_encoders_random_values_against_libraries():
    rng = np.random.default_rng(123)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 20, 200000))
    assert np.array_equal(oracle.encode(x, oracle.F16), f16_bits(x))
    with np.errstate(over="ignore"):             # values past fp32's range become inf
        x32 = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 130, 200000))).astype(
            np.float32)
    x32 = x32[np.isfinite(x32)]
    assert np.array_equal(oracle.encode(x32.astype(np.float64), oracle.BF16),
                          bf16_bits_from_f32(x32))


def test_encoder_special_values():
    E = oracle.encode
    # fp16 overflow threshold: 65504 is the largest finite; 65520 ties to "65536" = inf
    assert E(np.array([65504.0, 65519.99, 65520.0, 1e300]), oracle.F16).tolist() == \
        [0x7BFF, 0x7BFF, 0x7C00, 0x7C00]
    assert E(np.array([-65520.0]), oracle.F16)[0] == 0xFC00
    # fp16 subnormals: 2^-24 is the smallest; half of it ties to 0, 3/4 of it rounds up
    assert E(np.array([2.0 ** -24, 2.0 ** -25, 0.75 * 2.0 ** -24, 2.0 ** -14]),
             oracle.F16).tolist() == [0x0001, 0x0000, 0x0001, 0x0400]
    # bf16: largest finite (2 - 2^-7) 2^127; the midpoint to 2^128 ties to inf
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert E(np.array([big, (2.0 - 2.0 ** -8) * 2.0 ** 127]), oracle.BF16).tolist() == \
        [0x7F7F, 0x7F80]
    assert E(np.array([2.0 ** -133, 2.0 ** -134, 2.0 ** -126]), oracle.BF16).tolist() == \
        [0x0001, 0x0000, 0x0080]
    assert E(np.array([0.0, -0.0, np.inf, -np.inf]), oracle.F16).tolist() == \
        [0x0000, 0x8000, 0x7C00, 0xFC00]
    assert (E(np.array([np.nan]), oracle.F16)[0] & 0x7C00) == 0x7C00
    assert (E(np.array([np.nan]), oracle.F16)[0] & 0x03FF) != 0


# -------------------------------------------------------------------- GEMM ----

def _bits(values, dtype):
    v = np.asarray(values, dtype=np.float64)
    return f16_bits(v) if dtype == oracle.F16 else bf16_bits_from_f32(v.astype(np.float32))


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
@pytest.mark.parametrize("trans_b", [False, True])
def test_hand_computed_2x2x2(dtype, trans_b):
    g = json.load(open(os.path.join(GOLDEN, "hand_2x2x2.json")))
    name = "f16" if dtype == oracle.F16 else "bf16"
    A = _bits(g["A"], dtype)
    Bm = np.asarray(g["B"])
    B = _bits(Bm.T if trans_b else Bm, dtype)
    for relu, key in ((False, "C_none_bits"), (True, "C_relu_bits")):
        C = oracle.gemm(A, B, 2, 2, 2, dtype=dtype, trans_b=trans_b, relu=relu)
        assert C.tolist() == g[key][name]


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_identity_and_permutation(dtype):
    rng = np.random.default_rng(5)
    n, N = 37, 23
    Bv = rng.uniform(-1, 1, (n, N))
    B = _bits(Bv, dtype)
    Bexact = oracle.decode(B, dtype)
    I = _bits(np.eye(n), dtype)
    C = oracle.gemm(I, B, n, N, n, dtype=dtype)
    assert np.array_equal(C, B)                              # I.B = B exactly
    C = oracle.gemm(I, B, n, N, n, dtype=dtype, relu=True)
    want = _bits(np.maximum(Bexact, 0.0), dtype)
    assert np.array_equal(C, want)                           # relu(B)
    perm = rng.permutation(n)
    P = _bits(np.eye(n)[perm], dtype)
    C = oracle.gemm(P, B, n, N, n, dtype=dtype)
    assert np.array_equal(C, B[perm])                        # rows of B permuted
    # B = I on the right: A.I = A, with A transposed in storage as well
    Av = _bits(rng.uniform(-1, 1, (N, n)), dtype)
    C = oracle.gemm(Av.T.copy(), I, N, n, n, dtype=dtype, trans_a=True)
    assert np.array_equal(C, Av)


@pytest.mark.parametrize("K", [1, 7, 64, 4100])
def test_all_ones_gives_k(K):
    ones16 = _bits(np.ones((3, K)), oracle.F16)
    C = oracle.gemm(ones16, ones16, 3, 3, K, dtype=oracle.F16, trans_b=True)
    assert np.all(oracle.decode(C, oracle.F16) == float(K))       # fp16: K <= 4100 exact
    onesbf = _bits(np.ones((3, K)), oracle.BF16)
    C = oracle.gemm(onesbf, onesbf, 3, 3, K, dtype=oracle.BF16, trans_b=True)
    want = {1: 1.0, 7: 7.0, 64: 64.0, 4100: 4096.0}[K]            # bf16 spacing 32 at 4096
    assert np.all(oracle.decode(C, oracle.BF16) == want)


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_rank1_and_relu_zeroing(dtype):
    rng = np.random.default_rng(9)
    M, N, K = 19, 21, 5
    u = _bits(rng.uniform(-1, 1, M), dtype)
    v = _bits(rng.uniform(-1, 1, N), dtype)
    A = np.zeros((M, K), np.uint16)
    A[:, 0] = u                              # A = u e0^T
    B = np.zeros((K, N), np.uint16)
    B[0, :] = v                              # B = e0 v^T
    uv = np.outer(oracle.decode(u, dtype), oracle.decode(v, dtype))   # exact products
    C = oracle.gemm(A, B, M, N, K, dtype=dtype)
    assert np.array_equal(C, oracle.encode(uv, dtype))
    assert np.array_equal(C, _bits(uv, dtype) if dtype == oracle.F16 else C)
    C = oracle.gemm(A, B, M, N, K, dtype=dtype, relu=True)
    assert np.array_equal(C, oracle.encode(np.maximum(uv, 0.0), dtype))
    # all-negative products: relu gives +0 everywhere, no epilogue gives the product
    An = _bits(-np.abs(rng.uniform(0.1, 1, (M, K))), dtype)
    Bp = _bits(np.abs(rng.uniform(0.1, 1, (K, N))), dtype)
    C = oracle.gemm(An, Bp, M, N, K, dtype=dtype, relu=True)
    assert np.all(C == 0)
    C = oracle.gemm(An, Bp, M, N, K, dtype=dtype)
    assert np.all(oracle.decode(C, dtype) < 0)


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_k1_single_rounding(dtype):
    rng = np.random.default_rng(11)
    a = _bits(rng.uniform(-1, 1, (8, 1)), dtype)
    b = _bits(rng.uniform(-1, 1, (1, 9)), dtype)
    prod = oracle.decode(a, dtype) @ oracle.decode(b, dtype)   # one exact product each
    C = oracle.gemm(a, b, 8, 9, 1, dtype=dtype)
    assert np.array_equal(C, oracle.encode(prod, dtype))
    if dtype == oracle.F16:
        assert np.array_equal(C, f16_bits(prod))


def test_k0_gives_zero_and_degenerate_sizes():
    A = np.zeros((4, 1), np.uint16)
    C = oracle.gemm(A, A, 4, 3, 0, lda=1, ldb=3, dtype=oracle.F16, relu=True)
    assert C.shape == (4, 3) and np.all(C == 0)
    C = oracle.gemm(A, A, 0, 3, 5, lda=5, ldb=3, dtype=oracle.F16)
    assert C.shape == (0, 3)


@pytest.mark.parametrize("trans_a", [False, True])
@pytest.mark.parametrize("trans_b", [False, True])
@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_integer_products_against_numpy(trans_a, trans_b, dtype):
    """Small-integer operands: numpy's int64 product is exact; padded leading dims."""
    rng = np.random.default_rng(17 + 2 * trans_a + trans_b)
    M, N, K = 45, 29, 70
    lo, hi = (-2, 3) if dtype == oracle.F16 else (-1, 2)
    Ai = rng.integers(lo, hi, (M, K))
    Bi = rng.integers(lo, hi, (K, N))
    want = Ai @ Bi
    pad = 3
    As = Ai.T if trans_a else Ai
    Bs = Bi.T if trans_b else Bi
    Ast = np.zeros((As.shape[0], As.shape[1] + pad), np.int64)
    Ast[:, :As.shape[1]] = As
    Bst = np.zeros((Bs.shape[0], Bs.shape[1] + pad), np.int64)
    Bst[:, :Bs.shape[1]] = Bs
    Ab, Bb = _bits(Ast, dtype), _bits(Bst, dtype)
    C = oracle.gemm(Ab, Bb, M, N, K, lda=Ast.shape[1], ldb=Bst.shape[1], ldc=N + 5,
                    dtype=dtype, trans_a=trans_a, trans_b=trans_b)
    assert np.array_equal(oracle.decode(C, dtype), want.astype(np.float64))
    Cr = oracle.gemm(Ab, Bb, M, N, K, lda=Ast.shape[1], ldb=Bst.shape[1], dtype=dtype,
                     trans_a=trans_a, trans_b=trans_b, relu=True)
    assert np.array_equal(oracle.decode(Cr, dtype), np.maximum(want, 0).astype(np.float64))


def test_exact_rational_sums_within_binary64_bound():
    """Random fp16 operands: the oracle's binary64 sum is within K*2^-53*sum|terms| of the
    exact rational sum, and its rounded output matches the correctly rounded exact sum
    wherever the exact sum is not within that bound of a tie."""
    rng = np.random.default_rng(21)
    M, N, K = 6, 7, 33
    A = _bits(rng.uniform(-1, 1, (M, K)), oracle.F16)
    B = _bits(rng.uniform(-1, 1, (K, N)), oracle.F16)
    Av, Bv = oracle.decode(A, oracle.F16), oracle.decode(B, oracle.F16)
    C, S = oracle.gemm(A, B, M, N, K, dtype=oracle.F16, want_sums=True)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(Av[i, k])) * Fraction(float(Bv[k, j])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = K * 2.0 ** -53 * float(sum(abs(t) for t in terms))
            assert abs(Fraction(float(S[i, j])) - exact) <= Fraction(bound)
            assert C[i, j] == f16_bits(float(exact))


def test_entries_match_full_product_and_threads_do_not_change_bits():
    rng = np.random.default_rng(31)
    M, N, K = 50, 40, 300
    A = _bits(rng.uniform(-1, 1, (K, M)), oracle.BF16)
    B = _bits(rng.uniform(-1, 1, (N, K)), oracle.BF16)
    kw = dict(dtype=oracle.BF16, trans_a=True, trans_b=True, relu=True)
    C1 = oracle.gemm(A, B, M, N, K, threads=1, **kw)
    C4 = oracle.gemm(A, B, M, N, K, threads=4, **kw)
    assert np.array_equal(C1, C4)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    E = oracle.gemm_entries(A, B, M, N, K, rows, cols, **kw)
    assert np.array_equal(E, C1[rows, cols])


def test_rejects_bad_arguments():
    A = np.zeros(16, np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(A, A, 4, 4, 4, lda=2)          # lda < K
    with pytest.raises(ValueError):
        oracle.gemm_entries(A, A, 4, 4, 4, [4], [0])   # row out of range


# ---- FP8 operands (E4M3 / E5M2) ------------------------------------------------------

FP8_TORCH = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def _codes8(values, fmt):
    """8-bit codes of `values` via torch's own float8 conversion (exact when representable)."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float32)).to(FP8_TORCH[fmt])
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_fp8_decoders_all_codes_against_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode8(codes, fmt)
    ref = torch.from_numpy(codes).view(FP8_TORCH[fmt]).to(torch.float64).numpy()
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()


def test_fp8_defining_values():
    """The formats' definitions: E4M3 (bias 7, finite only, NaN = S.1111.111) and E5M2
    (bias 15, IEEE-style infinities)."""
    d4 = lambda c: float(oracle.decode8(np.array([c], np.uint8), oracle.E4M3)[0])
    d5 = lambda c: float(oracle.decode8(np.array([c], np.uint8), oracle.E5M2)[0])
    assert d4(0x38) == 1.0 and d4(0x40) == 2.0 and d4(0xB8) == -1.0
    assert d4(0x7E) == 448.0                       # 1.75 * 2^8, the largest
    assert d4(0x01) == 2.0 ** -9                   # smallest subnormal
    assert d4(0x08) == 2.0 ** -6                   # smallest normal
    assert np.isnan(d4(0x7F)) and np.isnan(d4(0xFF))
    assert d4(0x78) == 256.0                       # exponent 15 is finite here
    assert d5(0x3C) == 1.0 and d5(0x7B) == 57344.0
    assert d5(0x7C) == np.inf and d5(0xFC) == -np.inf and np.isnan(d5(0x7D))
    assert d5(0x01) == 2.0 ** -16 and d5(0x04) == 2.0 ** -14


@pytest.mark.parametrize("out_dtype", [oracle.F16, oracle.BF16])
def test_fp8_identity_and_power_of_two_scale(out_dtype):
    """A = I (E4M3 ones) against E5M2 values: C = alpha * B exactly (every E4M3/E5M2
    value times a power of two in range is exact in fp16 and bf16)."""
    rng = np.random.default_rng(41)
    K = N = 24
    Bv = oracle.decode8(rng.integers(0, 256, (K, N)).astype(np.uint8), oracle.E5M2)
    Bv = np.where(np.isfinite(Bv) & (np.abs(Bv) <= 4096), Bv, 1.5)
    B = _codes8(Bv, oracle.E5M2)
    A = _codes8(np.eye(K), oracle.E4M3)
    for alpha in (1.0, 0.25, 4.0):
        C = oracle.gemm_fp8(A, B, K, N, K, a_fmt=oracle.E4M3, b_fmt=oracle.E5M2,
                            out_dtype=out_dtype, alpha=alpha)
        assert np.array_equal(oracle.decode(C, out_dtype), alpha * Bv)


@pytest.mark.parametrize("trans_a", [False, True])
@pytest.mark.parametrize("trans_b", [False, True])
def test_fp8_integer_products_against_numpy(trans_a, trans_b):
    """Small integers are exact in both formats; numpy's int64 product is the exact sum;
    mixed formats, padded leading dimensions, ReLU."""
    rng = np.random.default_rng(43 + 2 * trans_a + trans_b)
    M, N, K = 37, 29, 90
    Ai = rng.integers(-4, 5, (M, K))
    Bi = rng.integers(-3, 4, (K, N))
    want = Ai @ Bi
    pad = 5
    As = Ai.T if trans_a else Ai
    Bs = Bi.T if trans_b else Bi
    Ast = np.zeros((As.shape[0], As.shape[1] + pad), np.int64)
    Ast[:, :As.shape[1]] = As
    Bst = np.zeros((Bs.shape[0], Bs.shape[1] + pad), np.int64)
    Bst[:, :Bs.shape[1]] = Bs
    A8, B8 = _codes8(Ast, oracle.E4M3), _codes8(Bst, oracle.E5M2)
    kw = dict(a_fmt=oracle.E4M3, b_fmt=oracle.E5M2, out_dtype=oracle.F16,
              lda=Ast.shape[1], ldb=Bst.shape[1], trans_a=trans_a, trans_b=trans_b)
    C = oracle.gemm_fp8(A8, B8, M, N, K, ldc=N + 3, **kw)
    assert np.array_equal(oracle.decode(C, oracle.F16), want.astype(np.float64))
    Cr = oracle.gemm_fp8(A8, B8, M, N, K, relu=True, alpha=0.5, **kw)
    assert np.array_equal(oracle.decode(Cr, oracle.F16),
                          np.maximum(0.5 * want, 0).astype(np.float64))


def test_fp8_exact_rational_sums_and_entries():
    """Random E4M3 operands: the binary64 sum times alpha is within the binary64 bound of
    the exact rational value and rounds like it; sampled entries equal the full product."""
    rng = np.random.default_rng(47)
    M, N, K = 5, 6, 41
    A = _codes8(rng.uniform(-3, 3, (M, K)), oracle.E4M3)
    B = _codes8(rng.uniform(-3, 3, (N, K)), oracle.E4M3)
    Av, Bv = oracle.decode8(A, oracle.E4M3), oracle.decode8(B, oracle.E4M3)
    alpha = 0.3
    C, S = oracle.gemm_fp8(A, B, M, N, K, trans_b=True, alpha=alpha, out_dtype=oracle.F16,
                           want_sums=True)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(Av[i, k])) * Fraction(float(Bv[j, k])) for k in range(K)]
            exact = Fraction(alpha) * sum(terms, Fraction(0))
            bound = (K + 1) * 2.0 ** -53 * alpha * float(sum(abs(t) for t in terms))
            assert abs(Fraction(float(S[i, j])) - exact) <= Fraction(bound)
            assert C[i, j] == f16_bits(float(exact))
    rows, cols = rng.integers(0, M, 30), rng.integers(0, N, 30)
    E = oracle.gemm_fp8_entries(A, B, M, N, K, rows, cols, trans_b=True, alpha=alpha,
                                out_dtype=oracle.F16)
    assert np.array_equal(E, C[rows, cols])


# ---- attention: O = softmax(Q K^T / sqrt(D)) V, [B, S, H, D] -------------------------

# ---- the block-scaled (MX) FP8 product ---------------------------------------------
# Pinned against: the plain FP8 oracle (all scales 2^0), a closed form over blocks of
# ones, a numpy product of torch-decoded operands scaled block by block, an exact
# scale-shift invariance, and NaN codes.


def _mx_codes(rng, shape, fmt):
    """Random finite 8-bit codes (torch's conversion of normal samples)."""
    v = torch.from_numpy(rng.normal(0.0, 2.0, shape).astype(np.float32))
    return v.to(FP8_TORCH[fmt]).view(torch.uint8).numpy()


def test_mx_unit_scales_reduce_to_the_fp8_product():
    rng = np.random.default_rng(41)
    M, N, K = 9, 11, 96
    for fa, fb in ((oracle.E4M3, oracle.E4M3), (oracle.E5M2, oracle.E4M3)):
        A, B = _mx_codes(rng, (M, K), fa), _mx_codes(rng, (N, K), fb)
        SA = np.full((M, K // 32), 127, np.uint8)
        SB = np.full((N, K // 32), 127, np.uint8)
        c, s = oracle.gemm_mx(A, B, SA, SB, M, N, K, a_fmt=fa, b_fmt=fb, want_sums=True)
        c8, s8 = oracle.gemm_fp8(A, B, M, N, K, a_fmt=fa, b_fmt=fb, trans_b=True,
                                 want_sums=True)
        assert np.array_equal(c, c8) and np.array_equal(s, s8)


def test_mx_blocks_of_ones_closed_form():
    # A = B = 1.0: C[i,j] = sum over blocks b of 32 * 2^(SA[i,b]-127) * 2^(SB[j,b]-127)
    rng = np.random.default_rng(42)
    M, N, K = 5, 6, 128
    one = int(_codes8(np.array([1.0]), oracle.E4M3)[0])
    A = np.full((M, K), one, np.uint8)
    B = np.full((N, K), one, np.uint8)
    SA = rng.integers(110, 140, (M, K // 32)).astype(np.uint8)
    SB = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    _, s = oracle.gemm_mx(A, B, SA, SB, M, N, K, want_sums=True)
    for i in range(M):
        for j in range(N):
            want = sum(Fraction(32) * Fraction(2) ** (int(SA[i, b]) + int(SB[j, b]) - 254)
                       for b in range(K // 32))
            assert Fraction(s[i, j]) == want


def test_mx_against_numpy_blockwise_scaling():
    rng = np.random.default_rng(43)
    M, N, K = 7, 10, 160
    A, B = _mx_codes(rng, (M, K), oracle.E4M3), _mx_codes(rng, (N, K), oracle.E5M2)
    SA = rng.integers(115, 135, (M, K // 32)).astype(np.uint8)
    SB = rng.integers(115, 135, (N, K // 32)).astype(np.uint8)
    a = torch.from_numpy(A).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    b = torch.from_numpy(B).view(torch.float8_e5m2).to(torch.float64).numpy()
    a = a * np.repeat(np.exp2(SA.astype(np.float64) - 127), 32, axis=1)
    b = b * np.repeat(np.exp2(SB.astype(np.float64) - 127), 32, axis=1)
    _, s = oracle.gemm_mx(A, B, SA, SB, M, N, K, b_fmt=oracle.E5M2, want_sums=True)
    np.testing.assert_allclose(s, a @ b.T, rtol=1e-13, atol=1e-300)
    # entries computed one by one agree bit for bit with the full product
    rows, cols = np.array([0, 3, 6]), np.array([9, 0, 4])
    c = oracle.gemm_mx(A, B, SA, SB, M, N, K, b_fmt=oracle.E5M2)
    e = oracle.gemm_mx_entries(A, B, SA, SB, M, N, K, rows, cols, b_fmt=oracle.E5M2)
    assert np.array_equal(e, c[rows, cols])


def test_mx_scale_shift_invariance_and_nan_code():
    rng = np.random.default_rng(44)
    M, N, K = 4, 5, 64
    A, B = _mx_codes(rng, (M, K), oracle.E4M3), _mx_codes(rng, (N, K), oracle.E4M3)
    SA = rng.integers(120, 130, (M, 2)).astype(np.uint8)
    SB = rng.integers(120, 130, (N, 2)).astype(np.uint8)
    _, s0 = oracle.gemm_mx(A, B, SA, SB, M, N, K, want_sums=True)
    # 2^d on every A scale of block 1 and 2^-d on every B scale of block 1: same sums
    SA2, SB2 = SA.copy(), SB.copy()
    SA2[:, 1] += 3
    SB2[:, 1] -= 3
    _, s1 = oracle.gemm_mx(A, B, SA2, SB2, M, N, K, want_sums=True)
    assert np.array_equal(s0, s1)
    # doubling a row's scales doubles its row of sums exactly
    SA3 = SA.copy()
    SA3[2] += 1
    _, s3 = oracle.gemm_mx(A, B, SA3, SB, M, N, K, want_sums=True)
    assert np.array_equal(s3[2], 2 * s0[2]) and np.array_equal(np.delete(s3, 2, 0), np.delete(s0, 2, 0))
    # E8M0 255 is NaN: only the rows it scales become NaN
    SA4 = SA.copy()
    SA4[1, 0] = 255
    _, s4 = oracle.gemm_mx(A, B, SA4, SB, M, N, K, want_sums=True)
    assert np.all(np.isnan(s4[1])) and np.all(np.isfinite(np.delete(s4, 1, 0)))


def test_mx_rejects_bad_arguments():
    A = np.zeros((4, 48), np.uint8)
    S = np.zeros((4, 2), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_mx(A, A, S, S, 4, 4, 48)                 # K not a multiple of 32
    with pytest.raises(ValueError):
        oracle.gemm_mx(A, A, S, S, 4, 4, 32, sfa_ld=0)       # scale rows too short


def _t16(x, dtype):
    return torch.as_tensor(np.asarray(x, np.float32)).to(
        torch.float16 if dtype == oracle.F16 else torch.bfloat16)


def _vals(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_attention_equal_scores_give_the_mean_of_v(dtype):
    """K = 0: every score is 0, softmax is uniform over the visible keys, O = mean of V
    (over all keys, or over keys 0..i when causal)."""
    rng = np.random.default_rng(51)
    B, S, H, D = 2, 9, 3, 16
    Q = _t16(rng.normal(size=(B, S, H, D)), dtype)
    K = _t16(np.zeros((B, S, H, D)), dtype)
    V = _t16(rng.normal(size=(B, S, H, D)), dtype)
    Vv = _vals(V)
    O, sums = oracle.attention(Q, K, V, dtype=dtype, want_sums=True)
    assert np.allclose(sums, np.broadcast_to(Vv.mean(axis=1, keepdims=True), Vv.shape),
                       rtol=0, atol=1e-12)
    Oc, sc = oracle.attention(Q, K, V, dtype=dtype, causal=True, want_sums=True)
    prefix = np.cumsum(Vv, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    assert np.allclose(sc, prefix, rtol=0, atol=1e-12)
    assert np.array_equal(Oc[:, 0], V[:, 0].view(torch.int16).numpy().view(np.uint16))


def test_attention_one_dominant_key_selects_its_value_row():
    """Scores differing by more than ~750 leave exp() of the others below 2^-1000: the
    output is the dominant key's V row, exactly after rounding."""
    B, S, H, D = 1, 6, 2, 64
    Q = np.zeros((B, S, H, D)); Q[..., 0] = 64.0
    K = np.zeros((B, S, H, D)); K[0, 4, :, 0] = 100.0     # s = 64*100/8 = 800 for key 4
    V = np.arange(B * S * H * D, dtype=np.float64).reshape(B, S, H, D) % 37 - 18
    Qt, Kt, Vt = (_t16(x, oracle.F16) for x in (Q, K, V))
    O = oracle.attention(Qt, Kt, Vt, dtype=oracle.F16)
    want = np.broadcast_to(V[:, 4:5], V.shape)
    assert np.array_equal(oracle.decode(O, oracle.F16), want)


def test_attention_against_numpy_softmax_and_key_permutation():
    rng = np.random.default_rng(53)
    B, S, H, D = 2, 13, 2, 32
    Q, K, V = (_t16(rng.normal(size=(B, S, H, D)), oracle.BF16) for _ in range(3))
    Qv, Kv, Vv = _vals(Q), _vals(K), _vals(V)
    for causal in (False, True):
        _, sums = oracle.attention(Q, K, V, dtype=oracle.BF16, causal=causal, want_sums=True)
        s = np.einsum("bihd,bjhd->bhij", Qv, Kv) / np.sqrt(D)
        if causal:
            s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
        p = np.exp(s - s.max(axis=-1, keepdims=True))
        p /= p.sum(axis=-1, keepdims=True)
        want = np.einsum("bhij,bjhd->bihd", p, Vv)
        assert np.allclose(sums, want, rtol=1e-12, atol=1e-13)
    perm = rng.permutation(S)
    O1 = oracle.attention(Q, K, V, dtype=oracle.BF16)
    O2 = oracle.attention(Q, K[:, perm], V[:, perm], dtype=oracle.BF16)
    assert np.array_equal(O1, O2)


def test_attention_rows_match_full_output():
    rng = np.random.default_rng(55)
    B, S, H, D = 2, 11, 3, 16
    Q, K, V = (_t16(rng.normal(size=(B, S, H, D)), oracle.F16) for _ in range(3))
    O = oracle.attention(Q, K, V, dtype=oracle.F16, causal=True)
    bs, is_, hs = rng.integers(0, B, 20), rng.integers(0, S, 20), rng.integers(0, H, 20)
    R = oracle.attention_rows(Q, K, V, bs, is_, hs, dtype=oracle.F16, causal=True)
    assert np.array_equal(R, O[bs, is_, hs])
