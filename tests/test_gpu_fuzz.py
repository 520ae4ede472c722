"""Seeded random cases across the whole plan space, each checked against the oracle.

Every case draws a shape (ragged in M, N and K), a layout (all four transposes), a
dtype, and a legal forced plan (1-CTA or CTA-pair tiles of every width, either stage
depth, any stage count that fits, stream-K forced on or off, a persistent grid below
the tile count, the operand swap, 16/32-column tiles, plain stores), or the planner's
own choice.  Operands are small integers, so every fp32 partial sum is exact and the
result must match the oracle bit for bit; the canary guard band around C checks that
every element is written once and nothing outside C is touched.  The 8-bit path, the
block-scaled 8-bit product and the attention pass get their own random cases.  The
seeds are fixed: a failure is reproducible from the case's printed parameters.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import assert_bit_exact, assert_within_tolerance, oracle_full, run_tl

pytestmark = pytest.mark.gpu

# (bm, bn, bk, max stages) of the 16-bit kernels
TILINGS16 = ((128, 64, 64, 8), (128, 128, 64, 6), (128, 256, 64, 4), (256, 128, 64, 8),
             (256, 256, 64, 6), (128, 64, 128, 4), (128, 128, 128, 3), (128, 256, 128, 2),
             (256, 128, 128, 4), (256, 256, 128, 3), (128, 16, 128, 6), (128, 32, 128, 5))


def _case16(seed):
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 700, 3))
    ta, tb = bool(rng.integers(2)), bool(rng.integers(2))
    dtype = workloads.F16 if rng.integers(2) else workloads.BF16
    relu = bool(rng.integers(2))
    plan = None
    if rng.random() < 0.85:
        bm, bn, bk, smax = TILINGS16[rng.integers(len(TILINGS16))]
        swap = int(bn < 64 and rng.random() < 0.7)
        if bn < 64:
            if swap and ta:                       # the swapped B is A: needs K-major A
                ta = False
            if not swap and not tb:               # narrow tiles need a K-major B
                tb = True
        stages = int(rng.integers(2, smax + 1))
        grid = 0 if rng.random() < 0.7 else int(rng.integers(1, 9)) * (bm // 128)
        stream_k = int(rng.choice([-1, 0, 1]))
        tma_store = -1 if rng.random() < 0.15 else 0
        plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=int(rng.integers(1, 9)),
                           grid=grid, stream_k=stream_k, swap_ab=swap, tma_store=tma_store)
    return M, N, K, ta, tb, dtype, relu, plan


@pytest.mark.parametrize("seed", range(100))
def test_random_16bit_cases_bit_exact(seed):
    M, N, K, ta, tb, dtype, relu, plan = _case16(1000 + seed)
    w = workloads.Workload("fuzz", M, N, K, dtype, ta, tb, relu, "int_small"
                           if dtype == workloads.F16 else "int_unit",
                           "int_small" if dtype == workloads.F16 else "int_unit", seed=seed)
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, M, N, K, dtype, ta, tb, relu, plan=plan)
    c.check_guards()
    ref = oracle_full(a, b, M, N, K, dtype, ta, tb, relu)
    assert_bit_exact(got, ref)


# 192- and 224-column tiles (K-major B): their own seeds, so the cases above keep theirs
TILINGS_ODD = ((256, 224, 128, 3), (256, 192, 128, 3), (128, 224, 128, 2), (128, 192, 128, 2))


@pytest.mark.parametrize("seed", range(24))
def test_random_odd_width_cases_bit_exact(seed):
    rng = np.random.default_rng(3000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 900, 3))
    ta = bool(rng.integers(2))
    dtype = workloads.F16 if rng.integers(2) else workloads.BF16
    relu = bool(rng.integers(2))
    bm, bn, bk, smax = TILINGS_ODD[rng.integers(len(TILINGS_ODD))]
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, int(rng.integers(2, smax + 1)),
                       raster_group=int(rng.integers(1, 9)),
                       grid=0 if rng.random() < 0.6 else int(rng.integers(1, 9)) * (bm // 128),
                       stream_k=int(rng.choice([-1, 0, 1])),
                       tma_store=-1 if rng.random() < 0.15 else 0)
    dist = "int_small" if dtype == workloads.F16 else "int_unit"
    w = workloads.Workload("fuzz_odd", M, N, K, dtype, ta, True, relu, dist, dist, seed=seed)
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, M, N, K, dtype, ta, True, relu, plan=plan)
    c.check_guards()
    assert_bit_exact(got, oracle_full(a, b, M, N, K, dtype, ta, True, relu))


@pytest.mark.parametrize("seed", range(40))
def test_random_fp8_cases_bit_exact(seed):
    from test_gpu_fp8 import TILINGS8, _oracle, run_fp8
    rng = np.random.default_rng(2000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 700, 3))
    ta, tb = bool(rng.integers(2)), bool(rng.integers(2))
    plan = None
    if rng.random() < 0.8:
        bm, bn, bk, smax = TILINGS8[rng.integers(len(TILINGS8))]
        if not tb and (bn // (bm // 128)) % 128 != 0:
            tb = True
        plan = tl.plan_for(0, 0, 0, bm, bn, bk, int(rng.integers(2, smax + 1)),
                           raster_group=int(rng.integers(1, 9)),
                           stream_k=int(rng.choice([-1, 0, 1])))
    w = workloads.Workload("fuzz8", M, N, K, workloads.E4M3 if rng.integers(2) else workloads.E5M2,
                           ta, tb, bool(rng.integers(2)), "int_small", "int_small", seed=seed,
                           b_dtype=workloads.E4M3 if rng.integers(2) else workloads.E5M2,
                           out_dtype=workloads.F16 if rng.integers(2) else workloads.BF16,
                           alpha=float(2.0 ** int(rng.integers(-3, 3))))
    a, b = workloads.make_inputs(w)
    assert_bit_exact(run_fp8(w, a, b, plan=plan), _oracle(w, a, b))


@pytest.mark.parametrize("seed", range(24))
def test_random_attention_cases(seed):
    from test_gpu_attention import _inputs, _run
    rng = np.random.default_rng(3000 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    S = int(rng.integers(1, 700))
    D = int(rng.choice([64, 128]))
    causal = bool(rng.integers(2))
    dtype = torch.float16 if rng.integers(2) else torch.bfloat16
    q, k, v = _inputs(B, S, H, D, dtype, 4000 + seed)
    got = _run(q, k, v, causal)
    code = oracle.F16 if dtype == torch.float16 else oracle.BF16
    ref = oracle.attention(q, k, v, dtype=code, causal=causal)
    assert_within_tolerance(got.reshape(-1, D), ref.reshape(-1, D), code)


@pytest.mark.parametrize("seed", range(24))
def test_random_block_scaled_cases_bit_exact(seed):
    from test_gpu_mx import _oracle, run_mx
    rng = np.random.default_rng(5000 + seed)
    M, N = (int(x) for x in rng.integers(1, 700, 2))
    K = 32 * int(rng.integers(1, 48))
    w = workloads.MxWorkload("fuzzmx", M, N, K,
                             a_fmt=workloads.E4M3 if rng.integers(2) else workloads.E5M2,
                             b_fmt=workloads.E4M3 if rng.integers(2) else workloads.E5M2,
                             out_dtype=workloads.F16 if rng.integers(2) else workloads.BF16,
                             relu=bool(rng.integers(2)), dist="int_small", sf_lo=126,
                             sf_hi=128, sf_pad=16 * int(rng.integers(0, 3)), seed=seed)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    assert_bit_exact(run_mx(w, a, b, sa, sb), _oracle(w, a, b, sa, sb))
