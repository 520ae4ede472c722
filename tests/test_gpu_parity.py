"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars:
* small-integer operands: bit-exact (every fp32 partial sum is an exact integer, so
  the only rounding is the final round-to-nearest-even, identical on both sides);
* random operands: |C - C_ref| <= 1e-2 + 1e-2 |C_ref| element by element;
* full-size workloads: the whole output against the oracle (8192^3: every tile's
  edge rows and columns, the whole first and last rows and columns, and random
  entries, computed one by one), their small-integer variants bit for bit in full
  against the exact integer product, and the canary guard band for coverage.
"""
import dataclasses
import itertools

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import (GuardedC, assert_bit_exact, assert_within_tolerance,
                         exact_integer_product, oracle_full, run_tl, sample_indices,
                         to_device_padded)

pytestmark = pytest.mark.gpu

F16, BF16 = workloads.F16, workloads.BF16
GUARD_ODD = 65            # C one element past a 128-byte boundary: not 16-byte aligned


def _w(M, N, K, dtype, ta, tb, relu, dist, seed):
    return workloads.Workload("t", M, N, K, dtype, ta, tb, relu, dist, dist, seed=seed)


def _check_full(w, plan=None, exact=False, **kw):
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu, plan=plan, **kw)
    c.check_guards()
    ref = oracle_full(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    if exact:
        assert_bit_exact(got, ref)
    return assert_within_tolerance(got, ref, w.dtype)


# ------------------------------------------------------------- ragged, all layouts --

@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("relu", [False, True])
def test_ragged_all_transposes_integer_bit_exact(dtype, ta, tb, relu):
    dist = "int_small" if dtype == F16 else "int_unit"
    _check_full(_w(300, 520, 200, dtype, ta, tb, relu, dist, 3), exact=True)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_ragged_all_transposes_random_tolerance(dtype, ta, tb):
    _check_full(_w(333, 777, 515, dtype, ta, tb, True, "uniform", 4))


# ------------------------------------------------------------------ every tiling --

# (bm, bn, bk, max stages): bm = 256 is a CTA pair sharing each MMA (cta_group::2);
# bk = 128 stages hold two 64-element K chunks
TILINGS = ((128, 64, 64, 8), (128, 128, 64, 6), (128, 256, 64, 4), (256, 128, 64, 8),
           (256, 256, 64, 6), (128, 64, 128, 4), (128, 128, 128, 3), (128, 256, 128, 2),
           (256, 128, 128, 4), (256, 256, 128, 3))
PLANS = [(bm, bn, bk, s) for bm, bn, bk, smax in TILINGS for s in range(2, smax + 1)]


@pytest.mark.parametrize("bm,bn,bk,stages", PLANS)
def test_every_tiling_integer_bit_exact(bm, bn, bk, stages):
    # ragged K and N: 2-D boxes with zero fill at the edges
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=3)
    w = _w(bm * 3 + 17, bn * 2 + 40, 64 * 9 + 7, F16, stages % 2 == 1, bn == 128, True,
           "int_small", bm + bn + stages)
    _check_full(w, plan=plan, exact=True)


@pytest.mark.parametrize("bm,bn,bk,stages", [p for p in PLANS if p[3] in (2, 3)])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_every_tiling_aligned_shapes_bit_exact(bm, bn, bk, stages, ta, tb):
    # M, N, K multiples of 64: the 3-D one-box-per-stage maps are used where they apply
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=2)
    w = _w(bm * 2 + 64, bn * 2 + 64, 64 * 11, BF16, ta, tb, False, "int_unit",
           bm + bn + bk + stages + 2 * ta + tb)
    _check_full(w, plan=plan, exact=True)


@pytest.mark.parametrize("bn,bk", [(128, 64), (256, 64), (128, 128), (256, 128)])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_cta_pairs_all_transposes_random(bn, bk, ta, tb):
    plan = tl.plan_for(0, 0, 0, 256, bn, bk, 3, raster_group=2)
    _check_full(_w(700, 900, 515, BF16, ta, tb, False, "uniform", 70 + bn + bk), plan=plan)
    _check_full(_w(768, 1024, 640, BF16, ta, tb, False, "uniform", 71 + bn + bk), plan=plan)


# Tiles of 192 and 224 columns (K-major B only): 64-column epilogue steps, plus, for 224,
# a last 32-column step written by plain stores; the second accumulator at column 256.
ODD = [(bm, bn, s) for bm in (128, 256) for bn in (192, 224) for s in (2, 3)
       if bm == 256 or s == 2]                      # one CTA: 2 stages fit shared memory


@pytest.mark.parametrize("bm,bn,stages", ODD)
@pytest.mark.parametrize("ta", [False, True])
def test_odd_width_tiles_ragged_integer_bit_exact(bm, bn, stages, ta):
    # ragged M, N and K (2-D boxes, zero fill), several tiles per CTA on a short grid
    plan = tl.plan_for(0, 0, 0, bm, bn, 128, stages, raster_group=3, grid=2 * bm // 128)
    w = _w(bm * 3 + 17, bn * 3 + 40, 64 * 9 + 7, F16, ta, True, True, "int_small",
           bm + bn + stages + ta)
    _check_full(w, plan=plan, exact=True)


@pytest.mark.parametrize("bm,bn", [(128, 192), (128, 224), (256, 192), (256, 224)])
@pytest.mark.parametrize("ta", [False, True])
def test_odd_width_tiles_aligned_and_random(bm, bn, ta):
    # 3-D one-box-per-stage maps; then random inputs within tolerance
    plan = tl.plan_for(0, 0, 0, bm, bn, 128, 3 if bm == 256 else 2, raster_group=2)
    _check_full(_w(bm * 2 + 64, bn * 2, 128 * 5, BF16, ta, True, False, "int_unit",
                   bm + bn + 5 * ta), plan=plan, exact=True)
    _check_full(_w(bm * 2 + 5, bn * 3 + 7, 700, BF16, ta, True, True, "uniform", bm + bn + 9),
                plan=plan)


@pytest.mark.parametrize("bm,bn", [(256, 224), (128, 224), (256, 192)])
def test_odd_width_tiles_stream_k_bit_exact(bm, bn):
    # the last waves split by k-block: partial sums of the 32-column tail step included
    plan = tl.plan_for(0, 0, 0, bm, bn, 128, 3 if bm == 256 else 2, stream_k=1)
    w = _w(1100, 2000, 1536 + 64, F16, False, True, True, "int_small", bm + bn + 11)
    _check_full(w, plan=plan, exact=True)


def test_odd_width_tiles_unaligned_c_plain_stores():
    # C at an odd element offset: every step, the 64-column ones included, by plain stores
    plan = tl.plan_for(0, 0, 0, 256, 224, 128, 3)
    w = _w(600, 500, 384, BF16, False, True, False, "int_unit", 77)
    _check_full(w, plan=plan, exact=True, ldc=507, c_off=GUARD_ODD)


# Cluster split-K: two CTAs of a cluster share each tile's k-blocks; the second hands its
# fp32 partial sum to the first through distributed shared memory.
KSPLIT_CASES = [
    # bn, bk, stages, M, N, K, grid (0: one cluster per tile), trans_a, trans_b
    (128, 64, 3, 1024, 1024, 1024, 0, False, False),   # the quickstart tiling
    (128, 64, 3, 1000, 900, 777, 0, True, False),      # ragged K: 13 k-blocks, 6 + 7
    (64, 128, 3, 300, 520, 1000, 0, False, True),      # 8 k-blocks of 128
    (128, 128, 2, 400, 384, 2048, 0, True, True),
    (128, 64, 3, 700, 900, 515, 4, False, True),       # 2 clusters walking 48 tiles
    (64, 64, 4, 257, 333, 128, 6, True, True),         # 2 k-blocks: one each; 3 clusters
    (64, 64, 4, 129, 200, 320, 0, False, False),       # 5 k-blocks: 2 + 3
]


@pytest.mark.parametrize("bn,bk,stages,M,N,K,grid,ta,tb", KSPLIT_CASES)
def test_cluster_split_k_bit_exact(bn, bk, stages, M, N, K, grid, ta, tb):
    plan = tl.plan_for(0, 0, 0, 128, bn, bk, stages, raster_group=3, grid=grid, ksplit=2)
    p = tl.tl_plan_complete(M, N, K, 128, bn, bk, stages, trans_a=int(ta), trans_b=int(tb),
                            num_sms=152, raster_group=3, grid=grid, ksplit=2)
    assert p.ksplit == 2 and p.grid % 2 == 0 and p.sk_iters == 0
    w = _w(M, N, K, F16, ta, tb, True, "int_small", bn + bk + M + K)
    _check_full(w, plan=plan, exact=True)
    _check_full(_w(M, N, K, BF16, ta, tb, False, "uniform", bn + K), plan=plan)


@pytest.mark.parametrize("bn,stages,M", [(16, 6, 16), (32, 5, 30)])
def test_cluster_split_k_with_the_operand_swap_bit_exact(bn, stages, M):
    # skinny products: C^T tiles of 128 x bn, k-blocks shared by a cluster of two
    plan = tl.plan_for(0, 0, 0, 128, bn, 128, stages, swap_ab=1, ksplit=2)
    w = _w(M, 2000, 1536 + 40, BF16, False, True, False, "int_unit", bn + M)
    _check_full(w, plan=plan, exact=True)


def test_cluster_split_k_deterministic_over_repeats_and_graph_replay():
    w = _w(640, 768, 1000, BF16, False, True, True, "normal_over_sqrtk", 52)
    plan = tl.plan_for(0, 0, 0, 128, 128, 64, 3, ksplit=2)
    a, b = workloads.make_inputs(w)
    got1, _ = run_tl(a, b, w.M, w.N, w.K, w.dtype, False, True, True, plan=plan)
    got2, _ = run_tl(a, b, w.M, w.N, w.K, w.dtype, False, True, True, plan=plan)
    assert np.array_equal(got1, got2)
    ad, bd = a.cuda(), b.cuda()
    out = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tl.gemm(ad, bd, trans_b=True, relu=True, out=out, plan=plan, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), got1)


# stream-K: the k-blocks of the last waves split evenly over all units, partial sums
# added by each split tile's finisher
SPLIT_CASES = [
    # bm, bn, bk, stages, M, N, K, grid
    (128, 128, 64, 3, 1024, 1024, 1024, 0),      # quickstart tiling: 64 tiles over all SMs
    (128, 64, 64, 4, 300, 520, 200, 0),          # short K: tiles split over many units
    (128, 256, 64, 4, 1000, 900, 777, 0),        # ragged K: 2-D boxes
    (256, 256, 128, 3, 2048, 2048, 1536, 0),     # pairs, 3-D boxes, DP waves then split
    (256, 128, 64, 3, 700, 900, 515, 6),         # pairs, few units
    (128, 64, 128, 4, 16, 8192, 2048, 0),        # skinny
    (128, 128, 64, 3, 512, 512, 64, 0),          # one k-block: nothing to split
]


@pytest.mark.parametrize("bm,bn,bk,stages,M,N,K,grid", SPLIT_CASES)
def test_stream_k_split_bit_exact(bm, bn, bk, stages, M, N, K, grid):
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=3, grid=grid, stream_k=1)
    _check_full(_w(M, N, K, F16, False, bn == 128, True, "int_small", M + N + K + bm),
                plan=plan, exact=True)
    _check_full(_w(M, N, K, BF16, True, False, False, "uniform", M + N + K + bn), plan=plan)


# Skinny products on C^T (swap_ab): the kernel's rows are N, its narrow columns M, and
# it writes C transposed with plain stores.  Narrow tiles (bn 16, 32) need A K-major.
SWAP_CASES = [
    # bn, stages, M, N, K, trans_a, trans_b, stream_k
    (16, 6, 1, 1000, 1100, False, True, 1),       # one row of C, ragged N and K
    (16, 6, 16, 2100, 1024, False, False, 1),     # M-major B (the kernel's A)
    (16, 4, 7, 300, 777, False, True, -1),        # whole tiles, ragged K tail
    (32, 5, 17, 1300, 2000, False, True, 1),
    (32, 3, 32, 129, 130, False, False, -1),
    (64, 4, 64, 2000, 1500, True, True, 1),       # M-major A needs 64-wide boxes
    (64, 4, 50, 700, 300, True, False, -1),
    (128, 3, 128, 1500, 2100, False, True, 1),
    (128, 3, 100, 333, 1000, True, True, 0),
]


@pytest.mark.parametrize("bn,stages,M,N,K,ta,tb,sk", SWAP_CASES)
def test_swapped_operands_for_skinny_products(bn, stages, M, N, K, ta, tb, sk):
    plan = tl.plan_for(0, 0, 0, 128, bn, 128, stages, raster_group=4, stream_k=sk, swap_ab=1)
    _check_full(_w(M, N, K, F16, ta, tb, True, "int_small", M + N + K + bn),
                plan=plan, exact=True)
    _check_full(_w(M, N, K, BF16, ta, tb, False, "uniform", M + N + K + 3), plan=plan)


# C^T with C's pitch a multiple of 8 elements goes out by 16-byte stores after an 8 x 8
# transpose across lanes: a ragged N (the kernel's rows) ends inside a vector, a ragged
# M inside a transposed block; the guards also cover the pitch padding
SWAP_VEC_CASES = [
    # bn, stages, M, N, K, ldc, ksplit
    (16, 6, 13, 1003, 900, 1008, 1),
    (16, 6, 16, 2048, 1536, 2048, 2),
    (32, 5, 30, 2001, 1536, 2008, 2),
    (64, 4, 61, 517, 640, 520, 2),
    (128, 3, 100, 333, 1000, 336, 1),
    (128, 3, 128, 1030, 1024, 1040, 2),
]


@pytest.mark.parametrize("bn,stages,M,N,K,ldc,ks", SWAP_VEC_CASES)
def test_swapped_operands_vector_stores(bn, stages, M, N, K, ldc, ks):
    plan = tl.plan_for(0, 0, 0, 128, bn, 128, stages, raster_group=4, swap_ab=1, ksplit=ks)
    _check_full(_w(M, N, K, F16, False, True, True, "int_small", M + N + bn), plan=plan,
                exact=True, ldc=ldc)
    _check_full(_w(M, N, K, BF16, False, True, False, "uniform", M + K + bn), plan=plan,
                ldc=ldc)


@pytest.mark.parametrize("bn,stages", [(16, 6), (32, 5)])
def test_narrow_tiles_without_swap(bn, stages):
    # N itself narrow: bn 16/32 tiles of C with a K-major B (trans_b)
    plan = tl.plan_for(0, 0, 0, 128, bn, 128, stages, raster_group=2)
    _check_full(_w(700, bn + 5, 900, BF16, False, True, True, "int_unit", 71 + bn),
                plan=plan, exact=True)
    _check_full(_w(300, bn - 3, 1300, F16, True, True, False, "uniform", 72 + bn), plan=plan)


@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_one_wave_of_narrow_tiles_auto_plan(ta, tb):
    # the planner's own pick when every 128 x 64 tile has an SM: ragged M, N and K, the
    # last k-block partial
    M, N, K = 700, 650, 1100
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = tl.tl_gemm_plan(M, N, K, F16, int(ta), int(tb), sms)
    assert (p.bm, p.bn, p.bk, p.sk_iters) == (128, 64, 128, 0)
    if ta == tb:
        _check_full(_w(M, N, K, F16, ta, tb, True, "int_small", 81 + ta), exact=True)
    else:
        _check_full(_w(M, N, K, BF16, ta, tb, False, "uniform", 85 + ta))


@pytest.mark.parametrize("bm,bn,bk,stages", [(128, 64, 64, 4), (128, 256, 128, 2),
                                             (256, 128, 64, 3), (256, 256, 128, 3)])
def test_plain_stores_instead_of_tma_stores(bm, bn, bk, stages):
    # tma_store = -1: C from registers, 16-byte vectors for whole chunks, scalars at the
    # ragged right edge
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, raster_group=3, tma_store=-1)
    _check_full(_w(333, 64 * 7 + 40, 700, F16, False, True, True, "int_small", bm + bn + 5),
                plan=plan, exact=True)
    _check_full(_w(512, 512, 256, BF16, True, False, False, "uniform", bm + bn + 6), plan=plan)


def test_stream_k_results_are_deterministic_and_replay_in_graphs():
    w = _w(1024, 1024, 1024, F16, False, False, True, "uniform", 90)
    a, b = workloads.make_inputs(w)
    ad, bd = a.cuda(), b.cuda()
    plan = tl.plan_for(0, 0, 0, 128, 128, 64, 3, stream_k=1)
    outs = []
    for _ in range(3):
        outs.append(tl.gemm(ad, bd, relu=True, plan=plan).cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    out = torch.empty(1024, 1024, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tl.gemm(ad, bd, relu=True, out=out, plan=plan, stream=s)
    for _ in range(3):                      # replays reuse the launch's flags and token
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), outs[0])
    st, word = tl.tl_device_status(reset=True)
    assert st == tl.TL_OK, hex(word)


@pytest.mark.parametrize("l2_prefetch", [0, 1, 3, 5, 100])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, True)])
def test_l2_prefetch_distances(l2_prefetch, ta, tb):
    plan = tl.plan_for(0, 0, 0, 128, 128, 64, 3, raster_group=4, l2_prefetch=l2_prefetch)
    _check_full(_w(400, 700, 64 * 11 + 9, F16, ta, tb, True, "int_small", 60 + l2_prefetch),
                plan=plan, exact=True)


@pytest.mark.parametrize("bm,grid", [(128, 1), (128, 2), (128, 7), (256, 2), (256, 6)])
def test_persistent_ctas_cover_every_tile_once(bm, grid):
    # fewer CTAs than tiles: each CTA (pair) walks several tiles and both accumulator
    # buffers
    plan = tl.plan_for(0, 0, 0, bm, 128, 64, 4, raster_group=2, grid=grid)
    _check_full(_w(700, 900, 300, BF16, False, True, False, "int_unit", 30 + grid),
                plan=plan, exact=True)


# ------------------------------------------------------------------- tiny shapes --

TINY = [1, 2, 3, 7, 16, 17, 63, 64, 65, 127, 128, 129]


@pytest.mark.parametrize("M,N,K", [(m, n, k) for m, n, k in itertools.product(TINY, TINY, TINY)
                                   if (m * 7 + n * 3 + k) % 23 == 0][:40] + [(1, 1, 1), (129, 129, 129)])
def test_tiny_shapes(M, N, K):
    _check_full(_w(M, N, K, F16, False, False, True, "int_small", M * 1000 + N * 10 + K),
                exact=True)
    _check_full(_w(M, N, K, BF16, True, True, False, "uniform", M + N + K))


def test_k_zero_fills_zero_and_empty_outputs_are_untouched():
    a = torch.zeros(4, 1, dtype=torch.float16)
    got, c = run_tl(a, torch.zeros(1, 5, dtype=torch.float16), 4, 5, 0, F16, relu=True,
                    lda=1, ldb=5, ldc=8)
    c.check_guards()
    assert np.all(got == 0)
    c = GuardedC(1, 1, 1, torch.float16)
    for M, N in ((0, 5), (5, 0)):
        assert tl.tl_gemm(0, 0, c.ptr, M, N, 3, 3, max(N, 1), max(N, 1), F16, 0, 0, 0,
                          0) == tl.TL_OK
    torch.cuda.synchronize()
    assert np.all(c.host_bits() == 0x7E55)


# ------------------------------------------------ pitches the TMA unit cannot use --

def test_unaligned_lda_is_repacked():
    # lda = K = 4100 fp16 is 8200 bytes: not a multiple of 16
    _check_full(_w(300, 264, 4100, F16, False, False, True, "int_small", 40), exact=True)


def test_offset_operands_and_unaligned_c():
    w = _w(200, 136, 300, BF16, False, True, True, "int_unit", 41)
    a, b = workloads.make_inputs(w)
    ref = oracle_full(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    # A and B start 2 bytes past alignment, C has an odd leading dimension and offset
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu,
                    a_off=1, b_off=3, ldc=139, c_off=65)
    c.check_guards()
    assert_bit_exact(got, ref)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu,
                    lda=305, ldb=301)
    c.check_guards()
    assert_bit_exact(got, ref)


# ------------------------------------------------------------------ the workloads --

SMALL = ["gemm_relu_256_f16", "gemm_relu_1024_f16_128x128x64s3"]


def _workload_plan(w):
    if w.plan is None:
        return None
    bm, bn, bk, st = w.plan
    return tl.plan_for(0, 0, 0, bm, bn, bk, st)


@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_full_output(name):
    w = workloads.WORKLOADS[name]
    _check_full(w, plan=_workload_plan(w))
    _check_full(workloads.integer_variant(w), plan=_workload_plan(w), exact=True)


# Every output element of these is compared with the oracle (the oracle takes seconds to
# about half a minute each on 16 host cores); 8192^3 is compared on the sample below.
FULL = ["gemm_4096_bf16_tb", "gemm_relu_3000x5000x4100_f16", "gemm_m16_n8192_k8192_bf16",
        "gemm_m64_n8192_k8192_bf16", "gemm_m128_n8192_k8192_bf16"]


def _scale_bound(stats, ref_bits, dtype):
    # a tighter bound that follows from the arithmetic: two roundings of nearly equal
    # sums differ by at most one unit in the last place of the output format, plus the
    # fp32 accumulation error; relative to the output's scale this stays near 2^-7
    scale = np.abs(oracle.decode(ref_bits, dtype)).max()
    assert stats["max_abs"] <= scale * 2.0 ** -6, (stats, scale)


@pytest.mark.parametrize("name", FULL)
def test_large_workloads_full_output(name):
    w = workloads.WORKLOADS[name]
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu,
                    plan=_workload_plan(w))
    c.check_guards()
    ref = oracle_full(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    stats = assert_within_tolerance(got, ref, w.dtype)
    _scale_bound(stats, ref, w.dtype)


def test_largest_square_workload_sampled():
    # 8192^3 (the oracle would take minutes): every row and column tile's first and last
    # row/column, the whole first and last rows and columns, and random entries
    w = workloads.WORKLOADS["gemm_8192_bf16_tb"]
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    c.check_guards()
    rng = np.random.default_rng(7)
    rows, cols = sample_indices(w.M, w.N, 6000, rng)
    ref = oracle.gemm_entries(a, b, w.M, w.N, w.K, rows, cols, dtype=w.dtype,
                              trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu)
    stats = assert_within_tolerance(got[rows, cols], ref, w.dtype)
    _scale_bound(stats, ref, w.dtype)


def test_unit_variance_variant_of_the_square_workload_sampled():
    # "N(0,1)/sqrt(K) entries" read for both operands gives C a standard deviation of
    # 1/sqrt(K) = 1/64, where the absolute 1e-2 term of the tolerance is loose.  With
    # A ~ N(0,1) and only B scaled, C ~ N(0,1) and the relative term decides.
    w = dataclasses.replace(workloads.WORKLOADS["gemm_4096_bf16_tb"], name="unit_variance",
                            dist_a="normal", seed=12)
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    c.check_guards()
    rng = np.random.default_rng(8)
    rows, cols = sample_indices(w.M, w.N, 6000, rng)
    ref = oracle.gemm_entries(a, b, w.M, w.N, w.K, rows, cols, dtype=w.dtype,
                              trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu)
    stats = assert_within_tolerance(got[rows, cols], ref, w.dtype)
    assert 0.8 < np.std(oracle.decode(ref, w.dtype)) < 1.25
    # the fp32 sum and the binary64 sum round to the same bf16 value except near ties,
    # where they differ by one unit in the last place (2^-7 relative at most)
    assert stats["norm_max"] <= 2.0 ** -6 and stats["rel_rms"] <= 2.0 ** -7, stats


@pytest.mark.parametrize("name", ["gemm_8192_bf16_tb", "gemm_relu_3000x5000x4100_f16",
                                  "gemm_m16_n8192_k8192_bf16"])
def test_large_workloads_integer_sampled_bit_exact(name):
    w = workloads.integer_variant(workloads.WORKLOADS[name])
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu)
    c.check_guards()
    rng = np.random.default_rng(8)
    rows, cols = sample_indices(w.M, w.N, 4000, rng)
    ref = oracle.gemm_entries(a, b, w.M, w.N, w.K, rows, cols, dtype=w.dtype,
                              trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu)
    assert_bit_exact(got[rows, cols], ref)


@pytest.mark.parametrize("name", ["gemm_8192_bf16_tb"] + FULL)
def test_large_workloads_integer_full_output_bit_exact(name):
    # small-integer operands: the exact product is an integer matrix (closed form), and
    # its round-to-nearest-even by the oracle's encoder must equal every output bit for
    # bit -- the whole of C at the full sizes, 8192^3 included
    w = workloads.integer_variant(workloads.WORKLOADS[name])
    a, b = workloads.make_inputs(w)
    got, c = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu,
                    plan=_workload_plan(w))
    c.check_guards()
    exact = exact_integer_product(a, b, w.trans_a, w.trans_b, w.relu)
    assert np.abs(exact).max() < 2 ** 24        # each fp32 partial sum is exact too
    assert_bit_exact(got, oracle.encode(exact, w.dtype))


# ------------------------------------------------------------- streams and graphs --

def test_repeated_calls_are_deterministic_and_stream_ordered():
    w = _w(640, 768, 1000, BF16, False, True, True, "normal_over_sqrtk", 50)
    a, b = workloads.make_inputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got1, _ = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu, stream=s)
        got2, _ = run_tl(a, b, w.M, w.N, w.K, w.dtype, w.trans_a, w.trans_b, w.relu, stream=s)
    assert np.array_equal(got1, got2)


def test_graph_capture_and_replay():
    w = _w(384, 512, 640, F16, False, False, True, "int_small", 51)
    a, b = workloads.make_inputs(w)
    ad, bd = a.cuda(), b.cuda()
    out = torch.empty(w.M, w.N, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tl.gemm(ad, bd, relu=True, out=out)       # first call sets kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.fill_(0)
    with torch.cuda.graph(g, stream=s):
        tl.gemm(ad, bd, relu=True, out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    ref = oracle_full(a, b, w.M, w.N, w.K, w.dtype, False, False, True)
    assert_bit_exact(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)


# ------------------------------------------------------------------------ errors --

def test_host_pointer_is_rejected():
    a = torch.zeros(64, 64, dtype=torch.float16)          # CPU memory
    c = GuardedC(64, 64, 64, torch.float16)
    st = tl.tl_gemm(a.data_ptr(), a.data_ptr(), c.ptr, 64, 64, 64, 64, 64, 64, F16, 0, 0, 0, 0)
    assert st == tl.TL_ERR_DEVICE


def test_alias_is_rejected_on_device_buffers():
    buf = torch.zeros(4096, dtype=torch.float16, device="cuda")
    p = buf.data_ptr()
    # A = [p, p + 512), B = [p + 2048, p + 2560): C at p + 256 overlaps A, at p + 2304 B
    st = tl.tl_gemm(p, p + 2048, p + 256, 16, 16, 16, 16, 16, 16, F16, 0, 0, 0, 0)
    assert st == tl.TL_ERR_ALIAS
    st = tl.tl_gemm(p, p + 2048, p + 2304, 16, 16, 16, 16, 16, 16, F16, 0, 0, 0, 0)
    assert st == tl.TL_ERR_ALIAS


def test_device_status_clean_after_all_calls():
    st, word = tl.tl_device_status(reset=False)
    assert st == tl.TL_OK, f"bounded wait gave up: {word:#x}"


def test_concurrent_streams_and_host_threads():
    # Two host threads, each with its own stream, enqueue split GEMMs (stream-K forced,
    # so each call has its own partial-sum workspace and flags), block-scaled products
    # and attention back to back with no synchronisation between them.  Every result
    # must still be the oracle's.
    import threading

    from test_gpu_mx import _oracle as mx_oracle
    plan = tl.plan_for(0, 0, 0, 128, 128, 64, 3, raster_group=3, stream_k=1)
    jobs = []
    for t in range(2):
        w = _w(700, 900, 2100, F16, False, True, True, "int_small", 80 + t)
        a, b = workloads.make_inputs(w)
        wm = workloads.MxWorkload("c", 300, 500, 1024, dist="int_small", sf_lo=126, sf_hi=128,
                                  seed=90 + t)
        am, bm, sam, sbm = workloads.make_mx_inputs(wm)
        g = torch.Generator().manual_seed(95 + t)
        qkv = [torch.randn((2, 600, 4, 64), generator=g).to(torch.bfloat16) for _ in range(3)]
        jobs.append({
            "w": w, "a": a, "b": b, "wm": wm, "mx": (am, bm, sam, sbm), "qkv": qkv,
            "dev": [x.cuda() for x in (a, b)], "dev_mx": [x.cuda() for x in (am, bm, sam, sbm)],
            "dev_qkv": [x.cuda() for x in qkv],
            "out_g": [torch.empty((w.M, w.N), dtype=torch.float16, device="cuda") for _ in range(3)],
            "out_m": [torch.empty((wm.M, wm.N), dtype=torch.bfloat16, device="cuda") for _ in range(3)],
            "out_a": [torch.empty((2, 600, 4, 64), dtype=torch.bfloat16, device="cuda")
                      for _ in range(3)]})
    torch.cuda.synchronize()
    errors = []

    def worker(job):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            for rep in range(3):
                tl.gemm(job["dev"][0], job["dev"][1], trans_b=True, relu=True,
                        out=job["out_g"][rep], plan=plan, stream=s)
                tl.gemm_mx(*job["dev_mx"], out=job["out_m"][rep], stream=s)
                tl.attention(*job["dev_qkv"], causal=True, out=job["out_a"][rep], stream=s)
            s.synchronize()
        except Exception as e:          # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    st, word = tl.tl_device_status(reset=True)
    assert st == tl.TL_OK, hex(word)
    for job in jobs:
        w, wm = job["w"], job["wm"]
        ref_g = oracle_full(job["a"], job["b"], w.M, w.N, w.K, w.dtype, False, True, True)
        ref_m = mx_oracle(wm, *job["mx"])
        ref_a = oracle.attention(*job["qkv"], dtype=oracle.BF16, causal=True)
        for rep in range(3):
            assert_bit_exact(job["out_g"][rep].cpu().view(torch.int16).numpy().view(np.uint16),
                             ref_g)
            assert_bit_exact(job["out_m"][rep].cpu().view(torch.int16).numpy().view(np.uint16),
                             ref_m)
            got_a = job["out_a"][rep].cpu().view(torch.int16).numpy().view(np.uint16)
            assert_within_tolerance(got_a.reshape(-1, 64), ref_a.reshape(-1, 64), oracle.BF16)
