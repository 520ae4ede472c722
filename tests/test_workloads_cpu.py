"""The seeded input generators on CPU: determinism, storage layouts, the integer
variants' exactness bound, and the MX encoding of the block-scaled workloads (per block
of 32 K elements, the shared exponent floor(log2 max|x|) minus the element format's
largest exponent, the elements x / 2^exponent clamped to the format's largest value).
The generators hold none of the method's arithmetic; these tests pin the input recipe,
not the GEMM."""
import math

import numpy as np
import pytest
import torch

import workloads


def _bits(t):
    return t.contiguous().view(torch.uint8).numpy()


def test_draws_are_seeded_and_in_storage_layout():
    for trans_a, trans_b in ((False, False), (True, True)):
        w = workloads.Workload("t", 70, 90, 130, workloads.BF16, trans_a, trans_b, False,
                               "uniform", "normal", seed=5)
        a1, b1 = workloads.make_inputs(w)
        a2, b2 = workloads.make_inputs(w)
        assert np.array_equal(_bits(a1), _bits(a2)) and np.array_equal(_bits(b1), _bits(b2))
        assert tuple(a1.shape) == ((130, 70) if trans_a else (70, 130))
        assert tuple(b1.shape) == ((90, 130) if trans_b else (130, 90))
        assert a1.dtype == b1.dtype == torch.bfloat16
        a3, _ = workloads.make_inputs(w, seed=6)
        assert not np.array_equal(_bits(a1), _bits(a3))
        assert float(a1.abs().max()) <= 1.0             # U[-1, 1]


def test_every_workload_names_its_shapes_and_seed():
    seeds = set()
    for name, w in workloads.WORKLOADS.items():
        assert w.name == name and w.M > 0 and w.N > 0 and w.K > 0
        assert w.flops == 2 * w.M * w.N * w.K
        assert w.a_shape() == ((w.K, w.M) if w.trans_a else (w.M, w.K))
        assert w.b_shape() == ((w.N, w.K) if w.trans_b else (w.K, w.N))
        seeds.add(w.seed)
    assert len(seeds) == len(workloads.WORKLOADS)     # independent draws per workload
    assert workloads.HEADLINE in workloads.WORKLOADS
    # the headline: the largest square product, at the planner's own tiling
    hw = workloads.WORKLOADS[workloads.HEADLINE]
    assert (hw.M, hw.N, hw.K, hw.trans_b, hw.plan) == (8192, 8192, 8192, True, None)
    # the quickstart workload keeps the pages' fixed tiling
    assert workloads.WORKLOADS["gemm_relu_1024_f16_128x128x64s3"].plan == (128, 128, 64, 3)


def test_integer_variants_keep_every_fp32_partial_sum_exact():
    # |entries| <= 2 (fp16) or 1 (bf16): a partial sum is bounded by 4K (or K), below
    # 2^24 for every K the workloads use, so fp32 adds it exactly in any order
    k_max = max(w.K for w in workloads.WORKLOADS.values())
    assert 4 * k_max < 2 ** 24
    w = workloads.integer_variant(workloads.WORKLOADS["gemm_relu_1024_f16_128x128x64s3"],
                                  M=64, N=48, K=200)
    a, b = workloads.make_inputs(w)
    assert set(a.float().unique().tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    wb = workloads.integer_variant(workloads.WORKLOADS["gemm_4096_bf16_tb"], M=64, N=48,
                                   K=200)
    a, b = workloads.make_inputs(wb)
    assert set(b.float().unique().tolist()) <= {-1.0, 0.0, 1.0}


@pytest.mark.parametrize("fmt,emax,vmax", [(workloads.E4M3, 8, 448.0),
                                           (workloads.E5M2, 15, 57344.0)])
def test_mx_encoding_of_random_rows(fmt, emax, vmax):
    w = workloads.MxWorkload("t", 40, 24, 320, a_fmt=fmt, b_fmt=fmt, seed=9, sf_pad=16)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    assert tuple(a.shape) == (40, 320) and tuple(b.shape) == (24, 320)
    assert tuple(sa.shape) == (40, w.sf_ld) and w.sf_ld == 16 * math.ceil(4 * 3 / 16) + 16
    # redraw the same values to compare with the encoding
    g = torch.Generator().manual_seed(9)
    xa = torch.randn((40, 320), generator=g, dtype=torch.float32)
    nblk = 320 // 32
    vals = a.to(torch.float32).reshape(40, nblk, 32)
    amax = xa.reshape(40, nblk, 32).abs().amax(dim=-1)
    e = torch.floor(torch.log2(amax)) - emax
    assert torch.equal(sa[:, :nblk].to(torch.int64), (e + 127).to(torch.int64))
    assert torch.all(sa[:, nblk:] == 127)                 # 2^0 past K/32 and in the padding
    # each block's largest element lands in the format's top binade (clamped at vmax)
    top = vals.abs().amax(dim=-1)
    assert torch.all(top >= 2.0 ** emax) and torch.all(top <= vmax)
    # decoding codes x 2^(scale - 127) gives back x: rounding costs at most half a step
    # of the top binade (2^-4 of the block max for E4M3, 2^-3 for E5M2); clamping a
    # block max under 2^(emax+1) to vmax costs less than 1 - vmax / 2^(emax+1) = 1/8
    # of it in both formats
    dec = vals * torch.exp2(sa[:, :nblk].to(torch.float32) - 127).unsqueeze(-1)
    err = (dec - xa.reshape(40, nblk, 32)).abs()
    assert 1 - vmax / 2.0 ** (emax + 1) == 0.125
    assert torch.all(err <= 0.125 * amax.unsqueeze(-1))
    unclamped = top < vmax
    half_step = 2.0 ** -4 if fmt == workloads.E4M3 else 2.0 ** -3
    assert torch.all(err.amax(dim=-1)[unclamped] <= half_step * amax[unclamped])


def test_mx_bit_exact_variant_draws_small_codes_and_near_unit_scales():
    w = workloads.MxWorkload("t", 16, 16, 64, dist="int_small", sf_lo=126, sf_hi=128, seed=3)
    a, b, sa, sb = workloads.make_mx_inputs(w)
    assert set(a.to(torch.float32).unique().tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    assert int(sa.min()) >= 126 and int(sa.max()) <= 128
