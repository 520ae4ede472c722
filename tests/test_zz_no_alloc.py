"""tl_gemm_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot let a library allocate: a framework that owns all device memory
through its own pool, a serving process that has reserved nearly all HBM, a
real-time loop that must not allocate after start-up.  tl_gemm_noalloc() runs the
same GEMM as tl_gemm() but copies operands that need a padded pitch into one fixed
32 MiB device array of the library instead of asking the stream-ordered allocator.

These tests call it through the C ABI with operands that do need the copy (a
leading dimension of 4100 fp16 elements is 8200 bytes, not a multiple of 16), on two
calls in a row with different inputs, and compare each result with tl_gemm()'s
within the tolerance used by every parity test, |C - C_ref| <= 1e-2 + 1e-2 |C_ref|.
This file is collected last so that a run stopping at its first failure has run
everything else; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import GuardedC, assert_within_tolerance, to_device_padded

pytestmark = pytest.mark.gpu


def _run(entry, a_ptr, b_ptr, M, N, K, lda, ldb, dtype, relu, stream):
    c = GuardedC(M, N, N, torch.float16 if dtype == tl.TL_F16 else torch.bfloat16)
    st = entry(a_ptr, b_ptr, c.ptr, M, N, K, lda, ldb, N, dtype, 0, 0,
               tl.TL_EPI_RELU if relu else tl.TL_EPI_NONE, stream)
    assert st == tl.TL_OK, tl.tl_status_string(st)
    torch.cuda.synchronize()
    dev_st, word = tl.tl_device_status(reset=True)
    assert dev_st == tl.TL_OK, f"device-side wait gave up: {word:#x}"
    c.check_guards()
    return c.result()


def test_noalloc_matches_tl_gemm_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    shapes = [(300, 264, 4100, workloads.F16, True, 81),      # A repacked (lda 4100)
              (517, 392, 4100, workloads.F16, False, 82)]     # a second, larger call
    for M, N, K, dtype, relu, seed in shapes:
        w = workloads.Workload("noalloc", M, N, K, dtype, False, False, relu, "uniform",
                               "uniform", seed=seed)
        a_cpu, b_cpu = workloads.make_inputs(w)
        pa, lda, keep_a = to_device_padded(a_cpu)          # lda = K: needs the padded copy
        pb, ldb, keep_b = to_device_padded(b_cpu, ld=N + 1, offset=1)   # B too (odd pitch)
        assert (lda * 2) % 16 != 0 and (ldb * 2) % 16 != 0
        ref = _run(tl.tl_gemm, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
        got = _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
        assert_within_tolerance(got, ref, dtype)
        del keep_a, keep_b


def test_noalloc_rejects_operands_beyond_its_scratch():
    limit = tl.tl_gemm_noalloc_scratch_bytes()
    assert limit == 32 << 20
    M, K, N = 5000, 4100, 64          # A copy: 5000 x 4104 x 2 bytes > 32 MiB
    assert M * 4104 * 2 > limit
    a = torch.zeros(M * K + 8, dtype=torch.float16, device="cuda")
    b = torch.zeros(K * N, dtype=torch.float16, device="cuda")
    c = torch.full((M * N,), 7.0, dtype=torch.float16, device="cuda")
    st = tl.tl_gemm_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K, N, N,
                            tl.TL_F16, 0, 0, tl.TL_EPI_NONE,
                            torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((c == 7.0).all())      # nothing was enqueued
