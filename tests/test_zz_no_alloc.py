"""tl_gemm_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot let a library allocate: a framework that owns all device memory
through its own pool, a serving process that has reserved nearly all HBM, a
real-time loop that must not allocate after start-up.  tl_gemm_noalloc() runs the
same GEMM as tl_gemm() but copies operands that need a padded pitch into one fixed
32 MiB device array of the library instead of asking the stream-ordered allocator.

These tests call it through the C ABI with operands that do need the copy (a
leading dimension of 4100 fp16 elements is 8200 bytes, not a multiple of 16), on two
calls in a row with different inputs:
  * small-integer operands, bit for bit against the CPU oracle (every fp32 partial
    sum is exact, so the only rounding is the final one, the same on both sides);
  * uniform operands, against tl_gemm()'s output on the same inputs within the
    tolerance of every parity test, |C - C_ref| <= 1e-2 + 1e-2 |C_ref|;
  * a call where only B needs the copy (it then starts at the array's first byte);
  * the device's stream-ordered memory pool records no allocation during the calls,
    while a tl_gemm() call on the same operands does (the probe itself works).
This file is collected last so that a run stopping at its first failure has run
everything else; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import GuardedC, assert_bit_exact, assert_within_tolerance, to_device_padded

pytestmark = pytest.mark.gpu

CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8     # CUmemPool_attribute: high-water mark of used bytes


class DefaultPoolHighWater:
    """High-water mark of the current device's default stream-ordered memory pool, read
    and reset through the CUDA driver API (the pool the library's cudaMallocAsync draws
    from; PyTorch's own caching allocator does not use it)."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        assert self.cu.cuInit(0) == 0
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def reset(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(zero)) == 0

    def value(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(v)) == 0
        return v.value


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


# (M, N, K, dtype, relu, seed, ldb, b offset): A always needs the copy (lda = K = 4100)
CALLS = [(300, 264, 4100, workloads.F16, True, 81, 265, 1),
         (517, 392, 4100, workloads.BF16, False, 82, 393, 1)]


def _operands(M, N, K, dtype, relu, seed, ldb, b_off, dist):
    w = workloads.Workload("noalloc", M, N, K, dtype, False, False, relu, dist, dist,
                           seed=seed)
    a_cpu, b_cpu = workloads.make_inputs(w)
    pa, lda, keep_a = to_device_padded(a_cpu)                  # lda = K: needs the copy
    pb, ldb, keep_b = to_device_padded(b_cpu, ld=ldb, offset=b_off)   # odd pitch: B too
    assert (lda * 2) % 16 != 0 and (ldb * 2) % 16 != 0
    return a_cpu, b_cpu, pa, lda, pb, ldb, (keep_a, keep_b)


def test_noalloc_matches_the_oracle_bit_for_bit_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, dtype, relu, seed, ldb_, b_off in CALLS:
        dist = "int_small" if dtype == workloads.F16 else "int_unit"
        a_cpu, b_cpu, pa, lda, pb, ldb, keep = _operands(M, N, K, dtype, relu, seed, ldb_,
                                                         b_off, dist)
        got = _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
        ref = oracle.gemm(a_cpu, b_cpu, M, N, K, dtype=dtype, relu=relu)
        assert_bit_exact(got, ref)
        del keep


def test_noalloc_matches_tl_gemm_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, dtype, relu, seed, ldb_, b_off in CALLS:
        a_cpu, b_cpu, pa, lda, pb, ldb, keep = _operands(M, N, K, dtype, relu, seed + 10,
                                                         ldb_, b_off, "uniform")
        ref = _run(tl.tl_gemm, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
        got = _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
        assert_within_tolerance(got, ref, dtype)
        del keep


def test_noalloc_with_only_b_copied():
    # A aligned (K = 4096), B with an odd pitch: B's copy is the only one and starts at
    # the first byte of the array
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K = 200, 136, 4096
    w = workloads.Workload("noalloc_b", M, N, K, workloads.F16, False, False, True,
                           "int_small", "int_small", seed=84)
    a_cpu, b_cpu = workloads.make_inputs(w)
    pa, lda, keep_a = to_device_padded(a_cpu)
    pb, ldb, keep_b = to_device_padded(b_cpu, ld=N + 3, offset=1)
    assert (lda * 2) % 16 == 0 and pa % 16 == 0 and (ldb * 2) % 16 != 0
    got = _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, workloads.F16, True, stream)
    assert_bit_exact(got, oracle.gemm(a_cpu, b_cpu, M, N, K, dtype=workloads.F16, relu=True))
    del keep_a, keep_b


def test_noalloc_allocates_nothing_where_tl_gemm_does():
    stream = torch.cuda.current_stream().cuda_stream
    pool = DefaultPoolHighWater()
    M, N, K, dtype, relu, seed, ldb_, b_off = CALLS[0]
    a_cpu, b_cpu, pa, lda, pb, ldb, keep = _operands(M, N, K, dtype, relu, seed + 20, ldb_,
                                                     b_off, "uniform")
    torch.cuda.synchronize()
    pool.reset()                       # the mark restarts from the bytes in use now
    before = pool.value()
    _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
    _run(tl.tl_gemm_noalloc, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
    assert pool.value() == before, "tl_gemm_noalloc drew on the stream-ordered allocator"
    # the probe sees the workspace tl_gemm takes for the same padded copies
    _run(tl.tl_gemm, pa, pb, M, N, K, lda, ldb, dtype, relu, stream)
    assert pool.value() >= before + M * 4104 * 2
    del keep


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
