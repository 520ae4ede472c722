"""Failure detection on the GPU, without a fault: a wait that nothing ends.

Every wait in the kernel is bounded.  The library's test hook (tl_debug_set_stall)
makes the MMA thread wait on a barrier that nothing arrives on, as if its operands
never came.  With a short limit the wait runs out; the kernel must then record
TL_ERR_TIMEOUT (with the wait site) in the device status word, unwind every role
(loads already issued land, Tensor Memory is freed) and return, leaving the context
usable: the next, normal call on the same stream must give the right answer.
"""
import numpy as np
import pytest
import torch

import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import assert_bit_exact, oracle_full

pytestmark = pytest.mark.gpu

SITE_INJECTED = 7
DEFAULT_TIMEOUT_NS = 1_000_000_000


@pytest.fixture
def short_limit():
    tl.tl_device_status(reset=True)
    tl.tl_set_wait_timeout_ns(2_000_000)          # 2 ms of waiting at a 4 GHz count
    try:
        yield
    finally:
        tl.tl_debug_set_stall(0)
        tl.tl_set_wait_timeout_ns(DEFAULT_TIMEOUT_NS)
        torch.cuda.synchronize()
        tl.tl_device_status(reset=True)


@pytest.mark.parametrize("bm,bn,bk,stages,ksplit", [(128, 128, 64, 3, 1), (128, 128, 64, 3, 2),
                                                    (256, 256, 128, 3, 0)])
def test_a_wait_that_nothing_ends_times_out_and_the_context_survives(short_limit, bm, bn, bk,
                                                                     stages, ksplit):
    # ksplit 2: two CTAs of a cluster per tile, both stalled, their partial-sum hand-over
    # never reached
    w = workloads.Workload("stall", 600, 700, 1000, workloads.F16, False, False, True,
                           "int_small", "int_small", seed=bm + bn)
    a, b = workloads.make_inputs(w)
    ad, bd = a.cuda(), b.cuda()
    plan = tl.plan_for(0, 0, 0, bm, bn, bk, stages, ksplit=ksplit)
    out = torch.full((w.M, w.N), 3.0, dtype=torch.float16, device="cuda")

    tl.tl_debug_set_stall(1)
    tl.gemm(ad, bd, relu=True, out=out, plan=plan)      # enqueues fine
    tl.tl_debug_set_stall(0)
    st, word = tl.tl_device_status(reset=True)          # synchronises
    assert st == tl.TL_ERR_TIMEOUT, (st, hex(word))
    assert word & 0xFF == tl.TL_ERR_TIMEOUT
    if bm == 128:       # one CTA per tile: the injected wait is the first to run out
        assert (word >> 8) & 0xFF == SITE_INJECTED, hex(word)
    assert torch.cuda.current_stream().query()          # nothing left running

    # the same stream, the same buffers: a normal call now gives the exact result
    tl.gemm(ad, bd, relu=True, out=out, plan=plan)
    torch.cuda.synchronize()
    st, word = tl.tl_device_status(reset=True)
    assert st == tl.TL_OK, hex(word)
    ref = oracle_full(a, b, w.M, w.N, w.K, w.dtype, False, False, True)
    assert_bit_exact(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)
