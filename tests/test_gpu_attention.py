"""GPU parity of the attention forward pass (tl_attention_fwd) against the CPU oracle.

O = softmax(Q K^T / sqrt(D)) V over [B, S, H, D], causal or not.  The kernel keeps
scores and softmax statistics in fp32 but, like the pages' kernel, feeds the
probabilities to the PV product rounded to the 16-bit type, so the comparison is
within the tolerance |O - O_ref| <= 1e-2 + 1e-2 |O_ref| rather than bit-exact.
Closed forms that the rounding cannot disturb are checked exactly: with K = 0 every
probability is the same power-of-two fraction, and the first causal row is V[0].
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_gemm_gb300 as tl
import workloads
from gpu_helpers import assert_bit_exact, assert_within_tolerance

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _inputs(B, S, H, D, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn((B, S, H, D), generator=g) * scale).to(dtype) for _ in range(3)]


def _run(q, k, v, causal):
    B, S, H, D = q.shape
    guard = 256
    buf = torch.full((q.numel() + 2 * guard,), 0x7E55, dtype=torch.int16, device="cuda")
    out = buf[guard:guard + q.numel()].view(q.dtype).view(q.shape)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    st = tl.tl_attention_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B, S, H,
                             D, tl.TL_F16 if q.dtype == torch.float16 else tl.TL_BF16,
                             int(causal), torch.cuda.current_stream().cuda_stream)
    assert st == tl.TL_OK, tl.tl_status_string(st)
    torch.cuda.synchronize()
    dev_st, word = tl.tl_device_status(reset=True)
    assert dev_st == tl.TL_OK, f"device-side wait gave up: {word:#x}"
    b = _bits(buf)
    assert np.all(b[:guard] == 0x7E55) and np.all(b[-guard:] == 0x7E55), "guard band written"
    return _bits(out)


CASES = [
    # B, S, H, D, causal
    (1, 128, 1, 64, False),
    (1, 128, 1, 64, True),
    (2, 300, 3, 64, False),        # ragged last tile of queries and keys
    (2, 300, 3, 64, True),
    (1, 1000, 2, 128, True),
    (1, 1000, 2, 128, False),
    (3, 77, 2, 128, False),        # one tile, mostly past the end
    (1, 1, 4, 64, True),           # a single position
    (1, 513, 1, 128, True),
]


@pytest.mark.parametrize("B,S,H,D,causal", CASES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_attention_against_oracle(B, S, H, D, causal, dtype):
    code = oracle.F16 if dtype == torch.float16 else oracle.BF16
    q, k, v = _inputs(B, S, H, D, dtype, B * 1000 + S + H + D + int(causal))
    got = _run(q, k, v, causal)
    ref = oracle.attention(q, k, v, dtype=code, causal=causal)
    assert_within_tolerance(got.reshape(-1, D), ref.reshape(-1, D), code)


def _sampled_rows(B, S, H, rng, n):
    """Row indices spread over every batch, head and position, with the first and last
    query of every 128-tile among them."""
    bs = rng.integers(0, B, n)
    hs = rng.integers(0, H, n)
    is_ = rng.integers(0, S, n)
    edges = np.unique(np.clip(np.concatenate([np.arange(0, S, 128), np.arange(127, S, 128),
                                              [S - 1]]), 0, S - 1))
    m = min(edges.size, n // 2)
    is_[:m] = edges[:m]
    return bs, is_, hs


# More units (128-query tiles of a batch and head) than SMs: every CTA walks several, and
# causal work goes in pairs of tiles (n-1-k, k) -- S = 1920 has an odd tile count, so one
# pair is a single middle tile.
WALK_CASES = [(2, 2048, 40, 64, True), (2, 2048, 40, 64, False), (2, 1920, 24, 128, True),
              (1, 4000, 20, 128, False)]


@pytest.mark.parametrize("B,S,H,D,causal", WALK_CASES)
def test_attention_many_units_per_cta_sampled(B, S, H, D, causal):
    dtype = torch.bfloat16
    q, k, v = _inputs(B, S, H, D, dtype, 7000 + S + H + int(causal))
    got = _run(q, k, v, causal).reshape(B, S, H, D)
    rng = np.random.default_rng(S + H)
    bs, is_, hs = _sampled_rows(B, S, H, rng, 600)
    ref = oracle.attention_rows(q, k, v, bs, is_, hs, dtype=oracle.BF16, causal=causal)
    assert_within_tolerance(got[bs, is_, hs], ref, oracle.BF16)


@pytest.mark.parametrize("name", ["attn_fwd_b4_h32_s4096_d128_causal_bf16",
                                  "attn_fwd_b4_h32_s4096_d128_bf16"])
def test_attention_workloads_sampled(name):
    w = workloads.ATTN_WORKLOADS[name]
    q, k, v = workloads.make_attn_inputs(w)
    got = _run(q, k, v, w.causal).reshape(w.B, w.S, w.H, w.D)
    rng = np.random.default_rng(13)
    bs, is_, hs = _sampled_rows(w.B, w.S, w.H, rng, 400)
    code = oracle.F16 if w.dtype == workloads.F16 else oracle.BF16
    ref = oracle.attention_rows(q, k, v, bs, is_, hs, dtype=code, causal=w.causal)
    assert_within_tolerance(got[bs, is_, hs], ref, code)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_closed_forms_exact(causal):
    # K = 0: every visible key gets probability exp2(0) = 1 before normalisation, so
    # P = 1 exactly and O = (sum of visible V rows) / count, with V small integers and
    # a power-of-two count per row when not causal
    B, S, H, D = 1, 256, 2, 64
    g = torch.Generator().manual_seed(5)
    q = torch.randn((B, S, H, D), generator=g).to(torch.bfloat16)
    k = torch.zeros((B, S, H, D), dtype=torch.bfloat16)
    v = torch.randint(-3, 4, (B, S, H, D), generator=g).to(torch.bfloat16)
    got = _run(q, k, v, causal)
    ref = oracle.attention(q, k, v, dtype=oracle.BF16, causal=causal)
    if causal:
        assert_bit_exact(got[:, 0], ref[:, 0])                    # row 0 is V[0]
        assert_within_tolerance(got.reshape(-1, D), ref.reshape(-1, D), oracle.BF16)
    else:
        assert_bit_exact(got, ref)


def test_attention_large_scores_and_tensor_call():
    # sharp softmax (scores up to ~50): the running max and rescale path
    B, S, H, D = 1, 640, 2, 128
    q, k, v = _inputs(B, S, H, D, torch.float16, 7, scale=2.5)
    out = tl.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
    ref = oracle.attention(q, k, v, dtype=oracle.F16, causal=True)
    assert_within_tolerance(_bits(out).reshape(-1, D), ref.reshape(-1, D), oracle.F16)


def test_attention_argument_errors():
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(4 * 128 * 64 + 8, dtype=torch.float16, device="cuda")
    o = torch.zeros_like(x)
    p, po = x.data_ptr(), o.data_ptr()
    assert tl.tl_attention_fwd(p, p, p, po, 1, 128, 1, 96, tl.TL_F16, 0, s) == tl.TL_ERR_UNSUPPORTED
    assert tl.tl_attention_fwd(p, p, p, po, 1, 128, 1, 64, 7, 0, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_attention_fwd(p, p, p, po, 1, 128, 1, 64, tl.TL_F16, 2, s) == tl.TL_ERR_INVALID_ARG
    assert tl.tl_attention_fwd(p + 2, p, p, po, 1, 128, 1, 64, tl.TL_F16, 0, s) == tl.TL_ERR_ALIGNMENT
    assert tl.tl_attention_fwd(p, p, p, p, 1, 128, 1, 64, tl.TL_F16, 0, s) == tl.TL_ERR_ALIAS
    assert tl.tl_attention_fwd(p, p, p, po, 0, 128, 1, 64, tl.TL_F16, 0, s) == tl.TL_OK
    assert tl.tl_device_status(reset=True)[0] == tl.TL_OK
