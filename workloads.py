"""Seeded synthetic workloads for the tiled GEMM: shapes, layouts and input draws.

This module only draws inputs; it holds none of the GEMM's arithmetic.  Both the
CPU oracle's tests and the CUDA path's tests and benchmark take their inputs from
here, so the two sides see bit-identical operands.

Recipe (stated once, used everywhere): one CPU ``torch.Generator`` per workload,
seeded with the workload's seed; A is drawn first, then B, each in fp32 in the
shape of its *storage* (A is [M, K], or [K, M] when ``trans_a``; B is [K, N], or
[N, K] when ``trans_b``), then converted to the 16-bit dtype by torch's
round-to-nearest-even cast (8-bit E4M3 / E5M2 operands: torch's float8 cast of the
same fp32 draw).  Distributions follow the workloads the GEMM is
described with (the pages' quickstart GEMM at 1024^3 with fp16 operands and
128x128x64 tiles in 3 stages; square bf16 GEMMs with a column-major B; a ragged
shape that is a multiple of no tile; decode-like skinny products).
"""
from __future__ import annotations

import dataclasses
import math

import torch

F16 = 0
BF16 = 1
E4M3 = 2
E5M2 = 3
_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn,
                E5M2: torch.float8_e5m2}
_NAME = {F16: "f16", BF16: "bf16", E4M3: "e4m3", E5M2: "e5m2"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: int
    trans_a: bool
    trans_b: bool
    relu: bool
    dist_a: str            # "uniform" | "normal_over_sqrtk" | "normal"
    dist_b: str
    std_a: float = 1.0     # used by "normal"
    std_b: float = 1.0
    seed: int = 0
    plan: tuple | None = None   # (BM, BN, BK, stages) when the workload fixes the tiling
    description: str = ""
    # 8-bit operands only: B's own format (default: dtype), the output type, the scale
    b_dtype: int | None = None
    out_dtype: int = BF16
    alpha: float = 1.0

    @property
    def fp8(self) -> bool:
        return self.dtype in (E4M3, E5M2)

    @property
    def torch_dtype(self) -> torch.dtype:
        """Output (and, for 16-bit workloads, operand) dtype."""
        return _TORCH_DTYPE[self.out_dtype if self.fp8 else self.dtype]

    @property
    def c_dtype(self) -> int:
        return self.out_dtype if self.fp8 else self.dtype

    @property
    def a_torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]

    @property
    def b_torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.b_dtype if self.b_dtype is not None else self.dtype]

    @property
    def b_fmt(self) -> int:
        return self.b_dtype if self.b_dtype is not None else self.dtype

    @property
    def dtype_name(self) -> str:
        return _NAME[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 1 if self.fp8 else 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_moved(self) -> int:
        """Algorithmic HBM bytes: read A and B once, write C (2-byte elements) once."""
        return self.elem_bytes * (self.M * self.K + self.K * self.N) + 2 * self.M * self.N

    def a_shape(self) -> tuple[int, int]:
        return (self.K, self.M) if self.trans_a else (self.M, self.K)

    def b_shape(self) -> tuple[int, int]:
        return (self.N, self.K) if self.trans_b else (self.K, self.N)


def _draw(shape, dist: str, std: float, K: int, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal_over_sqrtk":
        return torch.randn(shape, generator=g, dtype=torch.float32) / math.sqrt(K)
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32) * std
    if dist == "int_small":
        # integers in [-2, 2]: every partial sum is an exact small integer in fp32
        return torch.randint(-2, 3, shape, generator=g).to(torch.float32)
    if dist == "int_unit":
        # integers in [-1, 1]: exact in bf16 and in every fp32 partial sum
        return torch.randint(-1, 2, shape, generator=g).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(w: Workload, seed: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """CPU tensors (A, B) in storage layout and the workload's dtype; A drawn first."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    a = _draw(w.a_shape(), w.dist_a, w.std_a, w.K, g).to(w.a_torch_dtype)
    b = _draw(w.b_shape(), w.dist_b, w.std_b, w.K, g).to(w.b_torch_dtype)
    return a, b


def integer_variant(w: Workload, M=None, N=None, K=None, seed=None) -> Workload:
    """Same layout and dtype with small-integer entries, so that every fp32 partial sum
    is exact and GPU and oracle must agree bit for bit."""
    dist = "int_small" if w.dtype in (F16, E4M3, E5M2) else "int_unit"
    return dataclasses.replace(
        w, name=w.name + "_int", M=M or w.M, N=N or w.N, K=K or w.K,
        dist_a=dist, dist_b=dist, seed=w.seed if seed is None else seed)


WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("gemm_relu_256_f16", 256, 256, 256, F16, False, False, True,
              "uniform", "uniform", seed=0,
              description="GEMM+ReLU 256^3 fp16, A,B row-major U[-1,1]"))
_add(Workload("gemm_relu_1024_f16_128x128x64s3", 1024, 1024, 1024, F16, False, False, True,
              "uniform", "uniform", seed=1, plan=(128, 128, 64, 3),
              description="GEMM+ReLU 1024^3 fp16 (quickstart size), tiles 128x128x64, "
                          "3 stages, U[-1,1]"))
_add(Workload("gemm_4096_bf16_tb", 4096, 4096, 4096, BF16, False, True, False,
              "normal_over_sqrtk", "normal_over_sqrtk", seed=2,
              description="GEMM 4096^3 bf16, B column-major, N(0,1)/sqrt(K)"))
_add(Workload("gemm_8192_bf16_tb", 8192, 8192, 8192, BF16, False, True, False,
              "normal_over_sqrtk", "normal_over_sqrtk", seed=3,
              description="GEMM 8192^3 bf16, B column-major, N(0,1)/sqrt(K)"))
_add(Workload("gemm_relu_3000x5000x4100_f16", 3000, 5000, 4100, F16, False, False, True,
              "uniform", "uniform", seed=4,
              description="ragged GEMM+ReLU 3000x5000x4100 fp16, U[-1,1]"))
for _m, _seed in ((16, 5), (64, 6), (128, 7)):
    _add(Workload(f"gemm_m{_m}_n8192_k8192_bf16", _m, 8192, 8192, BF16, False, True, False,
                  "normal", "normal", std_a=1.0, std_b=0.02, seed=_seed,
                  description=f"skinny decode-like GEMM M={_m}, N=K=8192 bf16, activations "
                              "N(0,1), weights N(0,0.02) stored [N,K]"))

# 8-bit operands (one product scale): square products with weights stored [N, K]
for _n, _seed in ((4096, 8), (8192, 9)):
    _add(Workload(f"gemm_{_n}_e4m3_tb", _n, _n, _n, E4M3, False, True, False,
                  "normal", "normal", seed=_seed, out_dtype=BF16, alpha=1.0 / 64,
                  description=f"FP8 GEMM {_n}^3, E4M3 operands from N(0,1), B column-major, "
                              "alpha 1/64, bf16 output"))

# ---- block-scaled (MX) 8-bit products: A [M,K], B [N,K], one E8M0 scale per 32 K ----

@dataclasses.dataclass(frozen=True)
class MxWorkload:
    name: str
    M: int
    N: int
    K: int
    a_fmt: int = E4M3
    b_fmt: int = E4M3
    out_dtype: int = BF16
    relu: bool = False
    dist: str = "mx"        # "mx": N(0, std) values quantised block by block (below);
                            # otherwise codes converted from draws of _draw and scale
                            # codes drawn uniformly in [sf_lo, sf_hi]
    std: float = 1.0
    sf_lo: int = 120
    sf_hi: int = 134
    sf_pad: int = 0         # extra scale bytes per row (a multiple of 16)
    seed: int = 0
    description: str = ""

    @property
    def sf_ld(self) -> int:
        """Scale pitch in bytes: 4*ceil(K/128) rounded up to 16, plus sf_pad."""
        return 16 * ((4 * ((self.K + 127) // 128) + 15) // 16) + self.sf_pad

    @property
    def fp8(self) -> bool:
        return True

    @property
    def dtype_name(self) -> str:
        return f"{_NAME[self.a_fmt]}x{_NAME[self.b_fmt]}-mx"

    @property
    def c_torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.out_dtype]

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_moved(self) -> int:
        return (self.M + self.N) * (self.K + self.sf_ld) + 2 * self.M * self.N


# largest normal exponent and value of each 8-bit element format
_FP8_EMAX = {E4M3: (8, 448.0), E5M2: (15, 57344.0)}


def _mx_quantise(x: torch.Tensor, fmt: int, sf_ld: int):
    """The usual MX encoding of fp32 rows x [rows, K]: per block of 32, the shared
    exponent is floor(log2(max |x|)) minus the element format's largest exponent (as an
    E8M0 code, clamped to [0, 254]), and the elements are x / 2^exponent converted to
    the 8-bit format, clamped to its largest normal value.  Scale bytes past K/32 are
    the code of 2^0."""
    rows, K = x.shape
    blk = x.reshape(rows, K // 32, 32)
    amax = blk.abs().amax(dim=-1).clamp_min(2.0 ** -120)
    emax, vmax = _FP8_EMAX[fmt]
    e = (torch.floor(torch.log2(amax)) - emax).clamp(-127, 127)
    q = (blk / torch.exp2(e).unsqueeze(-1)).clamp(-vmax, vmax)
    codes = q.reshape(rows, K).to(_TORCH_DTYPE[fmt])
    sf = torch.full((rows, sf_ld), 127, dtype=torch.uint8)
    sf[:, :K // 32] = (e + 127).to(torch.uint8)
    return codes, sf


def make_mx_inputs(w: MxWorkload, seed: int | None = None):
    """CPU tensors (A, B, SA, SB): 8-bit A [M,K] and B [N,K] and uint8 scale codes
    SA [M, sf_ld] and SB [N, sf_ld].  dist "mx": A's then B's N(0, std) values, each
    quantised by _mx_quantise; otherwise A's and B's codes from _draw, then SA and SB
    uniform in [sf_lo, sf_hi]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    if w.dist == "mx":
        xa = torch.randn((w.M, w.K), generator=g, dtype=torch.float32) * w.std
        xb = torch.randn((w.N, w.K), generator=g, dtype=torch.float32) * w.std
        a, sa = _mx_quantise(xa, w.a_fmt, w.sf_ld)
        b, sb = _mx_quantise(xb, w.b_fmt, w.sf_ld)
        return a, b, sa, sb
    a = _draw((w.M, w.K), w.dist, w.std, w.K, g).to(_TORCH_DTYPE[w.a_fmt])
    b = _draw((w.N, w.K), w.dist, w.std, w.K, g).to(_TORCH_DTYPE[w.b_fmt])
    sa = torch.randint(w.sf_lo, w.sf_hi + 1, (w.M, w.sf_ld), generator=g).to(torch.uint8)
    sb = torch.randint(w.sf_lo, w.sf_hi + 1, (w.N, w.sf_ld), generator=g).to(torch.uint8)
    return a, b, sa, sb


MX_WORKLOADS: dict[str, MxWorkload] = {}
for _n, _seed in ((4096, 30), (8192, 31)):
    _w = MxWorkload(f"gemm_mx_{_n}_e4m3", _n, _n, _n, seed=_seed,
                    description=f"block-scaled 8-bit GEMM {_n}^3: N(0,1) operands in the MX "
                                "encoding (E4M3 elements, one E8M0 scale per 32 K), bf16 "
                                "output")
    MX_WORKLOADS[_w.name] = _w

# ---- attention forward: O = softmax(Q K^T / sqrt(D)) V over [B, S, H, D] ------------

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    name: str
    B: int
    S: int
    H: int
    D: int
    dtype: int
    causal: bool
    seed: int = 0
    description: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]

    @property
    def dtype_name(self) -> str:
        return _NAME[self.dtype]

    @property
    def flops(self) -> int:
        """Two products of 2*S*S*D per (batch, head); half of that when causal."""
        full = 4 * self.B * self.H * self.S * self.S * self.D
        return full // 2 if self.causal else full

    @property
    def bytes_moved(self) -> int:
        return 4 * 2 * self.B * self.S * self.H * self.D          # Q, K, V read, O written


def make_attn_inputs(w: AttnWorkload, seed: int | None = None):
    """CPU tensors (Q, K, V), each [B, S, H, D] drawn N(0,1) in fp32 in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.S, w.H, w.D)
    return tuple(torch.randn(shape, generator=g, dtype=torch.float32).to(w.torch_dtype)
                 for _ in range(3))


ATTN_WORKLOADS: dict[str, AttnWorkload] = {}
for _w in (AttnWorkload("attn_fwd_b1_h8_s1024_d64_causal_f16", 1, 1024, 8, 64, F16, True, 20,
                        "the pages' FlashAttention example size: batch 1, 8 heads, seq 1024, "
                        "dim 64, causal, fp16, N(0,1)"),
           AttnWorkload("attn_fwd_b4_h32_s4096_d128_bf16", 4, 4096, 32, 128, BF16, False, 21,
                        "attention 4x32 heads, seq 4096, dim 128, bf16, N(0,1)"),
           AttnWorkload("attn_fwd_b4_h32_s4096_d128_causal_bf16", 4, 4096, 32, 128, BF16, True,
                        22, "causal attention 4x32 heads, seq 4096, dim 128, bf16, N(0,1)")):
    ATTN_WORKLOADS[_w.name] = _w

# The benchmark's headline workload: the largest square product, 8192^3 bf16 with a
# column-major B, where the tensor-peak fraction is stated.
HEADLINE = "gemm_8192_bf16_tb"
