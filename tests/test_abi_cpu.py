"""Host-side checks of the C ABI that need no GPU.

* The shared library loads and exports every function that include/tl_gemm.h
  declares, and the Python binding passes every argument with the width and kind
  (pointer, 4- or 8-byte integer, float) that the header declares.
* The host planner reproduces the pages' printed resource numbers for the
  quickstart tiling (tests/golden/pages_resource_numbers.json): 16 KB per operand
  tile, 64/96/128 KB of operand ring for 2/3/4 stages, B ring at offset 48 KB,
  16 k-blocks at K = 1024, two such blocks per 228 KB SM.
* Argument errors are returned before anything touches a device.
"""
import ctypes
import json
import os
import re

import pytest

import tiled_gemm_gb300 as tl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tl_gemm.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "pages_resource_numbers.json")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for required in ("tl_gemm", "tl_gemm_plan", "tl_gemm_with_plan", "tl_plan_complete",
                     "tl_gemm_fp8", "tl_gemm_mx", "tl_attention_fwd", "tl_gemm_noalloc",
                     "tl_gemm_noalloc_scratch_bytes", "tl_status_string", "tl_device_status",
                     "tl_last_device_status",
                     "tl_set_wait_timeout_ns", "tl_version"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tl.LIBRARY._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings():
    for code, name in enumerate(tl.STATUS_NAMES):
        assert tl.tl_status_string(code) == name
    assert tl.tl_status_string(99) == "TL_ERR_UNKNOWN"
    assert tl.tl_version() >= 100


def test_planner_reproduces_the_pages_resource_numbers():
    g = json.load(open(GOLDEN))
    bm, bn, bk = g["tile"]
    for stages, ring in g["ring_bytes_by_stages"].items():
        p = tl.tl_plan_complete(1024, 1024, 1024, bm, bn, bk, int(stages))
        assert p.ring_bytes == ring
        assert p.ring_bytes // int(stages) == 2 * g["bytes_per_operand_tile"]
    p = tl.tl_plan_complete(1024, 1024, 1024, bm, bn, bk, 3)
    assert p.k_blocks == g["k_blocks_at_k_1024"]
    assert 3 * bm * bk * g["elem_bytes"] == g["b_ring_offset_bytes_3_stages"]
    assert p.tx_bytes == 2 * g["bytes_per_operand_tile"]
    assert g["smem_per_sm_bytes_h100"] // p.ring_bytes == g["blocks_per_sm_3_stages_h100"]
    # the quickstart grid: ceil(N/128) x ceil(M/128) = 64 tiles
    assert (p.tiles_m, p.tiles_n, p.tiles) == (8, 8, 64)


@pytest.mark.parametrize("M,N,K", [(3000, 5000, 4100), (256, 256, 256), (16, 8192, 8192),
                                   (8192, 8192, 8192), (1, 1, 1)])
def test_plan_tiles_cover_the_output_exactly_once(M, N, K):
    p = tl.tl_gemm_plan(M, N, K, num_sms=148)
    rows, cols = (N, M) if p.swap_ab else (M, N)    # swap_ab: tiles of C^T
    assert p.tiles_m * p.bm >= rows > (p.tiles_m - 1) * p.bm
    assert p.tiles_n * p.bn >= cols > (p.tiles_n - 1) * p.bn
    assert p.k_blocks * p.bk >= K > (p.k_blocks - 1) * p.bk
    assert p.tiles == p.tiles_m * p.tiles_n
    cg = p.bm // 128                       # CTAs per tile
    per_unit = cg * p.ksplit               # cluster split-K: two CTAs share a tile
    assert p.grid % per_unit == 0
    if p.sk_iters == 0:                    # whole tiles only: one unit per tile at most
        assert 1 <= p.grid <= per_unit * min(148 // per_unit, p.tiles)
        assert p.dp_tiles == p.tiles
    else:                                  # split: every unit takes a share
        assert p.grid == cg * (148 // cg)
        assert p.dp_tiles % (p.grid // cg) == 0
        assert p.sk_iters == (p.tiles - p.dp_tiles) * p.k_blocks
        assert p.workspace_bytes == p.grid * 128 * p.bn * 4 + p.grid * 4 * 8
    assert p.smem_bytes <= 232448
    assert p.tmem_cols == max(32, 2 * p.bn) and p.tmem_cols in (32, 64, 128, 256, 512)
    assert p.tx_bytes == (128 + p.bn // cg) * p.bk * 2


def test_every_supported_tiling_fits_shared_memory_and_others_are_rejected():
    for bm, bn, bk, max_stages in ((128, 64, 64, 8), (128, 128, 64, 6), (128, 256, 64, 4),
                                   (256, 128, 64, 8), (256, 256, 64, 6), (128, 64, 128, 4),
                                   (128, 128, 128, 3), (128, 256, 128, 2), (256, 128, 128, 4),
                                   (256, 256, 128, 3), (128, 16, 128, 6), (128, 32, 128, 5)):
        for stages in range(2, max_stages + 1):
            p = tl.tl_plan_complete(4096, 4096, 4096, bm, bn, bk, stages, trans_b=1)
            assert p.smem_bytes <= 232448
            assert p.grid % (bm // 128) == 0
            assert p.ring_bytes == stages * (128 * bk + (bn // (bm // 128)) * bk) * 2
        if max_stages < 8:
            with pytest.raises(tl.TLError):
                tl.tl_plan_complete(4096, 4096, 4096, bm, bn, bk, max_stages + 1, trans_b=1)
    for bad in ((64, 128, 64, 3), (128, 96, 64, 3), (128, 128, 32, 3), (128, 128, 64, 1),
                (128, 128, 64, 9), (256, 64, 64, 4), (512, 256, 64, 4), (128, 128, 256, 2),
                (128, 16, 64, 4), (128, 32, 64, 4), (256, 32, 128, 4), (128, 8, 128, 4)):
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(1024, 1024, 1024, *bad)


def test_stream_k_split_choices():
    # short tiles stay whole (the fix-up would cost more than it saves), whole waves are
    # never split, the ragged 3.2-wave shape is split, forcing works both ways
    p = tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152, ksplit=1)
    assert (p.dp_tiles, p.sk_iters, p.grid) == (64, 0, 64)
    p = tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152, stream_k=1)
    assert (p.dp_tiles, p.sk_iters, p.grid) == (0, 64 * 16, 152)
    p = tl.tl_plan_complete(128 * 152, 128, 1024, 128, 128, 64, 3, num_sms=152)
    assert p.sk_iters == 0 and p.tiles == 152
    p = tl.tl_gemm_plan(3000, 5000, 4100, num_sms=152)
    assert (p.bm, p.bn) == (256, 256) and p.dp_tiles == 2 * 76
    assert p.sk_iters == (240 - 152) * p.k_blocks
    p = tl.tl_plan_complete(4096, 4096, 4096, 256, 256, 128, 3, num_sms=152, stream_k=-1)
    assert p.sk_iters == 0 and p.dp_tiles == 256
    with pytest.raises(tl.TLError):
        tl.tl_plan_complete(64, 64, 64, 128, 64, 64, 3, stream_k=2)


def test_one_wave_of_narrow_tiles():
    # every 128 x 64 tile of C has an SM of its own and K is moderate: whole 128 x 64 x 128
    # tiles, one per CTA, in every layout
    for M, N, K, ta, tb in ((1024, 1024, 1024, 0, 0), (768, 768, 2048, 1, 0),
                            (512, 2048, 4096, 0, 1), (1024, 1024, 6144, 1, 1),
                            (8 * 128, 19 * 64, 1024, 0, 0)):
        p = tl.tl_gemm_plan(M, N, K, trans_a=ta, trans_b=tb, num_sms=152)
        assert (p.bm, p.bn, p.bk, p.stages, p.swap_ab) == (128, 64, 128, 4, 0)
        assert p.sk_iters == 0 and p.grid == p.tiles <= 152
    # one tile more than SMs, long or short K, 8-bit operands, skinny M: the other rules
    assert tl.tl_gemm_plan(8 * 128, 19 * 64 + 1, 1024, num_sms=152).bn != 64
    assert tl.tl_gemm_plan(1024, 1024, 1024, num_sms=100).bm == 256
    assert tl.tl_gemm_plan(1024, 1024, 16384, num_sms=152).bm == 256
    assert tl.tl_gemm_plan(1024, 1024, 512, num_sms=152).bk != 128
    assert tl.tl_gemm_plan(1024, 1024, 2048, dtype=tl.TL_E4M3, trans_b=1, num_sms=152).bk == 256
    assert tl.tl_gemm_plan(16, 2048, 1024, num_sms=152).swap_ab == 1


def test_skinny_products_swap_operands():
    # M <= 64 against long N and K: the kernel runs on C^T with M as the MMA's N, the 64
    # tiles of 128 rows of C^T each shared by the two CTAs of a cluster (cluster split-K)
    for M, bn, stages in ((1, 16, 6), (16, 16, 6), (17, 32, 5), (32, 32, 5), (33, 64, 4),
                          (64, 64, 4), (65, 128, 3), (128, 128, 3)):
        p = tl.tl_gemm_plan(M, 8192, 8192, dtype=tl.TL_BF16, trans_b=1, num_sms=152)
        assert p.swap_ab == 1 and (p.bm, p.bn, p.bk, p.stages) == (128, bn, 128, stages)
        assert (p.tiles_m, p.tiles_n, p.k_blocks) == (64, 1, 64)
        assert p.ksplit == 2 and p.grid == 128 and p.dp_tiles == 64 and p.sk_iters == 0
        assert p.tma_store == 0 and p.tx_bytes == (128 + bn) * 128 * 2   # C^T: plain stores
        assert p.smem_bytes <= 232448
    # wider M, an M-major A, short N or K, or an N too long for the split at M > 64: the
    # direct form
    assert tl.tl_gemm_plan(129, 8192, 8192, trans_b=1, num_sms=152).swap_ab == 0
    assert tl.tl_gemm_plan(128, 16384, 8192, trans_b=1, num_sms=152).swap_ab == 0
    assert tl.tl_gemm_plan(64, 16384, 8192, trans_b=1, num_sms=152).swap_ab == 1
    assert tl.tl_gemm_plan(16, 8192, 8192, trans_a=1).swap_ab == 0
    assert tl.tl_gemm_plan(16, 1024, 8192).swap_ab == 0
    assert tl.tl_gemm_plan(16, 8192, 512).swap_ab == 0
    # narrow tiles need the kernel's B operand K-major
    tl.tl_plan_complete(4096, 4096, 4096, 128, 16, 128, 4, trans_b=1)
    with pytest.raises(tl.TLError):
        tl.tl_plan_complete(4096, 4096, 4096, 128, 16, 128, 4, trans_b=0)
    tl.tl_plan_complete(16, 4096, 4096, 128, 16, 128, 4, trans_a=0, swap_ab=1)
    with pytest.raises(tl.TLError):
        tl.tl_plan_complete(16, 4096, 4096, 128, 16, 128, 4, trans_a=1, swap_ab=1)
    with pytest.raises(tl.TLError):
        tl.tl_plan_complete(16, 4096, 4096, 128, 64, 128, 4, swap_ab=2)


def test_planner_rejects_bad_arguments():
    with pytest.raises(tl.TLError):
        tl.tl_gemm_plan(-1, 4, 4)
    with pytest.raises(tl.TLError):
        tl.tl_gemm_plan(4, 4, 4, dtype=7)
    with pytest.raises(tl.TLError):
        tl.tl_gemm_plan(4, 4, 4, trans_a=2)


# Fake device addresses: every case below must be rejected before any CUDA call.
A, B, C = 0x10000, 0x20000000, 0x40000000


@pytest.mark.parametrize("args,code", [
    ((A, B, C, -1, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_INVALID_ARG),
    ((A, B, C, 4, 4, 4, 4, 4, 4, 2, 0, 0, 0), tl.TL_ERR_INVALID_ARG),      # dtype
    ((A, B, C, 4, 4, 4, 4, 4, 4, 0, 0, 0, 5), tl.TL_ERR_INVALID_ARG),      # epilogue
    ((A, B, C, 4, 4, 4, 4, 4, 4, 0, 3, 0, 0), tl.TL_ERR_INVALID_ARG),      # trans flag
    ((A, B, C, 4, 4, 8, 7, 4, 4, 0, 0, 0, 0), tl.TL_ERR_INVALID_ARG),      # lda < K
    ((A, B, C, 4, 5, 8, 8, 4, 5, 0, 0, 0, 0), tl.TL_ERR_INVALID_ARG),      # ldb < N
    ((A, B, C, 4, 5, 8, 8, 5, 4, 0, 0, 0, 0), tl.TL_ERR_INVALID_ARG),      # ldc < N
    ((A, B, C, 4, 4, 8, 3, 8, 4, 0, 1, 0, 0), tl.TL_ERR_INVALID_ARG),      # trans_a: lda < M
    ((A, B, 0, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_NULL_PTR),
    ((0, B, C, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_NULL_PTR),
    ((A, 0, C, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_NULL_PTR),
    ((A + 1, B, C, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_ALIGNMENT),
    ((A, B, C + 1, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_ALIGNMENT),
    ((A, B, A + 8, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_ALIAS),          # C inside A
    ((A, B, B - 8, 4, 4, 4, 4, 4, 4, 0, 0, 0, 0), tl.TL_ERR_ALIAS),          # C runs into B
])
def test_argument_errors_before_any_device_work(args, code):
    assert tl.tl_gemm(*args, None) == code


def test_empty_outputs_are_a_no_op():
    assert tl.tl_gemm(A, B, C, 0, 4, 4, 4, 4, 4, 0, 0, 0, 0, None) == tl.TL_OK
    assert tl.tl_gemm(A, B, C, 4, 0, 4, 4, 0, 0, 0, 0, 0, 0, None) == tl.TL_OK
    assert tl.tl_gemm(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == tl.TL_OK


def test_fp8_plans():
    # 8-bit operands: the same tiles with twice the K elements per stage (the same bytes)
    for M, N, K, tb in ((8192, 8192, 8192, 1), (4096, 4096, 4096, 0), (1000, 72, 2049, 1),
                        (16, 8192, 8192, 1), (3000, 5000, 4100, 0)):
        p = tl.tl_gemm_plan(M, N, K, dtype=tl.TL_E4M3, trans_b=tb, num_sms=152)
        cg = p.bm // 128
        assert p.bk in (128, 256) and p.swap_ab == 0 and p.bn >= 64
        assert p.ring_bytes == p.stages * (128 * p.bk + (p.bn // cg) * p.bk)
        assert p.tx_bytes == (128 + p.bn // cg) * p.bk
        assert p.smem_bytes <= 232448
        if not tb:
            assert (p.bn // cg) % 128 == 0
    big = tl.tl_gemm_plan(8192, 8192, 8192, dtype=tl.TL_E5M2, trans_b=1, num_sms=152)
    assert (big.bm, big.bn, big.bk, big.stages) == (256, 256, 256, 3)
    for bm, bn, bk, smax in ((128, 64, 128, 8), (128, 256, 256, 2), (256, 256, 256, 3),
                             (256, 128, 128, 8)):
        tl.tl_plan_complete(4096, 4096, 4096, bm, bn, bk, smax, dtype=tl.TL_E4M3, trans_b=1)
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(4096, 4096, 4096, bm, bn, bk, smax + 1, dtype=tl.TL_E4M3,
                                trans_b=1)
    for bad in ((128, 128, 64, 3), (128, 32, 128, 4), (128, 128, 512, 2)):
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(1024, 1024, 1024, *bad, dtype=tl.TL_E4M3, trans_b=1)
    # an N-major B needs 128-column boxes per CTA
    tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 128, 4, dtype=tl.TL_E4M3, trans_b=0)
    for bm, bn in ((128, 64), (256, 128)):
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(1024, 1024, 1024, bm, bn, 128, 4, dtype=tl.TL_E4M3, trans_b=0)


def _prototypes():
    """{name: (return type, [parameter types])} from the header's declarations."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w \t\*]*?)\s*\b(tl_[a-z0-9_]+)\s*\(([^)]*)\)\s*;",
                                        text):
        params = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        # drop the parameter name: the type is everything before the last identifier
        types = [re.sub(r"\s*\b\w+$", "", p) if re.search(r"[\w\*]\s+\w+$|\*\w+$", p) else p
                 for p in params]
        protos[name] = (ret.strip(), types)
    return protos


def _c_kind(t: str) -> str:
    t = t.replace("const", "").strip()
    if "*" in t or t == "tl_stream_t":
        return "ptr"
    if t in ("int64_t", "uint64_t"):
        return "8"
    if t in ("int", "int32_t", "uint32_t", "tl_dtype", "tl_epilogue", "tl_status"):
        return "4"
    if t in ("float", "double"):
        return "f4" if t == "float" else "f8"
    if t == "void":
        return "void"
    raise AssertionError(f"unexpected C type {t!r}")


def _ctypes_kind(t) -> str:
    if t is None:
        return "void"
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    if t in (ctypes.c_float, ctypes.c_double):
        return "f4" if t is ctypes.c_float else "f8"
    return str(ctypes.sizeof(t))


def test_binding_signatures_match_the_header():
    # every argument of every call crosses the ABI with the header's width: a 4-byte int
    # passed where the library reads an int64_t (or the reverse) would go unnoticed
    protos = _prototypes()
    assert set(protos) == set(declared_functions())
    for name, (ret, params) in protos.items():
        fn = getattr(tl.LIBRARY, name)
        want = [_c_kind(p) for p in params]
        got = [_ctypes_kind(a) for a in (fn.argtypes or [])]
        assert got == want, (name, got, want)
        assert _ctypes_kind(fn.restype) == _c_kind(ret), (name, fn.restype, ret)


def test_tensor_helpers_refuse_host_tensors_instead_of_falling_back():
    # every tensor-level call runs only through the CUDA library: host tensors are an
    # error before anything is enqueued, never a CPU computation
    import torch
    a = torch.zeros((8, 16), dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        tl.gemm(a, a.t().contiguous())
    f8 = torch.zeros((8, 32), dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="CUDA"):
        tl.gemm_fp8(f8, f8, trans_b=True)
    sf = torch.full((8, 16), 127, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        tl.gemm_mx(f8, f8, sf, sf)
    q = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        tl.attention(q, q, q)


def test_import_fails_loudly_without_the_built_library(tmp_path):
    # a copy of the package with no built library: importing it raises, naming the build
    # step; nothing else stands in for the CUDA library
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "tiled_gemm_gb300")
    shutil.copytree(src, tmp_path / "tiled_gemm_gb300",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import tiled_gemm_gb300"], cwd=tmp_path,
                       env=dict(os.environ, PYTHONPATH=str(tmp_path)), capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "not built" in r.stderr


def test_odd_width_tiles_need_a_k_major_b_and_fill_whole_waves():
    # 192- and 224-column tiles are loaded in boxes of whole K-major rows of B; an
    # N-major B (64-column boxes) cannot tile 96 or 112 columns per CTA
    for bm, bn in ((256, 224), (256, 192), (128, 224), (128, 192)):
        st = 3 if bm == 256 else 2            # one CTA holds all bn rows of B per stage
        p = tl.tl_plan_complete(4096, 4096, 4096, bm, bn, 128, st, dtype=tl.TL_BF16, trans_b=1,
                                num_sms=152)
        assert p.tmem_cols == 512 and p.tiles_n == -(-4096 // bn)
        assert p.tx_bytes == (128 + bn // (bm // 128)) * 128 * 2
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(4096, 4096, 4096, bm, bn, 128, st, dtype=tl.TL_BF16, trans_b=0)
        with pytest.raises(tl.TLError):       # 128-deep stages only
            tl.tl_plan_complete(4096, 4096, 4096, bm, bn, 64, st, dtype=tl.TL_BF16, trans_b=1)
    with pytest.raises(tl.TLError):           # 3 stages of 128 x 224 + 224 x 128 exceed smem
        tl.tl_plan_complete(4096, 4096, 4096, 128, 224, 128, 3, dtype=tl.TL_BF16, trans_b=1)
    # 4096^3 with a K-major B: 16 x 19 = 304 pair tiles of 256 x 224 are exactly four waves
    # of 76 SM pairs, where 256 x 256 tiles leave a last wave 37 % full
    p = tl.tl_gemm_plan(4096, 4096, 4096, dtype=tl.TL_BF16, trans_b=1, num_sms=152)
    assert (p.bm, p.bn, p.bk) == (256, 224, 128) and p.tiles == 304 and p.grid == 152
    assert p.sk_iters == 0
    assert p.raster_group == 16                 # one group spans all 16 tile rows
    # 8192^3 keeps the 256-column tiles (13.5 waves either way); an N-major B never takes
    # the odd widths
    p = tl.tl_gemm_plan(8192, 8192, 8192, dtype=tl.TL_BF16, trans_b=1, num_sms=152)
    assert (p.bm, p.bn) == (256, 256) and p.raster_group == 12
    p = tl.tl_gemm_plan(4096, 4096, 4096, dtype=tl.TL_BF16, trans_b=0, num_sms=152)
    assert p.bn not in (192, 224)


def test_cluster_split_k_plans():
    # the quickstart tiling (64 tiles of 128 x 128, 16 k-blocks): two CTAs per tile
    p = tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152)
    assert p.ksplit == 2 and p.grid == 128 and p.sk_iters == 0
    # its receive buffer (the peer's partial sums of 128 rows x 64 columns, fp32) is part
    # of each CTA's shared memory
    off = tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152, ksplit=1)
    assert off.ksplit == 1 and off.grid == 64
    assert p.smem_bytes == off.smem_bytes + 64 * 128 * 4
    # more tiles than half the SMs, or a short k-loop: no split
    assert tl.tl_plan_complete(2048, 2048, 1024, 128, 128, 64, 3, num_sms=152).ksplit == 1
    assert tl.tl_plan_complete(1024, 1024, 192, 128, 128, 64, 3, num_sms=152).ksplit == 1
    # pairs never split; a forced split that cannot apply is an error
    assert tl.tl_plan_complete(1024, 1024, 1024, 256, 256, 128, 3, num_sms=152).ksplit == 1
    for kw in ({"bm": 256, "bn": 256, "bk": 128, "stages": 3},
               {"bm": 128, "bn": 256, "bk": 64, "stages": 4}):        # smem does not fit
        with pytest.raises(tl.TLError):
            tl.tl_plan_complete(1024, 1024, 1024, num_sms=152, ksplit=2, **kw)
    with pytest.raises(tl.TLError):                                     # one k-block
        tl.tl_plan_complete(1024, 1024, 64, 128, 128, 64, 3, num_sms=152, ksplit=2)
    # each CTA finishes half the tile's columns: power-of-two widths only
    with pytest.raises(tl.TLError):
        tl.tl_plan_complete(1024, 1024, 1024, 128, 224, 128, 2, trans_b=1, num_sms=152,
                            ksplit=2)
    assert tl.tl_plan_complete(1024, 1024, 1024, 128, 224, 128, 2, trans_b=1,
                               num_sms=152).ksplit == 1
    with pytest.raises(tl.TLError):                                     # with stream-K
        tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152, ksplit=2,
                            stream_k=1)
    # a forced grid counts CTAs: 6 CTAs are 3 clusters
    g = tl.tl_plan_complete(1024, 1024, 1024, 128, 128, 64, 3, num_sms=152, ksplit=2, grid=6)
    assert g.grid == 6
