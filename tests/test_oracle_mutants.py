"""The oracle's pins catch plausible mistakes: each one is planted in a copy of the oracle.

A pin is only worth something if a wrong oracle fails it.  For every mistake listed in
MUTANTS below, this test writes a copy of ``oracle/tl_oracle.c`` with that one mistake
(a dropped or extra term, a wrong sign, bias, index, layout, rounding rule, scale or
mask), lets the oracle package build the copy into a temporary library, and runs the
whole of ``tests/test_oracle_pins.py`` against it in a child process: the pins must
fail (pytest exit status 1; a crash or a collection error does not count).  The same
harness run on an unmodified copy must pass, so the failures come from the planted
mistake and nothing else.

Everything here runs on the CPU; the committed oracle is never modified.  Every planted
mistake keeps each memory access of the pins' shapes inside its array.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_SRC = os.path.join(ROOT, "oracle", "tl_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in the oracle, its wrong replacement)
MUTANTS = [
    # the GEMM: C = epi(sum_k op(A)[i,k] op(B)[k,j]), binary64, k in order
    ("drops the last k term", "for (int64_t k = 0; k < K; ++k) {\n    s += op_a(",
     "for (int64_t k = 0; k < K - 1; ++k) {\n    s += op_a("),
    ("skips the first k term", "for (int64_t k = 0; k < K; ++k) {\n    s += op_a(",
     "for (int64_t k = 1; k < K; ++k) {\n    s += op_a("),
    ("subtracts the products", "    s += op_a(A, lda, trans_a, i, k, dtype) * op_b(",
     "    s -= op_a(A, lda, trans_a, i, k, dtype) * op_b("),
    ("ignores transpose_A", "return decode(trans_a ? A[k * lda + i] : A[i * lda + k], dtype);",
     "return decode(A[i * lda + k], dtype);"),
    ("writes C with pitch N instead of ldc", "if (C) C[i * ldc + j] = encode(s, dtype);",
     "if (C) C[i * N + j] = encode(s, dtype);"),
    ("leaves out the ReLU",
     "static double epilogue(double s, int relu) { return (relu && !(s > 0.0)) ? 0.0 : s; }",
     "static double epilogue(double s, int relu) { (void)relu; return s; }"),
    ("zeroes the positives instead of the negatives",
     "static double epilogue(double s, int relu) { return (relu && !(s > 0.0)) ? 0.0 : s; }",
     "static double epilogue(double s, int relu) { return (relu && (s > 0.0)) ? 0.0 : s; }"),
    ("sampled entries skip the epilogue",
     "epilogue(dot(A, B, K, lda, ldb, dtype, trans_a, trans_b, rows[t], cols[t]), relu);",
     "dot(A, B, K, lda, ldb, dtype, trans_a, trans_b, rows[t], cols[t]);"),
    # the 16-bit decoders
    ("binary16 subnormal exponent off by one", "v = ldexp((double)f, -24);",
     "v = ldexp((double)f, -25);"),
    ("binary16 normal numbers lose the hidden bit", "v = ldexp((double)(f + 1024), e - 25);",
     "v = ldexp((double)f, e - 25);"),
    ("bfloat16 exponent bias off by one", "v = ldexp((double)(f + 128), e - 134);",
     "v = ldexp((double)(f + 128), e - 133);"),
    # the round-to-nearest-even encoders
    ("ties round away from zero",
     "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
     "if (frac >= 0.5) r += 1.0;"),
    ("truncates instead of rounding",
     "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
     "if (frac > 1.0) r += 1.0;"),
    ("subnormals take a finer quantum", "if (E < emin) E = emin;", "(void)emin;"),
    ("no overflow to infinity", "if (bits >= inf_bits) bits = inf_bits;", "(void)inf_bits;"),
    ("drops the sign", "const uint16_t sign = signbit(v) ? 0x8000 : 0;",
     "const uint16_t sign = 0;"),
    ("binary16 minimum exponent off by one", "rne_encode(v, 10, -14, 0x7C00, 0x7E00)",
     "rne_encode(v, 10, -15, 0x7C00, 0x7E00)"),
    ("bfloat16 rounded to 8 fraction bits", "rne_encode(v, 7, -126, 0x7F80, 0x7FC0)",
     "rne_encode(v, 8, -126, 0x7F80, 0x7FC0)"),
    # the 8-bit decoders and the FP8 product
    ("E4M3 read with IEEE-style specials", "if (e == 15 && f == 7) {", "if (e == 15) {"),
    ("E4M3 exponent bias off by one", "v = ldexp((double)(f + 8), e - 10);",
     "v = ldexp((double)(f + 8), e - 11);"),
    ("E5M2 subnormal exponent off by one", "v = ldexp((double)f, -16);",
     "v = ldexp((double)f, -17);"),
    ("FP8 product without its scale alpha",
     "alpha * dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b, i, j), relu);",
     "dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b, i, j), relu);"),
    ("FP8 sampled entries without alpha",
     "epilogue(alpha * dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b,\n",
     "epilogue(dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b,\n"),
    ("FP8 A decoded in B's format",
     "const double a = decode8(trans_a ? A[k * lda + i] : A[i * lda + k], a_type);",
     "const double a = decode8(trans_a ? A[k * lda + i] : A[i * lda + k], b_type);"),
    # the block-scaled (MX) product
    ("E8M0 bias off by one", "ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 128)"),
    ("E8M0 255 read as a finite scale", "return e == 255 ? NAN : ldexp(1.0, (int)e - 127);",
     "return ldexp(1.0, (int)e - 127);"),
    ("scale blocks of 64 instead of 32", "SA[i * sfa_ld + k / 32]", "SA[i * sfa_ld + k / 64]"),
    ("B's scales taken from A's row index", "SB[j * sfb_ld + k / 32]", "SB[i * sfb_ld + k / 32]"),
    # attention: O = softmax(Q K^T / sqrt(D)) V over [B, S, H, D]
    ("scores not scaled by 1/sqrt(D)", "const double scale = 1.0 / sqrt((double)D);",
     "const double scale = 1.0;"),
    ("the causal mask hides the diagonal", "const int64_t n = causal ? i + 1 : S;",
     "const int64_t n = causal ? i : S;"),
    ("V read without the head offset", "const uint16_t* v = V + (b * S + j) * row + h * D;",
     "const uint16_t* v = V + (b * S + j) * row;"),
    ("Q read as [B, H, S, D]", "const uint16_t* q = Q + (b * S + i) * row + h * D;",
     "const uint16_t* q = Q + ((b * H + h) * S + i) * D;"),
    ("O written as [B, H, S, D]", "const int64_t base = ((b * S + i) * H + h) * D;",
     "const int64_t base = ((b * H + h) * S + i) * D;"),
    ("normalised by the key count, not the softmax sum",
     "for (int64_t d = 0; d < D; ++d) out[d] /= den;",
     "for (int64_t d = 0; d < D; ++d) out[d] /= (double)n;"),
    ("sampled rows ignore the causal mask",
     "attention_row(Q, K, V, S, H, D, dtype, causal, bs[t], hs[t], is[t], scores, row);",
     "attention_row(Q, K, V, S, H, D, dtype, 0, bs[t], hs[t], is[t], scores, row);"),
]

# Runs in the child: point the oracle package at the copy, then run the pins.
_CHILD = """
import sys
root, src, build_dir, lib = sys.argv[1:5]
sys.path.insert(0, root)
import oracle
oracle._SRC, oracle._BUILD_DIR, oracle._LIB_PATH = src, build_dir, lib
import pytest
sys.exit(pytest.main([sys.argv[5], "-x", "-q", "-p", "no:cacheprovider",
                      "-W", "ignore::RuntimeWarning"]))
"""


def _run_pins_on(source_text, work_dir):
    os.makedirs(work_dir, exist_ok=True)
    src = os.path.join(work_dir, "tl_oracle.c")
    with open(src, "w") as f:
        f.write(source_text)
    env = dict(os.environ, OMP_NUM_THREADS="2", CUDA_VISIBLE_DEVICES="")
    proc = subprocess.run(
        [sys.executable, "-c", _CHILD, ROOT, src, work_dir,
         os.path.join(work_dir, "liboracle.so"), PINS],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return proc.returncode, proc.stdout + proc.stderr


def _first_failure(output):
    for line in output.splitlines():
        if line.startswith("FAILED "):
            return line.split(" ")[1]
    return "?"


def test_every_mutant_site_is_in_the_oracle_once():
    text = open(ORACLE_SRC).read()
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))
    for name, old, new in MUTANTS:
        assert old != new, name
        assert text.count(old) == 1, f"{name}: the text to replace is not in the oracle once"


def test_the_harness_passes_on_the_unmodified_oracle(tmp_path):
    rc, out = _run_pins_on(open(ORACLE_SRC).read(), str(tmp_path / "unmodified"))
    assert rc == 0, out[-3000:]
    assert " passed" in out and "failed" not in out


def test_the_pins_fail_for_every_planted_mistake(tmp_path):
    text = open(ORACLE_SRC).read()

    def one(idx_mutant):
        idx, (name, old, new) = idx_mutant
        return name, _run_pins_on(text.replace(old, new, 1), str(tmp_path / f"m{idx:02d}"))

    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(max_workers=workers) as pool:
        results = list(pool.map(one, enumerate(MUTANTS)))
    survivors = [(name, rc, out[-1500:]) for name, (rc, out) in results if rc != 1]
    assert not survivors, "\n\n".join(f"{n}: exit status {rc}\n{o}" for n, rc, o in survivors)
    for name, (rc, out) in results:
        assert "failed" in out and _first_failure(out) != "?", name
