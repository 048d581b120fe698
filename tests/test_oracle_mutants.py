"""The oracle's pins, checked against planted mistakes (no GPU).

Each mutant below is a copy of ``oracle/gemm_oracle.c`` with one plausible
error planted by an exact text substitution: a dropped term of the sum, a
wrong sign, a transposed or reversed operand, a leading dimension ignored,
FP32 rounding of the fp64 sums, an off-by-one exponent bias in a widening,
a format's special values read the IEEE way, and the epilogue's alpha, beta,
bias, ReLU and GELU each written wrong.  Every mutant is compiled as the
oracle is, bound in place of the real library, and run through every pin of
``tests/test_oracle.py`` (each parametrization).  The test asserts that the
unchanged copy passes every pin and that each mutant fails at least one.

Every planted access stays inside the operands' buffers, and the pins run
in a child process, so even a mutant that misbehaves cannot take down the
test run.  A substitution that no longer matches the source exactly once
fails the test, so the table follows the oracle when it changes.
"""
import itertools
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gemm_oracle.c")

# name -> (text in the oracle, text planted in its place)
MUTANTS = {
    # -- the FP32 sum C = A.B
    "f32_drops_last_k": (
        "    for (int64_t k = 0; k < K; ++k) {\n        const double a = (double)A[i * lda + k];",
        "    for (int64_t k = 0; k < K - 1; ++k) {\n        const double a = (double)A[i * lda + k];"),
    "f32_subtracts_products": ("c[j] += a * (double)b[j];", "c[j] -= a * (double)b[j];"),
    "f32_reverses_b_columns": ("c[j] += a * (double)b[j];", "c[j] += a * (double)b[N - 1 - j];"),
    "f32_reads_b_transposed": (
        "c[j] += a * (double)b[j];",
        "c[j] += a * ((j < K && k < N) ? (double)B[j * ldb + k] : 0.0);"),
    "f32_sums_in_float": ("c[j] += a * (double)b[j];", "c[j] = (float)(c[j] + a * (double)b[j]);"),
    "f32_ignores_ldb": ("const float *b = B + k * ldb;", "const float *b = B + k * N;"),
    "f32_scale_keeps_signs": (
        "const double aa = fabs(a);\n            for (int64_t j = 0; j < N; ++j) d[j] += aa * fabs((double)b[j]);",
        "const double aa = a;\n            for (int64_t j = 0; j < N; ++j) d[j] += aa * (double)b[j];"),
    "f32_rows_ignores_row_list": ("row_f32(rows[r], N, K", "row_f32(r, N, K"),
    # -- BF16 / FP16 widening and sums
    "bf16_shift_15": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "f16_bias_off_by_one": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "f16_subnormal_with_implicit_one": ("ldexp((double)m, -24);", "ldexp((double)(1024 + m), -25);"),
    "f16_b_widened_as_bf16": (
        "for (int64_t j = 0; j < N; ++j) bw[j] = widen_f16(b[j]);",
        "for (int64_t j = 0; j < N; ++j) bw[j] = widen_bf16(b[j]);"),
    "h16_sums_in_float": (
        "            for (int64_t j = 0; j < N; ++j) bw[j] = widen_bf16(b[j]);\n"
        "        for (int64_t j = 0; j < N; ++j) c[j] += a * bw[j];",
        "            for (int64_t j = 0; j < N; ++j) bw[j] = widen_bf16(b[j]);\n"
        "        for (int64_t j = 0; j < N; ++j) c[j] = (float)(c[j] + a * bw[j]);"),
    "h16_rows_ignores_row_list": ("row_h16(fmt, rows[r], N, K", "row_h16(fmt, r, N, K"),
    # -- FP8
    "e4m3_ieee_specials": ("if (e == 15 && m == 7)\n        v = NAN;", "if (e == 15)\n        v = m ? NAN : INFINITY;"),
    "e4m3_subnormal_exponent": ("ldexp((double)m, -9);", "ldexp((double)m, -10);"),
    "e5m2_bias_off_by_one": ("ldexp((double)(4 + m), e - 17)", "ldexp((double)(4 + m), e - 16)"),
    "fp8_table_of_other_format": (
        "fmt == FMT8_E5M2 ? widen_e5m2((uint8_t)b) : widen_e4m3((uint8_t)b)",
        "fmt == FMT8_E5M2 ? widen_e4m3((uint8_t)b) : widen_e5m2((uint8_t)b)"),
    "fp8_skips_first_k": (
        "    for (int64_t k = 0; k < K; ++k) {\n        const double a = tab[A[i * lda + k]];",
        "    for (int64_t k = 1; k < K; ++k) {\n        const double a = tab[A[i * lda + k]];"),
    # -- the second loop order (the brute-force check itself)
    "jik_drops_last_k": (
        "for (int64_t k = 0; k < K; ++k)\n                s += (double)A[i * lda + k] * (double)B[k * ldb + j];",
        "for (int64_t k = 0; k < K - 1; ++k)\n                s += (double)A[i * lda + k] * (double)B[k * ldb + j];"),
    # -- the fused epilogue
    "epi_ignores_alpha": ("double x = alpha * acc[i * ld_acc + j];", "double x = acc[i * ld_acc + j];"),
    "epi_beta_sign": ("x += beta * read_old(", "x -= beta * read_old("),
    "epi_bias_by_row": ("x += (double)bias[j];", "x += (double)bias[i % N];"),
    "epi_relu_absolute": ("x = x > 0.0 ? x : 0.0;", "x = x > 0.0 ? x : -x;"),
    "epi_gelu_erf_of_half_x": ("erf(x / sqrt(2.0))", "erf(x / 2.0)"),
    "epi_gelu_drops_half": ("x = x * 0.5 * (1.0 + erf(", "x = x * (1.0 + erf("),
    "epi_old_bf16_read_as_f16": ("if (out == OUT_BF16) return widen_bf16(", "if (out == OUT_BF16) return widen_f16("),
}


def _pins():
    """(name, callable) for every pin of test_oracle, each parametrization expanded."""
    import test_oracle
    out = []
    for name in sorted(n for n in dir(test_oracle) if n.startswith("test_")):
        fn = getattr(test_oracle, name)
        axes = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names, values = mark.args[0], mark.args[1]
            names = [s.strip() for s in names.split(",")] if isinstance(names, str) else list(names)
            axes.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
        for combo in itertools.product(*axes):
            kw = {k: v for part in combo for k, v in part.items()}
            label = name + ("[" + ",".join(f"{k}={kw[k]}" for k in sorted(kw)) + "]" if kw else "")
            out.append((label, lambda fn=fn, kw=kw: fn(**kw)))
    return out


def _failing_pins(lib_path):
    """Run every pin against the library at lib_path; the labels of those that fail."""
    import oracle
    oracle._lib = oracle.bind(lib_path)
    failed = []
    for label, run in _pins():
        try:
            run()
        except Exception as e:            # an assertion, or any error the wrong values raise
            failed.append(f"{label}: {type(e).__name__}")
    return failed


def _plant(src_text, find, repl):
    assert src_text.count(find) == 1, f"substitution target no longer unique in the oracle: {find!r}"
    return src_text.replace(find, repl)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    text = open(SRC).read()
    variants = {"unchanged": text}
    for name, (find, repl) in MUTANTS.items():
        variants[name] = _plant(text, find, repl)

    def build(item):
        name, body = item
        c = tmp_path / f"{name}.c"
        c.write_text(body)
        return name, oracle.compile_library(str(c), str(tmp_path / f"lib_{name}.so"))

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        libs = dict(ex.map(build, variants.items()))

    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), json.dumps(libs)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed["unchanged"] == [], failed["unchanged"]
    missed = [name for name in MUTANTS if not failed[name]]
    assert not missed, f"planted mistakes that no pin catches: {missed}"


if __name__ == "__main__":
    # Child process: argv[1] is a JSON map name -> library path.
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    libs = json.loads(sys.argv[1])
    print(json.dumps({name: _failing_pins(path) for name, path in libs.items()}))
