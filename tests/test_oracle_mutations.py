"""The pins catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of the C oracle: a dropped term,
a wrong sign, a wrong index or offset, a transposed operand, a wrong rounding
rule.  The copy is compiled, and the pin suite (tests/test_oracle_pins.py)
runs against it in a child process (OPW_ORACLE_SRC names the copy; the real
source and library are not touched).  Every mutant must fail at least one pin.
A control run of an unchanged copy through the same route must pass, which
shows the route really uses the copy.

Every planted mistake keeps all reads and writes in bounds, so a failing pin,
not a crash, is what each run reports.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "opw_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# name -> (text in opw_oracle.c, replacement)
MUTANTS = {
    # bf16 codec
    "decode: shift by 15": (
        "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    "encode: ties away from zero": (
        "const double units = nearbyint(ldexp(a, -q));",
        "const double units = floor(ldexp(a, -q) + 0.5);"),
    "encode: subnormal spacing one binade off": (
        "if (e < -126) e = -126;", "if (e < -127) e = -127;"),
    "encode: one significand bit too many": (
        "const int q = e - 7;", "const int q = e - 8;"),
    "encode: NaN becomes infinity": (
        "if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);",
        "if (isnan(x)) return (uint16_t)(sign | 0x7F80u);"),
    "encode: infinity becomes NaN": (
        "if (isinf(x)) return (uint16_t)(sign | 0x7F80u);",
        "if (isinf(x)) return (uint16_t)(sign | 0x7FC0u);"),
    "encode: overflow saturates at the largest finite value": (
        "if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);",
        "if (r >= 0x1p128) return (uint16_t)(sign | 0x7F7Fu);"),
    # symmetric addresses and the gather
    "symm_at: bases swapped": (
        "return heap_base_pe + (ptr - heap_base_self);",
        "return heap_base_self + (ptr - heap_base_pe);"),
    "rank_ptr: every rank read from rank 0": (
        "const uint64_t pe_base = (uint64_t)(uintptr_t)heap + (uint64_t)rank_off[r];",
        "const uint64_t pe_base = (uint64_t)(uintptr_t)heap + (uint64_t)rank_off[0];"),
    "allgather: ranks in reverse order": (
        "memcpy(G + (int64_t)r * M_r * K, A_r,", "memcpy(G + (int64_t)(R - 1 - r) * M_r * K, A_r,"),
    # GEMM
    "gemm: last k term dropped": (
        "        for (int64_t k = 0; k < K; ++k) {\n"
        "            const double a = opw_oracle_bf16_to_f64(A[i * lda + k]);",
        "        for (int64_t k = 0; k < K - 1; ++k) {\n"
        "            const double a = opw_oracle_bf16_to_f64(A[i * lda + k]);"),
    "gemm: B columns reversed": (
        "for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];",
        "for (int64_t j = 0; j < N; ++j) c[j] += a * b[N - 1 - j];"),
    "gemm: products subtracted": (
        "for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];",
        "for (int64_t j = 0; j < N; ++j) c[j] -= a * b[j];"),
    "gemm rows: first k term dropped": (
        "for (int64_t j = 0; j < N; ++j) c[j] += av * opw_oracle_bf16_to_f64(b[j]);",
        "for (int64_t j = 0; j < N; ++j) c[j] += (k > 0) * av * opw_oracle_bf16_to_f64(b[j]);"),
    "ag_gemm rows: shard of row i taken as i mod R": (
        "const int r = (int)(i / M_r);", "const int r = (int)(i % R);"),
    # GEMM-RS
    "gemm_rs: only the last partial kept": (
        "for (int64_t i = 0; i < M * N; ++i) S[i] = S[i] + P[i];",
        "for (int64_t i = 0; i < M * N; ++i) S[i] = P[i];"),
    "gemm_rs: every rank multiplies rank 0's B": (
        "const uint16_t* B_r = (const uint16_t*)rank_ptr(heap, rank_off, r, b_off);\n"
        "        opw_oracle_gemm_f64(",
        "const uint16_t* B_r = (const uint16_t*)rank_ptr(heap, rank_off, 0, b_off);\n"
        "        opw_oracle_gemm_f64("),
    "gemm_rs: row blocks scattered to the mirrored rank": (
        "opw_oracle_bf16_encode_array(S + (int64_t)j * Mb * N, out_j, Mb * N);",
        "opw_oracle_bf16_encode_array(S + (int64_t)(R - 1 - j) * Mb * N, out_j, Mb * N);"),
    "gemm_rs rows: rank 0's partial dropped": (
        "for (int64_t j = 0; j < N; ++j) s[j] = s[j] + p[j];",
        "for (int64_t j = 0; j < N; ++j) s[j] = s[j] + (r > 0) * p[j];"),
    # signals and the consumer schedule
    "flags: previous epoch": (
        "for (int64_t i = 0; i < n_slots; ++i) out[i] = epoch;",
        "for (int64_t i = 0; i < n_slots; ++i) out[i] = epoch - 1;"),
    "row counters: epoch + T_k": (
        "out[i] = epoch * T_k;", "out[i] = epoch + T_k;"),
    "swizzle: rotated the wrong way": (
        "return (pid_m + rank * tiles_per_pe) % total_tiles;",
        "return (pid_m + total_tiles - (rank * tiles_per_pe) % total_tiles) % total_tiles;"),
    "consumer order: no alternating column sweep": (
        "const int64_t pid_n = (first / group_rows) % 2 == 0 ? col : T_N - 1 - col;",
        "const int64_t pid_n = col;"),
    "consumer order: row inside a rank's block dropped": (
        ": visit[pid_m / tiles_per_pe] * tiles_per_pe + pid_m % tiles_per_pe;",
        ": visit[pid_m / tiles_per_pe] * tiles_per_pe;"),
    "consumer order: stride G + 1": (
        "for (int64_t pos = c; pos < T_M * T_N; pos += G) {",
        "for (int64_t pos = c; pos < T_M * T_N; pos += G + 1) {"),
    # ring AllReduce and all-to-all
    "ring: partial sums travel the ring backwards": (
        "const int r = (c + k) % R;", "const int r = (c + R - k) % R;"),
    "alltoall: own slice index instead of the peer's": (
        "memcpy(recv_j + (int64_t)r * B, send_r + (int64_t)j * B, (size_t)B);",
        "memcpy(recv_j + (int64_t)r * B, send_r + (int64_t)r * B, (size_t)B);"),
}


def _run_pins(name, text, d):
    """Compile `text` as the oracle in directory d and run the pin suite
    against it; returns (name, compiled, return code, output tail)."""
    src = os.path.join(d, "opw_oracle.c")
    with open(src, "w") as f:
        f.write(text)
    cc = subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                         "-shared", "-o", os.path.join(d, "check.so"), src, "-lm"],
                        capture_output=True, text=True)
    if cc.returncode != 0:
        return name, False, cc.returncode, cc.stderr[-2000:]
    env = dict(os.environ, OPW_ORACLE_SRC=src, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return name, True, r.returncode, (r.stdout + r.stderr)[-3000:]


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    with open(SRC) as f:
        source = f.read()
    jobs = [("(unchanged copy)", source, str(tmp_path_factory.mktemp("control")))]
    for i, (name, (old, new)) in enumerate(MUTANTS.items()):
        assert source.count(old) == 1, f"{name}: the planted text must occur exactly once"
        jobs.append((name, source.replace(old, new), str(tmp_path_factory.mktemp(f"mutant{i}"))))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        out = list(ex.map(lambda job: _run_pins(*job), jobs))
    return {name: (compiled, rc, tail) for name, compiled, rc, tail in out}


def test_unchanged_copy_passes_every_pin(results):
    compiled, rc, tail = results["(unchanged copy)"]
    assert compiled and rc == 0, tail


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_the_planted_mistake(results, name):
    compiled, rc, tail = results[name]
    assert compiled, f"{name}: the mutant does not compile:\n{tail}"
    # pytest's code 1: tests ran and some failed (not a crash, not a collection error)
    assert rc == 1 and "FAILED" in tail, f"{name}: no pin failed (return code {rc}):\n{tail}"
