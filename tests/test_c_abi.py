"""The C ABI from a plain C program: tests/c_abi_checks.c is compiled with
gcc against include/opw.h, linked with the library, and run.  Every call it
makes returns before any CUDA call, so it needs no GPU."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_sees_the_documented_errors():
    from overlap_producer_warps_gb300 import api
    from overlap_producer_warps_gb300 import build as _b
    _b.build()
    lib_dir = os.path.dirname(api.LIB_PATH)
    exe = os.path.join(lib_dir, "c_abi_checks")  # the library's build folder (not tracked)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_checks.c"), "-o", exe,
                    "-L", lib_dir, "-l:" + os.path.basename(api.LIB_PATH),
                    "-Wl,-rpath," + lib_dir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all passed" in r.stdout
