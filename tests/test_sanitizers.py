"""The CPU-side tests again, under AddressSanitizer and UndefinedBehaviorSanitizer.

The oracle's C and libzc's host code (argument checks, sizes, the sigma closed form, the cost models, the QLC
table builder) are built a second time with -fsanitize=address,undefined (ZC_SANITIZE=1 makes the bindings
load those builds).  The oracle, stream-format, error and host-ABI tests then run in a child process that
preloads the sanitizer runtimes.  A report stops the child (UBSan is not recoverable in these builds), so the
test passes only if every one of those tests passes with no report.  No kernel runs: these are the host-side
stand-ins for the device checks of untrusted streams, which run on the GPU.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUBSET = ["tests/test_oracle_format.py", "tests/test_oracle_raw.py", "tests/test_oracle_qlc.py",
          "tests/test_oracle_stats.py", "tests/test_abi_cpu.py"]


def _runtime(name: str):
    gcc = shutil.which("gcc")
    if not gcc:
        return None
    path = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_cpu_tests_under_asan_and_ubsan():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("no sanitizer runtimes for this compiler")
    # build both instrumented libraries first, outside the preloaded child (the compilers are not instrumented)
    subprocess.check_call([sys.executable, "-c",
                           "import oracle; oracle.build(sanitize=True)\n"
                           "from lossless_bf16_exponent_zc_gb300 import _build; _build.build(sanitize=True)"],
                          cwd=ROOT)
    env = dict(os.environ, ZC_SANITIZE="1", LD_PRELOAD=f"{asan}:{ubsan}",
               # the interpreter's own allocations outlive it by design: leak reports would be about Python
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    # --capture=sys: a report written by the sanitizer runtime to fd 2 reaches this process
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "--capture=sys", "-m", "not gpu and not slow",
                        "-p", "no:cacheprovider"] + SUBSET, cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    report = r.stdout[-4000:] + r.stderr[-4000:]
    assert r.returncode == 0, report
    assert "AddressSanitizer" not in r.stderr and "runtime error:" not in r.stderr, report
    assert " passed" in r.stdout, report
