"""The oracle and the input generator (plain C) under AddressSanitizer and
UndefinedBehaviorSanitizer (CPU only): both are rebuilt instrumented, and
the oracle pins (which draw their inputs from the generator) run again in a
child process that
loads those builds. A read or write out of bounds, a use after free, a
signed overflow, a misaligned access or a shift out of range anywhere in
that code stops the child with the sanitizer's report."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    try:
        p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True,
                           check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_and_generator_clean_under_sanitizers(tmp_path):
    asan = _runtime("libasan.so")
    if asan is None:
        pytest.skip("gcc's AddressSanitizer runtime is not installed")
    sys.path.insert(0, ROOT)
    import k3synth
    import oracle
    try:
        olib = oracle.build(force=True, out=str(tmp_path / "liboracle_san.so"),
                            flags=oracle.SANITIZE_FLAGS)
        slib = k3synth.build(force=True, out=str(tmp_path / "libk3synth_san.so"),
                             flags=oracle.SANITIZE_FLAGS)
    except subprocess.CalledProcessError as e:
        pytest.skip(f"instrumented build failed: {e}")
    env = dict(os.environ, K3MOE_ORACLE_LIB=olib, K3SYNTH_LIB=slib, LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=0:exitcode=97",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1:exitcode=98")
    tests = sorted(f for f in os.listdir(os.path.join(ROOT, "tests"))
                   if f.startswith("test_oracle_") and f != "test_oracle_sanitized.py")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-s", "-m", "not gpu", "-p", "no:cacheprovider",
                        *[os.path.join("tests", t) for t in tests]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout + r.stderr
    assert "ERROR: AddressSanitizer" not in out and "runtime error:" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
    assert " passed" in out
