"""The host code of the C ABI (argument validation, the pipelined call's
stream and event handling) under AddressSanitizer and UndefinedBehaviorSanitizer:
the library is rebuilt with its host translation units instrumented and the
C-ABI validation tests run against it in a child process with the sanitizer
runtime preloaded.  Any report makes the child exit non-zero.  CPU only."""

import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT


def _runtime(name):
    try:
        path = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True,
                              check=True).stdout.strip()
    except Exception:
        return None
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_abi_validation_under_asan_and_ubsan():
    asan = _runtime("libasan.so")
    if asan is None:
        pytest.skip("no AddressSanitizer runtime for this compiler")
    from chunked_prefill_attention_gb300 import _build
    lib = _build.build_sanitized()
    env = dict(os.environ)
    env.update({
        "LD_PRELOAD": asan,
        "Q8ATTN_LIBRARY": lib,
        # the CUDA runtime maps memory in the shadow gap; leaks of the runtime's
        # own lifetime-long allocations are not this library's
        "ASAN_OPTIONS": "protect_shadow_gap=0:detect_leaks=0:abort_on_error=1",
        "UBSAN_OPTIONS": "halt_on_error=1:print_stacktrace=1",
    })
    probe = ("import ctypes; from chunked_prefill_attention_gb300 import q8attn; q8attn.load(); "
             "print(q8attn.LIB_PATH); print(hasattr(ctypes.CDLL(None), '__asan_init'))")
    r = subprocess.run([sys.executable, "-c", probe], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == [lib, "True"], r.stdout   # the instrumented build, ASan active
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi_cpu.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, out
    assert "AddressSanitizer" not in out and "runtime error" not in out, out
    assert " passed" in r.stdout, out
