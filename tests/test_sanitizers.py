"""The CPU oracle and the library's host code under AddressSanitizer and
UndefinedBehaviorSanitizer, every finding fatal: the oracle's own tests run
against the sanitized oracle, and the ABI / argument-validation tests against
the library whose host code is sanitized (no GPU needed; the device code is
the normal build's).  Each run is a child process with the sanitizer runtime
preloaded."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_TESTS = ["tests/test_oracle_pins.py", "tests/test_oracle_edge_rows.py", "tests/test_oracle_schemes.py",
                "tests/test_oracle_decode.py", "tests/test_oracle_attention.py",
                "tests/test_oracle_prefill_attention.py"]


def _asan_runtime() -> str:
    try:
        p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    except OSError:
        p = ""
    if not p or not os.path.isabs(p) or not os.path.exists(p):
        pytest.skip("no AddressSanitizer runtime for this compiler")
    return p


def _sanitized(lib: str) -> bool:
    syms = subprocess.run(["nm", "-D", lib], capture_output=True, text=True).stdout
    return "__asan" in syms and "__ubsan" in syms


def _run(tests, **env_extra):
    env = dict(os.environ, LD_PRELOAD=_asan_runtime(), ASAN_OPTIONS="detect_leaks=0", **env_extra)
    r = subprocess.run([sys.executable, "-m", "pytest", *tests, "-q", "-x", "-m", "not gpu", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    return r.stdout


def test_oracle_under_sanitizers():
    _asan_runtime()
    from oracle import build

    lib = build.build_oracle(sanitize=True)
    assert _sanitized(lib)
    out = _run(ORACLE_TESTS, ORACLE_LIBRARY="sanitized")
    assert "passed" in out


def test_host_code_under_sanitizers():
    _asan_runtime()
    from differentiated_kv_cache_dkv_gb300 import build

    lib = build.build(sanitize=True)
    assert _sanitized(lib)
    out = _run(["tests/test_abi.py"], DKV_LIBRARY="sanitized")
    assert "passed" in out
