"""The bounds-checked build (DKV_CHECKED): it compiles, reports itself, and
runs the smoke path (prefill compaction, generation steps, decode and prefill
attention, each against the oracle) with no check firing.  The normal build
reports itself as unchecked."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_normal_build_is_unchecked():
    from differentiated_kv_cache_dkv_gb300 import libdkv

    assert libdkv.load().dkv_build_flags() & 1 == 0


@pytest.mark.gpu
def test_checked_build_runs_the_smoke_path():
    from differentiated_kv_cache_dkv_gb300 import build

    build.build(checked=True)
    code = (
        "import __graft_entry__ as g\n"
        "from differentiated_kv_cache_dkv_gb300 import libdkv\n"
        "assert libdkv.LIB_PATH.endswith('libdkv_checked.so'), libdkv.LIB_PATH\n"
        "assert libdkv.load().dkv_build_flags() & 1 == 1\n"
        "g.smoke()\n"
        "print('checked smoke ok')\n"
    )
    env = dict(os.environ, DKV_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked smoke ok" in r.stdout
